"""The parity tolerance itself, checked on the CPU with a planted mistake.

The GPU-vs-oracle bound is applied per output: max|d| <= 1e-2 max|ref| on every
(sequence, head) row and sum|d| / sum|ref| <= 2e-3 on every sequence.  Applied
batch-wide instead, a
short sequence (whose z is a single cache row, |z| ~ 1) sets the scale and a
long sequence's z (|z| ~ 0.1: a softmax over a few hundred effective tokens)
can be wrong by several percent without moving the batch-wide figures.  The
planted mistake here is one a tail-masking bug would make: a decode that drops
the last 32 visible tokens of a 4097-token sequence in a ragged batch.
"""
import numpy as np
import pytest

import mla_inputs as mi
import oracle as orc
from helpers import MAX_REL, MEAN_REL, assert_close, err_stats


def _oracle_z(wl, b, drop=None):
    rows = orc.gather_rows(wl.pool, b, int(wl.seqlens[b]), wl.block_table if wl.paged else None,
                           wl.block_tokens, wl.seq_stride)
    if drop is not None:
        keep = np.ones(len(rows), dtype=bool)
        keep[drop] = False
        rows = rows[keep]
    z, _ = orc.decode_latent(orc.bf16_to_f64(wl.q[b]), rows, wl.scale, wl.d_latent)
    return z


def test_per_sequence_check_catches_a_dropped_tail_that_a_batch_wide_check_misses():
    lens = [1, 2, 3, 63, 64, 65, 127, 128, 129, 191, 4097]
    wl = mi.make_random(41, 16, 512, 64, lens, paged=True, poison=False)
    ref = np.stack([_oracle_z(wl, b) for b in range(len(lens))])
    bad = ref.copy()
    bad[-1] = _oracle_z(wl, len(lens) - 1, drop=slice(4065, 4097))   # last 32 tokens missing
    # the error is real: ~2 % of the long sequence's own output, 9x the mean bound
    d1 = np.abs(bad[-1] - ref[-1]).sum() / np.abs(ref[-1]).sum()
    assert d1 > 5 * MEAN_REL
    # batch-wide figures stay inside the bound ...
    mx, mn = err_stats(bad, ref)
    assert mx <= MAX_REL and mn <= MEAN_REL, (mx, mn)
    # ... the per-sequence check does not
    with pytest.raises(AssertionError, match="1 of 11 sequences beyond the mean bound"):
        assert_close(bad, ref, "planted dropped tile")
    # and the correct result passes it
    assert_close(ref, ref, "oracle against itself")


def test_check_reports_the_offending_row_and_sequence():
    ref = np.ones((3, 4, 8))
    got = ref.copy()
    got[2, 1, :] *= 1.02                                     # 2 % off on one (sequence, head) row
    with pytest.raises(AssertionError, match=r"1 of 12 rows.*row \(2, 1\).*1 of 3 sequences.*sequence 2"):
        assert_close(got, ref, "one row")
    got = ref.copy()
    got[1, :, :] *= 1.005                                    # 0.5 % off on a whole sequence: mean bound
    with pytest.raises(AssertionError, match=r"0 of 12 rows.*1 of 3 sequences.*sequence 1"):
        assert_close(got, ref, "one sequence")
