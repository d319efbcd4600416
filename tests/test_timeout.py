"""The device-side bounded wait, exercised on the GPU without a fault or a hang.

Every kernel of the library waits on its mbarriers through one bounded wait:
after its cycle budget it raises the CTA's abort flag, stores
MLA_ERR_DEVICE_TIMEOUT in the status word and returns false, and the CTA's
other roles leave their waits on that flag.  mla_selftest_bounded_wait runs
that wait against a barrier nothing arrives on, with a short budget, so the
whole path runs: the kernel returns, the status reads back as a timeout, and
the context stays usable for the next call.
"""
import time

import numpy as np
import pytest
import torch

import mla_inputs as mi
from helpers import bits_to_dev, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from __graft_entry__ import build
    build()
    import mla_latent_kv_76_b300 as m
    return m


def test_a_wait_that_runs_out_reports_a_timeout_and_returns(mla):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    mla.mla_selftest_bounded_wait(2_000_000, False, status, out)   # ~1 ms of SM cycles
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert mla.mla_read_status(status) == mla.MLA_ERR_DEVICE_TIMEOUT
    # the short wait gave up; the other role left its (2 s) wait on the abort flag
    assert out.tolist() == [0, 0]


def test_completed_barriers_report_nothing(mla):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    mla.mla_selftest_bounded_wait(2_000_000, True, status, out)
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == 0
    assert out.tolist() == [1, 1]


def test_the_context_is_usable_after_a_timeout(mla):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    mla.mla_selftest_bounded_wait(1_000_000, False, status, out)
    torch.cuda.synchronize()
    assert mla.mla_read_status(status) == mla.MLA_ERR_DEVICE_TIMEOUT
    # a regular decode right after runs and reports nothing
    wl = mi.make_random(77, 128, 512, 64, [300, 5], paged=True, poison=False)
    dims = mla.Dims.of(wl)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    z, _ = mla.mla_decode_attn(dims, bits_to_dev(wl.q), bits_to_dev(wl.pool), i32(wl.seqlens), wl.scale,
                               block_table=i32(wl.block_table), num_blocks=wl.num_blocks, dev_status=st2)
    torch.cuda.synchronize()
    assert mla.mla_read_status(st2) == 0
    assert bool(torch.isfinite(z).all())


def test_budget_outside_the_allowed_range_is_refused(mla):
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    for bad in (0, -5, 10**10):
        with pytest.raises(mla.MlaError) as e:
            mla.mla_selftest_bounded_wait(bad, False, None, out)
        assert e.value.code == mla.MLA_ERR_INVALID_ARG
