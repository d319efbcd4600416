"""The decode entry point that allocates nothing (mla_decode_attn_noalloc).

Some callers cannot allocate device memory when they call decode - a plugin
handed only its input and output buffers, or a serving loop that forbids
cudaMalloc after start-up.  This entry point keeps the split-KV partials in
the library's own fixed device array instead of a caller workspace.  Its
results must equal those of the regular entry point, also on the second of
two calls in a row (the array keeps the previous call's contents).
"""
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


def _inputs(wl):
    return dict(q=bits_to_dev(wl.q), pool=bits_to_dev(wl.pool), seqlens=i32(wl.seqlens),
                block_table=i32(wl.block_table) if wl.paged else None)


def test_noalloc_matches_regular_decode_on_two_calls_in_a_row(mla):
    # two different workloads, so the second call starts from the first's leftovers
    cases = [mi.make_random(31, 128, 512, 64, [1, 65, 700, 2048], paged=True),
             mi.make_random(32, 16, 512, 64, [3000, 5, 129], paged=False)]
    for wl in cases:
        dims = mla.Dims.of(wl)
        a = _inputs(wl)
        kw = dict(block_table=a["block_table"], num_blocks=wl.num_blocks, seq_stride=wl.seq_stride)
        z_ref, lse_ref = mla.mla_decode_attn(dims, a["q"], a["pool"], a["seqlens"], wl.scale, **kw)
        z = torch.empty_like(z_ref)
        lse = torch.empty_like(lse_ref)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        mla.mla_decode_attn_noalloc(dims, a["q"], a["pool"], a["seqlens"], wl.scale, z_out=z, lse_out=lse,
                                    dev_status=status, **kw)
        torch.cuda.synchronize()
        assert mla.mla_read_status(status) == 0
        # the same kernels, split plan and inputs: the results are bit for bit equal
        assert torch.equal(z.view(torch.int32), z_ref.view(torch.int32)), "z noalloc vs regular"
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), "lse noalloc vs regular"


def test_noalloc_second_call_allocates_nothing(mla):
    wl = mi.make_random(33, 128, 512, 64, [4096, 100], paged=True)
    dims = mla.Dims.of(wl)
    a = _inputs(wl)
    kw = dict(block_table=a["block_table"], num_blocks=wl.num_blocks, seq_stride=wl.seq_stride)
    z = torch.empty((wl.batch, 128, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((wl.batch, 128), dtype=torch.float32, device="cuda")
    mla.mla_decode_attn_noalloc(dims, a["q"], a["pool"], a["seqlens"], wl.scale, z_out=z, lse_out=lse, **kw)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    first = z.clone()
    mla.mla_decode_attn_noalloc(dims, a["q"], a["pool"], a["seqlens"], wl.scale, z_out=z, lse_out=lse, **kw)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.equal(z.view(torch.int32), first.view(torch.int32)), "z second call"


def test_noalloc_rejects_requests_beyond_its_scratch(mla):
    B = 300                                   # 128 heads x (G + 300) slots of 256 KiB > 64 MiB
    wl = mi.make_random(34, 128, 512, 64, [1] * B, paged=False)
    dims = mla.Dims.of(wl)
    a = _inputs(wl)
    need = mla.mla_decode_workspace_size(dims, B, 0)
    assert need > mla.MLA_NOALLOC_SCRATCH_BYTES
    z = torch.full((B, 128, 512), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_attn_noalloc(dims, a["q"], a["pool"], a["seqlens"], wl.scale, seq_stride=wl.seq_stride,
                                    z_out=z)
    assert e.value.code == mla.MLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((z == 7.0).all())             # nothing was enqueued


def test_noalloc_sizes_its_check_by_the_workers_it_uses(mla):
    # 150 sequences: above the limit for one worker per SM (the conservative
    # mla_decode_workspace_size(..., 0)), inside it for the tensor-core path's
    # one worker per SM pair, which is what the call launches
    B = 150
    wl = mi.make_random(35, 128, 512, 64, [1 + (7 * b) % 300 for b in range(B)], paged=False)
    dims = mla.Dims.of(wl)
    assert mla.mla_decode_workspace_size(dims, B, 0) > mla.MLA_NOALLOC_SCRATCH_BYTES
    a = _inputs(wl)
    z_ref, lse_ref = mla.mla_decode_attn(dims, a["q"], a["pool"], a["seqlens"], wl.scale, seq_stride=wl.seq_stride)
    z = torch.empty_like(z_ref)
    lse = torch.empty_like(lse_ref)
    mla.mla_decode_attn_noalloc(dims, a["q"], a["pool"], a["seqlens"], wl.scale, seq_stride=wl.seq_stride,
                                z_out=z, lse_out=lse)
    torch.cuda.synchronize()
    assert torch.equal(z.view(torch.int32), z_ref.view(torch.int32)), "z noalloc vs regular"
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), "lse noalloc vs regular"
