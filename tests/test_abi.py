"""The C ABI library: it loads, exports every symbol include/mla.h declares,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mla():
    from __graft_entry__ import build
    build()
    import mla_latent_kv_76_b300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("mla_absorb_q", "mla_append_cache", "mla_decode_attn", "mla_decode_workspace_size",
                 "mla_out_proj", "mla_read_status", "mla_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(mla):
    out = subprocess.run(["nm", "-D", "--defined-only", mla.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (mla_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(mla.lib, name)


def test_build_targets_sm_103a_only():
    from __graft_entry__ import _build_module
    assert _build_module().ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_build_works_from_a_checkout_without_the_library(tmp_path):
    """build() must not need the library it builds (fresh clone)."""
    dst = tmp_path / "repo"
    try:  # the tracked files are exactly what a fresh clone holds
        files = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True, check=True,
                               timeout=60).stdout.split()
    except (OSError, subprocess.SubprocessError):
        files = None
    if files:
        for rel in files:
            src = os.path.join(ROOT, rel)
            if os.path.isfile(src):
                os.makedirs(os.path.dirname(os.path.join(dst, rel)) or str(dst), exist_ok=True)
                shutil.copy2(src, os.path.join(dst, rel))
    else:
        shutil.copytree(ROOT, dst, ignore=shutil.ignore_patterns("*.so", "*.o", "_build", "__pycache__", ".git",
                                                                 "_work", "*.ncu-rep", "*.npz", "*.log", "*.csv"))
    r = subprocess.run([sys.executable, "-c", "import __graft_entry__ as g; g.build(); "
                        "import mla_latent_kv_76_b300 as m; print(m.mla_version())"],
                       cwd=dst, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().endswith("10000")


def test_status_strings_and_version(mla):
    assert mla.mla_status_string(0) == "ok"
    assert "workspace" in mla.mla_status_string(mla.MLA_ERR_WORKSPACE)
    assert mla.mla_status_string(12345) == "unknown status"
    assert mla.mla_version() >= 10000


def _dims(mla, **kw):
    d = dict(n_heads=128, d_head=128, d_v=128, d_latent=512, d_rope=64, block_tokens=64, rope_base=10000.0)
    d.update(kw)
    return mla.Dims(**d)


def test_host_validation_rejects_bad_arguments(mla):
    lib = mla.lib
    d = _dims(mla)
    # null dims / negative sizes
    assert lib.mla_absorb_q(None, 1, 16, 16, 16, 16, 16, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_absorb_q(ctypes.byref(d), -1, 16, 16, 16, 16, 16, None) == mla.MLA_ERR_INVALID_ARG
    # batch 0 is a no-op that succeeds without a GPU
    assert lib.mla_absorb_q(ctypes.byref(d), 0, None, None, None, None, None, None) == mla.MLA_OK
    assert lib.mla_out_proj(ctypes.byref(d), 0, None, None, None, None) == mla.MLA_OK
    # null pointers
    assert lib.mla_absorb_q(ctypes.byref(d), 2, None, 16, 16, 16, 16, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_out_proj(ctypes.byref(d), 2, 16, None, 16, None) == mla.MLA_ERR_INVALID_ARG
    # misaligned pointer
    assert lib.mla_out_proj(ctypes.byref(d), 2, 18, 16, 16, None) == mla.MLA_ERR_INVALID_ARG
    # odd rope dim / bad base
    bad = _dims(mla, d_rope=63)
    assert lib.mla_absorb_q(ctypes.byref(bad), 1, 16, 16, 16, 16, 16, None) == mla.MLA_ERR_INVALID_ARG
    bad = _dims(mla, rope_base=0.0)
    assert lib.mla_out_proj(ctypes.byref(bad), 1, 16, 16, 16, None) == mla.MLA_ERR_INVALID_ARG


def test_decode_validation(mla):
    lib = mla.lib
    d = _dims(mla)

    def call(dd, batch=1, q=16, pool=16, bt=None, mb=0, nb=0, ss=64, sl=16, scale=0.07, nw=0, flags=0,
             ws=16, wsb=1 << 30, z=16):
        return lib.mla_decode_attn(ctypes.byref(dd) if dd is not None else None, batch, q, pool, bt, mb, nb, ss,
                                   sl, scale, nw, flags, ws, wsb, z, 1, None, None, None)
    assert call(None) == mla.MLA_ERR_INVALID_ARG
    assert call(_dims(mla, d_latent=96)) == mla.MLA_ERR_UNSUPPORTED
    assert call(_dims(mla, n_heads=129)) == mla.MLA_ERR_UNSUPPORTED
    assert call(_dims(mla, d_rope=8)) == mla.MLA_ERR_UNSUPPORTED          # 520 not a multiple of 16
    assert call(d, batch=0) == mla.MLA_OK
    assert call(d, batch=-1) == mla.MLA_ERR_INVALID_ARG
    assert call(d, batch=5000) == mla.MLA_ERR_UNSUPPORTED
    assert call(d, q=None) == mla.MLA_ERR_INVALID_ARG
    assert call(d, sl=None) == mla.MLA_ERR_INVALID_ARG
    assert call(d, scale=float("nan")) == mla.MLA_ERR_INVALID_ARG
    assert call(d, flags=8) == mla.MLA_ERR_INVALID_ARG
    assert call(d, nw=-1) == mla.MLA_ERR_INVALID_ARG
    assert call(d, bt=16, mb=0) == mla.MLA_ERR_INVALID_ARG                # paged without capacity
    assert call(_dims(mla, block_tokens=32), bt=16, mb=4, nb=4) == mla.MLA_ERR_UNSUPPORTED
    assert call(d, ss=0) == mla.MLA_ERR_INVALID_ARG                      # contiguous without stride
    # workspace sizing: explicit worker counts need no device
    n1 = lib.mla_decode_workspace_size(ctypes.byref(d), 16, 10)
    n2 = lib.mla_decode_workspace_size(ctypes.byref(d), 16, 20)
    assert n2 - n1 >= 10 * 128 * 513 * 4 and n1 >= 26 * 128 * 512 * 4
    assert lib.mla_decode_workspace_size(ctypes.byref(_dims(mla, d_latent=96)), 16, 10) == 0
    assert lib.mla_decode_workspace_size(ctypes.byref(d), -1, 10) == 0


def test_append_validation(mla):
    lib = mla.lib
    d = _dims(mla)
    args = lambda **kw: dict(dict(T=1, dm=7168, h=16, w=16, si=16, pos=16, ns=1, bt=16, mb=4, nb=4, ss=0,
                                  pool=16), **kw)

    def call(dd, **kw):
        a = args(**kw)
        return lib.mla_append_cache(ctypes.byref(dd) if dd is not None else None, a["T"], a["dm"], a["h"],
                                    a["w"], a["si"], a["pos"], a["ns"], a["bt"], a["mb"], a["nb"], a["ss"],
                                    a["pool"], None, None)
    assert call(None) == mla.MLA_ERR_INVALID_ARG
    assert call(d, T=0) == mla.MLA_OK
    assert call(d, dm=7170) == mla.MLA_ERR_UNSUPPORTED
    assert call(d, h=None) == mla.MLA_ERR_INVALID_ARG
    assert call(d, mb=0) == mla.MLA_ERR_INVALID_ARG
    assert call(d, bt=None, ss=0) == mla.MLA_ERR_INVALID_ARG
    assert call(d, ns=0) == mla.MLA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(tmp_path):
    """A copy of the package without libmla.so must refuse to import."""
    pkg = os.path.join(ROOT, "mla_latent_kv_76_b300")
    dst = tmp_path / "mla_latent_kv_76_b300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import mla_latent_kv_76_b300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "libmla.so is missing" in r.stderr


def test_binding_refuses_undersized_buffers(mla):
    """The C ABI sees only pointers, so the binding checks every buffer against
    the element count the call will touch before anything is launched (these
    tensors live on the host: the size check comes first)."""
    import torch
    d = _dims(mla, n_heads=4, d_head=8, d_v=8, d_latent=64, d_rope=16)
    bf = dict(dtype=torch.bfloat16)
    B, D = 2, 80
    ok_q = torch.zeros(B, 4, D, **bf)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    sl = torch.ones(B, dtype=torch.int32)

    def raises(fn, name):
        with pytest.raises(ValueError, match=name + " holds"):
            fn()
    raises(lambda: mla.mla_absorb_q(d, torch.zeros(B, 4, 8, **bf), torch.zeros(B, 4, 16, **bf),
                                    torch.zeros(B, dtype=torch.int32), torch.zeros(4, 8, 63, **bf)), "w_uk")
    raises(lambda: mla.mla_absorb_q(d, torch.zeros(B, 4, 7, **bf), torch.zeros(B, 4, 16, **bf),
                                    torch.zeros(B, dtype=torch.int32), torch.zeros(4, 8, 64, **bf)), "q_c")
    raises(lambda: mla.mla_decode_attn(d, ok_q[:, :3], torch.zeros(B, 8, D, **bf), sl, 0.1, seq_stride=8,
                                       workspace=ws), "q")
    raises(lambda: mla.mla_decode_attn(d, ok_q, torch.zeros(B, 7, D, **bf), sl, 0.1, seq_stride=8,
                                       workspace=ws), "pool")
    raises(lambda: mla.mla_decode_attn(d, ok_q, torch.zeros(B, 8, D, **bf), sl[:1], 0.1, seq_stride=8,
                                       workspace=ws), "seqlens")
    raises(lambda: mla.mla_decode_attn(d, ok_q, torch.zeros(5, 64, D, **bf), sl, 0.1, workspace=ws,
                                       block_table=torch.zeros(B, 3, dtype=torch.int32), num_blocks=6), "pool")
    raises(lambda: mla.mla_decode_attn(d, ok_q, torch.zeros(B, 8, D, **bf), sl, 0.1, seq_stride=8, workspace=ws,
                                       z_out=torch.zeros(B, 4, 63)), "z_out")
    raises(lambda: mla.mla_decode_attn(d, ok_q, torch.zeros(B, 8, D, **bf), sl, 0.1, seq_stride=8, workspace=ws,
                                       lse_out=torch.zeros(B, 3)), "lse_out")
    with pytest.raises(TypeError, match="z_out"):
        mla.mla_decode_attn(d, ok_q, torch.zeros(B, 8, D, **bf), sl, 0.1, seq_stride=8, workspace=ws,
                            z_out=torch.zeros(B, 4, 64, dtype=torch.int32))
    raises(lambda: mla.mla_append_cache(d, torch.zeros(3, 16, **bf), torch.zeros(D, 16, **bf),
                                        torch.zeros(3, dtype=torch.int32), torch.zeros(3, dtype=torch.int32),
                                        torch.zeros(2, 8, D - 1, **bf), n_seqs=2, seq_stride=8), "pool")
    raises(lambda: mla.mla_append_cache(d, torch.zeros(3, 16, **bf), torch.zeros(D, 15, **bf),
                                        torch.zeros(3, dtype=torch.int32), torch.zeros(3, dtype=torch.int32),
                                        torch.zeros(2, 8, D, **bf), n_seqs=2, seq_stride=8), "w_dkv_kr")
    raises(lambda: mla.mla_append_cache(d, torch.zeros(3, 16, **bf), torch.zeros(D, 16, **bf),
                                        torch.zeros(2, dtype=torch.int32), torch.zeros(3, dtype=torch.int32),
                                        torch.zeros(2, 8, D, **bf), n_seqs=2, seq_stride=8), "seq_idx")
    raises(lambda: mla.mla_out_proj(d, torch.zeros(B, 4, 64, **bf), torch.zeros(4, 8, 64, **bf),
                                    o_out=torch.zeros(B, 4, 7, **bf)), "o_out")
    # right sizes get past the checks and stop at the device requirement
    with pytest.raises(ValueError, match="CUDA tensor"):
        mla.mla_out_proj(d, torch.zeros(B, 4, 64, **bf), torch.zeros(4, 8, 64, **bf))
