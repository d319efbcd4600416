#!/usr/bin/env python3
"""Benchmark of one MLA decode step on the DeepSeek-V3-shaped layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole path over one batch: absorb the query
(q^C W^UK + RoPE), append the decode token's latent to the cache, split-KV
latent decode (partial + combine) and the W^UV up-projection.  Workload:
16 sequences x 4096 tokens, 128 heads, d_c = 512, d_R = 64, contiguous bf16
cache, synthetic N(0, 1) data (seeded).  Layer state (cache + weights,
~117 MB) is kept in 3 copies used round-robin so no step finds its inputs in
the 126 MB L2.  Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (2 of the 16 sequences per step), scaled to the full batch.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/step, latent-cache HBM GB/s & TFLOP/s as % of B300 roofline"
UNIT = "µs/step"
ROTATE = 3
LAUNCHES_PER_STEP = {"absorb": 1, "append": 1, "decode": 2, "out_proj": 1}  # decode: partial pass + combine
DECODE_SOURCES = ["mla_latent_kv_76_b300/csrc/decode_tc.cu", "mla_latent_kv_76_b300/csrc/tc.cuh", "mla_latent_kv_76_b300/csrc/plan.cuh",
                  "mla_latent_kv_76_b300/csrc/common.cuh", "mla_latent_kv_76_b300/csrc/api.cu"]


def workload_desc(wl):
    return {
        "workload": f"DeepSeek-V3-shaped MLA layer decode: B={wl.batch}, seqlen={int(wl.seqlens[0])}, "
                    f"n_h={wl.n_heads}, d_c={wl.d_latent}, d_R={wl.d_rope}, contiguous bf16 cache, "
                    f"append 1 token/seq (d=7168)",
        "batch": wl.batch, "seqlen": int(wl.seqlens[0]), "n_heads": wl.n_heads, "d_latent": wl.d_latent,
        "d_rope": wl.d_rope, "d_head": wl.d_head, "d_model": wl.d_model,
        "step": "absorb_q || append_cache (two streams), then decode_attn (partial+combine), then out_proj",
        "l2": f"inputs larger than L2: {ROTATE} rotating copies of the layer state (cache + weights)",
    }


def algorithmic(wl):
    toks = int(np.asarray(wl.seqlens, dtype=np.int64).sum())
    D = wl.d_latent + wl.d_rope
    return {"bytes": toks * D * 2, "flops": toks * 2 * wl.n_heads * (D + wl.d_latent), "tokens": toks}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def decode_source_hash():
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode sources."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
        if j.get("source_hash") == decode_source_hash():
            return float(j["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        rows = [(t, l.split(", ")) for t, l in self.lines]
        win = [r for t, r in rows if self.t0 is not None and self.t0 - 0.15 <= t <= (self.t1 or t) + 0.15]
        use = win if win else [r for _, r in rows]
        sm = [float(r[1]) for r in use if len(r) > 8 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in use if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use if len(r) > 8 for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "window_samples": len(win),
                "power_w_max": max((float(r[3]) for r in use if len(r) > 8 and _isnum(r[3])), default=None)}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def other_configs(torch, mi, mla, dev, K: int = 30):
    """The decode call alone on the other configurations, graph-timed: the
    128-head ragged paged batch and long context (tensor-core kernel) and the
    16-head low-head batch (shape-generic kernel); their caches exceed L2.
    Supporting figures: the headline metric is the V3 step above."""
    out = {}
    peaks = load_peaks()
    for name in ("paged", "long", "lowhead"):
        wl = mi.make(name, poison=False)
        dims = mla.Dims.of(wl)
        to = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev).view(torch.bfloat16)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev)
        pool, q, sl = to(wl.pool), to(wl.q), i32(wl.seqlens)
        bt = i32(wl.block_table) if wl.paged else None
        ws = torch.empty(mla.mla_decode_workspace_size(dims, wl.batch, 0), dtype=torch.uint8, device=dev)
        z = torch.empty((wl.batch, wl.n_heads, wl.d_latent), dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def call():
            mla.mla_decode_attn(dims, q, pool, sl, wl.scale, block_table=bt, num_blocks=wl.num_blocks,
                                seq_stride=wl.seq_stride, workspace=ws, z_out=z, want_lse=False, dev_status=status)
        call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        for _ in range(5):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        if mla.mla_read_status(status) != 0:
            raise RuntimeError(f"device status during the {name} decode timing")
        us = e0.elapsed_time(e1) * 1e3 / K
        alg = algorithmic(wl)
        gbs = alg["bytes"] / (us * 1e-6) / 1e9
        out[name] = {"decode_us": round(us, 2), "batch": wl.batch, "tokens": alg["tokens"], "hbm_gbs": round(gbs, 1),
                     "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "tflops": round(alg["flops"] / (us * 1e-6) / 1e12, 1)}
        del pool, q, ws, z
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- our arm
def max_over_ranks(x: float, dist, device) -> float:
    """The largest `x` over all ranks (every rank gets it); `x` itself when
    there is no process group.  Replicas are timed independently and the job
    is as slow as its slowest rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(batch: int, world: int, us_per_step: float) -> float:
    """Whole-job throughput: every replica decodes `batch` sequences per step."""
    return batch * world / (us_per_step * 1e-6)


def run_ours(args, rank, world, local_rank):
    import torch
    import mla_inputs as mi
    from __graft_entry__ import build
    build()
    import mla_latent_kv_76_b300 as mla

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = mi.make("v3", poison=False)
    dims = mla.Dims.of(wl)
    to = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev).view(torch.bfloat16)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev)

    # layer state: cache + weights, ROTATE copies (each a distinct allocation)
    pool0, wuk0, wuv0, wkv0 = to(wl.pool), to(wl.w_uk), to(wl.w_uv), to(wl.w_dkv_kr)
    layers = [dict(pool=pool0.clone(), w_uk=wuk0.clone(), w_uv=wuv0.clone(), w_kv=wkv0.clone())
              for _ in range(ROTATE)]
    del pool0, wuk0, wuv0, wkv0
    B = wl.batch
    # per-step inputs, packed into one device buffer (256-byte aligned views) so
    # that the end-to-end step moves them with a single host -> device copy
    host_inputs = [np.ascontiguousarray(wl.q_c).view(np.uint8), np.ascontiguousarray(wl.q_r).view(np.uint8),
                   np.ascontiguousarray(wl.h).view(np.uint8)] + \
                  [np.ascontiguousarray(np.asarray(a, dtype=np.int32)).view(np.uint8)
                   for a in (wl.q_pos, wl.app_seq, wl.app_pos, wl.seqlens)]
    offs, total = [], 0
    for a in host_inputs:
        offs.append(total)
        total += (a.nbytes + 255) // 256 * 256
    packed_host = np.zeros(total, dtype=np.uint8)
    for a, o0 in zip(host_inputs, offs):
        packed_host[o0:o0 + a.nbytes] = a.reshape(-1)
    packed = torch.from_numpy(packed_host).to(dev)

    def view(k, dtype, shape):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        return packed[offs[k]:offs[k] + n].view(dtype).view(shape)

    q_c = view(0, torch.bfloat16, wl.q_c.shape)
    q_r = view(1, torch.bfloat16, wl.q_r.shape)
    h = view(2, torch.bfloat16, wl.h.shape)
    q_pos, app_seq, app_pos, seqlens = (view(3 + k, torch.int32, (B,)) for k in range(4))
    ws = torch.empty(mla.mla_decode_workspace_size(dims, B, 0), dtype=torch.uint8, device=dev)
    q = torch.empty((B, wl.n_heads, wl.row_dim), dtype=torch.bfloat16, device=dev)
    z = torch.empty((B, wl.n_heads, wl.d_latent), dtype=torch.bfloat16, device=dev)
    o = torch.empty((B, wl.n_heads, wl.d_v), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def step(i):
        # absorb and append touch disjoint data, so they run on two streams
        # (fork / join); decode needs both, out_proj needs decode
        L = layers[i % ROTATE]
        fork.record(stream)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            mla.mla_append_cache(dims, h, L["w_kv"], app_seq, app_pos, L["pool"], n_seqs=B,
                                 seq_stride=wl.seq_stride, dev_status=status)
            join.record(side)
        mla.mla_absorb_q(dims, q_c, q_r, q_pos, L["w_uk"], q_out=q)
        stream.wait_event(join)
        decode(i)
        mla.mla_out_proj(dims, z, L["w_uv"], o_out=o)

    def decode(i):
        L = layers[i % ROTATE]
        mla.mla_decode_attn(dims, q, L["pool"], seqlens, wl.scale, seq_stride=wl.seq_stride, workspace=ws,
                            z_out=z, want_lse=False, dev_status=status)

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # Each step (and each decode alone) is captured once per layer copy as a CUDA
    # graph; the timed region replays graphs, so host-side launch overhead does
    # not enter the device time.
    for i in range(ROTATE):
        step(i)  # first calls outside capture (one-time kernel attribute set-up)
    torch.cuda.synchronize()
    g_step, g_dec = [], []
    for i in range(ROTATE):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(i)
        g_step.append(g)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            decode(i)
        g_dec.append(g)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    for i in range(max(3, args.warmup)):
        g_step[i % ROTATE].replay()
    # pre-roll so the clock sampler sees the GPU under this load around the timed region
    t_end = time.time() + (0.6 if sampler else 0.0)
    i = 0
    while time.time() < t_end:
        g_step[i % ROTATE].replay()
        i += 1
        if i % 200 == 0:
            torch.cuda.synchronize()
    # ---- timed region: exactly K steps, device time via events on the launching stream
    K = args.steps
    barrier()
    if sampler:
        sampler.mark_begin()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(K):
        g_step[k % ROTATE].replay()
    t_stop.record(stream)
    barrier()
    if sampler:
        sampler.mark_end()
    total_ms = t_start.elapsed_time(t_stop)
    # decode alone (split-KV partial + combine), same rotation, for the roofline
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for k in range(K):
        g_dec[k % ROTATE].replay()
    d1.record(stream)
    barrier()
    dec_us_list = [max_over_ranks(d0.elapsed_time(d1) * 1e3 / K, dist, dev)]
    # post-roll for the sampler
    t_end = time.time() + (0.3 if sampler else 0.0)
    while time.time() < t_end:
        g_step[i % ROTATE].replay()
        i += 1
        if i % 200 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    st = mla.mla_read_status(status)
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")
    us_per_step = max_over_ranks(total_ms * 1e3 / K, dist, dev)

    # ---- end to end through the public API with host buffers: every step copies
    # its packed inputs from pinned host memory and reads the output back
    h_in = torch.from_numpy(packed_host).pin_memory()
    h_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    h2d = h_in.numel()
    d2h = h_o.numel() * h_o.element_size()

    def e2e_step(i):
        packed.copy_(h_in, non_blocking=True)
        step(i)
        h_o.copy_(o, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    barrier()
    # the eager path is bound by host-side work, which other tenants of the host
    # can disturb: three timed runs of K steps, the median reported
    e2e_runs = []
    for _ in range(3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(K):
            e2e_step(k)
        e1.record(stream)
        barrier()
        e2e_runs.append(e0.elapsed_time(e1) * 1e3 / K)
    e2e_us = max_over_ranks(statistics.median(e2e_runs), dist, dev)
    if sampler:
        sampler.stop()
    others = other_configs(torch, mi, mla, dev) if (rank == 0 and not args.no_others) else None

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    alg = algorithmic(wl)
    peaks = load_peaks()
    dec_us = statistics.mean(dec_us_list)
    dec_gbs = alg["bytes"] / (dec_us * 1e-6) / 1e9
    dec_tfs = alg["flops"] / (dec_us * 1e-6) / 1e12
    t_hbm = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["flops"] / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = measured_traffic()
    roof = {"bound": bound, "kernel": "mla_decode_attn (split-KV partial + combine)",
            "achieved": round(dec_gbs if bound == "hbm" else dec_tfs, 1),
            "peak": peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops"],
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": round((dec_gbs / peaks["hbm_gbs"]) if bound == "hbm" else (dec_tfs / peaks["bf16_tflops"]), 4),
            "traffic": traffic, "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": alg["bytes"], "algorithmic_flops_per_launch": alg["flops"],
            "tensor_achieved_tflops": round(dec_tfs, 1), "tensor_frac": round(dec_tfs / peaks["bf16_tflops"], 4),
            "roofline_time_us": round(max(t_hbm, t_tc) * 1e6, 2),
            "roofline_frac": round(max(t_hbm, t_tc) * 1e6 / dec_us, 4)}
    cpu = cpu_baseline(wl, args.cpu_seconds) if not args.no_cpu else None
    line = {
        "metric": METRIC, "value": round(us_per_step, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(us_per_step / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), random-init weights)",
        "config": dict(workload_desc(wl), parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "tokens_per_s": round(job_tokens_per_s(wl.batch, world, us_per_step), 1),
        "decode": {"us": round(dec_us, 3), "timing": "CUDA-graph replays of the decode call alone, same rotation",
                   "hbm_gbs": round(dec_gbs, 1), "tflops": round(dec_tfs, 1),
                   "tokens_per_s": round(wl.batch / (dec_us * 1e-6), 1)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "runs": [round(x, 1) for x in e2e_runs],
                "path": "eager public API calls; the packed inputs copied in from one pinned host buffer, the output copied out"},
        "timing": "CUDA-graph replay of each step (one graph per rotating layer copy), CUDA events",
        "other_configs": others,
        "gpu_launches": K * sum(LAUNCHES_PER_STEP.values()),
        "clocks": sampler.summary() if sampler else None,
    }
    if dist is not None:
        dist.destroy_process_group()
    return line


# --------------------------------------------------------------------------- CPU oracle
def oracle_step(wl, seqs, pool):
    """The oracle's whole step for the sequences in `seqs`: absorb, append,
    decode, up-project (fp64 numpy, as it stands)."""
    import oracle as orc
    sel = np.asarray(seqs)
    w_uk = orc.bf16_to_f64(wl.w_uk)
    w_uv = orc.bf16_to_f64(wl.w_uv)
    q_lat = orc.absorb_q(orc.bf16_to_f64(wl.q_c[sel]), orc.bf16_to_f64(wl.q_r[sel]), wl.q_pos[sel], w_uk,
                         wl.rope_base)
    new_pool = orc.append_cache(pool, wl.h[sel], wl.w_dkv_kr, wl.app_seq[sel], wl.app_pos[sel], wl.d_latent,
                                None, wl.block_tokens, wl.seq_stride, wl.rope_base)
    zs = []
    for i, b in enumerate(sel):
        rows = orc.gather_rows(new_pool, int(b), int(wl.seqlens[b]), None, wl.block_tokens, wl.seq_stride)
        z, _ = orc.decode_latent(q_lat[i], rows, wl.scale, wl.d_latent)
        zs.append(z)
    return orc.out_proj(np.stack(zs), w_uv)


def _threads():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(wl, seconds: float):
    """Oracle timed on the host cores on a bounded sample: whole steps over 2
    of the 16 sequences, repeated for about `seconds`; scaled to the batch."""
    n = 2
    seqs = list(range(n))
    pool = wl.pool
    oracle_step(wl, seqs, pool)  # warm
    times = []
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end or len(times) < 2:
        t0 = time.perf_counter()
        oracle_step(wl, seqs, pool)
        times.append(time.perf_counter() - t0)
    per = statistics.median(times) * (wl.batch / n)
    return {"value": round(per * 1e6, 1), "unit": UNIT, "cores": _threads(), "kind": "oracle",
            "sample": f"whole oracle steps over {n} of {wl.batch} sequences, x{len(times)} "
                      f"({sum(times):.1f} s), scaled by {wl.batch // n}"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import mla_inputs as mi
    wl = mi.make("v3", poison=False)
    n = 2
    seqs = list(range(n))
    for _ in range(max(0, args.warmup)):
        oracle_step(wl, seqs, wl.pool)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(wl, seqs, wl.pool)
        times.append(time.perf_counter() - t0)
    per_us = statistics.mean(times) * 1e6 * (wl.batch / n)
    cores = _threads()
    sample = f"each step: the whole oracle step over {n} of {wl.batch} sequences, scaled by {wl.batch // n}"
    return {
        "impl": "reference", "metric": METRIC, "value": round(per_us, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_us / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), random-init weights)",
        "config": dict(workload_desc(wl), parallelism="host cores (fp64 CPU oracle)"),
        "cpu_baseline": {"value": round(per_us, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(per_us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-others", action="store_true", help="skip the paged / long / low-head decode figures")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local_rank)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
