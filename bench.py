#!/usr/bin/env python
"""Benchmark of the FP8 lightning indexer on one GB300 (or N, one process per GPU).

Default workload: the 128K long-context decode step - batch 128, contexts
uniform in [64K, 128K] in a 2.2 GB paged k cache (block 64, 8704-byte blocks,
shuffled block tables). One step is the whole decode path: insert the new
token's k (fused quantisation), paged FP8 MQA logits over every visible
token, top-2048 per row, request-local -> physical slot conversion.
``value`` is query rows per second with every input resident in HBM; the k
cache (2.2 GB) is larger than L2, so no flush is needed between steps.

Other workloads (``--workload``): ``paged_decode`` (batch 64, 8K-32K),
``prefill`` (8192 queries on a 32K context), ``hierarchical`` (V4.1 sparse
decode at 128K).

``--impl reference`` times the CPU oracle (the only reference implementation
there is) on the same workload, metric and unit, on a bounded sample of rows.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_indexer_fp8_gb300 import workloads as W  # noqa: E402

PROFILE_DIR = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_hash(name: str) -> str:
    with open(os.path.join(ROOT, "sparse_attention_indexer_fp8_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(profile: str, kernel_src: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(PROFILE_DIR, profile)
    if not os.path.exists(p):
        return None
    fields = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha256_16") != source_hash(kernel_src):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        used = inside if inside else [p for _, p in self.samples]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[0]) for p in used if p[0].replace(".", "", 1).isdigit()]
        mx = [float(p[1]) for p in used if p[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in used for i in range(4) if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(used), "in_timed_region": len(inside)}


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, local, None


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------- oracle side

def oracle_decode_rows(wl: W.DecodeWorkload, rows, k_rows, reps: int = 1):
    """Time the oracle's decode step (new-token insert, logits, top-k, slots) on sample rows.

    ``k_rows[b]`` = (k8, kscale) of request b, prepared beforehand (the cache is
    state, not per-step work). Returns (seconds, per-row results).
    """
    from oracle import indexer as O

    out = {}
    t0 = time.perf_counter()
    for _ in range(reps):
        for b in rows:
            L = int(wl.pool.ctx_lens[b])
            k8, ks = k_rows[b]
            O.k_quant(np.zeros((1, 128), dtype=np.float32))          # the new token's insert
            lg = O.logits_row(wl.q8[b], wl.w[b], k8, ks)
            sel = O.topk_row(lg, 0, L, wl.topk)
            sl = O.req_to_global_slots(sel[None], None, wl.pool.block_table[b:b + 1],
                                       wl.pool.block_size, wl.block_span)
            out[b] = (lg, sel, sl[0])
    return time.perf_counter() - t0, out


def oracle_k_rows(wl: W.DecodeWorkload, rows, device):
    """Quantised k of sample requests, from the same generator the GPU arm drew them with."""
    from oracle import indexer as O
    from oracle.codecs import bf16_decode

    res = {}
    for b in rows:
        L = int(wl.pool.ctx_lens[b])
        if device is not None:
            kb = W.make_k_device(wl.seed, b, L, device).view(torch.int16).cpu().numpy().view(np.uint16)
        else:
            kb = W.make_k(wl.seed, b, L)
        res[b] = O.k_quant(bf16_decode(kb))
    return res


# ----------------------------------------------------------------------------- decode workloads

def decode_workload(name: str, rank: int) -> W.DecodeWorkload:
    if name == "long_decode":
        return W.long_decode(seed=1003 + 7919 * rank)
    if name == "paged_decode":
        return W.paged_decode(seed=1001 + 7919 * rank)
    raise ValueError(name)


def run_decode(args, rank, world, local, dist):
    import sparse_attention_indexer_fp8_gb300 as idx
    from sparse_attention_indexer_fp8_gb300.pipeline import fill_paged_cache

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = decode_workload(args.workload, rank)
    pool = wl.pool
    B = wl.batch
    L = pool.ctx_lens.astype(np.int64)
    stride = W.block_stride_bytes()
    cache = torch.zeros((pool.num_blocks, stride), dtype=torch.uint8, device=dev)
    fill_paged_cache(pool, wl.seed, cache, device_k=True)
    q = torch.from_numpy(wl.q8).to(dev)
    w = torch.from_numpy(wl.w).to(dev)
    bt = torch.from_numpy(pool.block_table).to(dev)
    ctx = torch.from_numpy(pool.ctx_lens).to(dev)
    # the new token of every request is its last position; its k comes from the same generator
    new_k = torch.stack([W.make_k_device(wl.seed, b, int(L[b]), dev)[-1] for b in range(B)])
    new_slots = torch.from_numpy(np.array([pool.slot_mapping(b)[-1] for b in range(B)])).to(dev)
    L_max = int(L.max())
    ld = (L_max + 63) // 64 * 64          # 256-byte aligned rows for the selection's vector loads
    logits = torch.empty((B, ld), dtype=torch.float32, device=dev)
    local_idx = torch.empty((B, wl.topk), dtype=torch.int32, device=dev)
    slots = torch.empty((B, wl.topk), dtype=torch.int32, device=dev)
    # selection workspace: the logits kernel histograms each row's first radix
    # digit, the top-k consumes and re-zeroes it
    ws = torch.zeros((B, 1024), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        idx.idx_k_quant_and_cache(new_k, new_slots, cache, pool.block_size, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        idx.idx_paged_mqa_logits_decode(q, w, cache, pool.block_size, bt, ctx, logits, ws=ws,
                                        stream=stream)
        if ev is not None:
            ev[1].record(stream)
        idx.idx_topk(logits, None, ctx, wl.topk, local_idx, ws=ws, stream=stream)
        idx.idx_req_to_global_slots(local_idx, None, bt, pool.block_size, wl.block_span, slots,
                                    stream=stream)

    launches_per_step = 4
    sampler = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    idx.idx_device_error(stream)
    # keep the GPU busy for a moment so the clock sampler sees it under load
    t_soak = time.time()
    while time.time() - t_soak < 1.0:
        for _ in range(20):
            step()
        torch.cuda.synchronize(dev)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(kev[i])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t1 = time.time()
    ms_total = e0.elapsed_time(e1)
    logits_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    idx.idx_device_error(stream)
    ms_total = max_over_ranks(dist, ms_total, dev)

    # end to end through the public API with host buffers: per step H2D of the
    # step's inputs from pinned memory, the step, D2H of the slot table
    h_q = torch.from_numpy(wl.q8).pin_memory()
    h_w = torch.from_numpy(wl.w).pin_memory()
    h_k = new_k.cpu().pin_memory()
    h_s = new_slots.cpu().pin_memory()
    h_ctx = torch.from_numpy(pool.ctx_lens).pin_memory()
    h_out = torch.empty((B, wl.topk), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_w, h_k, h_s, h_ctx))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        q.copy_(h_q, non_blocking=True)
        w.copy_(h_w, non_blocking=True)
        new_k.copy_(h_k, non_blocking=True)
        new_slots.copy_(h_s, non_blocking=True)
        ctx.copy_(h_ctx, non_blocking=True)
        step()
        h_out.copy_(slots, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    barrier(dist)
    torch.cuda.synchronize(dev)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2e_ms = max_over_ranks(dist, a0.elapsed_time(a1), dev)
    if sampler:
        sampler.stop()
    if rank != 0:
        return None

    # parity on sampled rows (also the rows the CPU baseline times)
    rng = np.random.default_rng(wl.seed)
    sample = sorted(rng.choice(B, size=min(args.cpu_rows, B), replace=False).tolist())
    k_rows = oracle_k_rows(wl, sample, dev)
    cpu_s, ref = oracle_decode_rows(wl, sample, k_rows)
    from tests.checks import assert_logits_close, assert_topk_row

    g_logits = logits.cpu().numpy()
    g_sel = local_idx.cpu().numpy()
    g_slots = slots.cpu().numpy()
    for b in sample:
        lg, _, _ = ref[b]
        Lb = int(L[b])
        assert_logits_close(g_logits[b, :Lb], lg, f"bench logits row {b}")
        assert_topk_row(g_sel[b], lg, wl.topk, f"bench top-k row {b}")
        want = np.where(g_sel[b] >= 0, pool.slot_mapping(b)[np.clip(g_sel[b], 0, Lb - 1)], -1)
        assert np.array_equal(g_slots[b], want), f"bench slots row {b}"

    peaks, peak_kind = measured_peaks()
    rows_total = B * world
    value = rows_total / (ms_total / 1e3 / args.steps)
    tok = int(L.sum())
    logits_bytes = tok * (W.TOKEN_BYTES + 4) + B * (64 * 128 + 64 * 4)
    achieved = logits_bytes / (logits_ms / 1e3) / 1e9
    traffic = profiled_traffic(f"mqa_logits_decode_{args.workload}.md", "logits.cu")
    line = {
        "metric": "decode indexer query-rows/s @128K ctx incl. top-2048; % of HBM roofline"
        if args.workload == "long_decode" else f"{args.workload} indexer query-rows/s incl. top-2048",
        "value": round(value, 1),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3xe4m3->f32",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "batch": B, "ctx_min": int(L.min()), "ctx_max": int(L.max()),
            "ctx_mean": float(L.mean()), "topk": wl.topk, "block_size": pool.block_size,
            "block_stride_bytes": stride, "cache_gb": round(pool.num_blocks * stride / 1e9, 3),
            "step": "k insert + paged logits + top-2048 + slot conversion",
            "l2": "inputs larger than L2 (k cache > 129 MB), no flush",
            "parallelism": f"rows sharded, {world} independent replica(s)",
        },
        "roofline": {
            "kernel": "mqa_logits_kernel<1> (paged decode)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": logits_bytes, "traffic": traffic,
            "kernel_ms": round(logits_ms, 5),
            "step_kcache_frac": round(tok * W.TOKEN_BYTES / (ms_total / args.steps / 1e3) / 1e9
                                      / peaks["hbm_gbs"], 4),
        },
        "cpu_baseline": {
            "value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{len(sample)} full rows of this workload (logits over every visible token, "
                      f"top-2048, slots), cache prepared untimed",
        },
        "e2e": {"value": round(rows_total / (e2e_ms / 1e3 / args.steps), 1), "unit": "rows/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "parity": f"ok on {len(sample)} sampled rows",
    }
    return line


def run_reference(args, rank):
    """The oracle on the host cores, same workload/metric, bounded sample per step."""
    if rank != 0:
        return None
    wl = decode_workload(args.workload, 0)
    B = wl.batch
    rng = np.random.default_rng(wl.seed)
    pool_rows = sorted(rng.choice(B, size=min(4, B), replace=False).tolist())
    k_rows = oracle_k_rows(wl, pool_rows, None)
    per_step = 1
    for i in range(args.warmup):
        oracle_decode_rows(wl, [pool_rows[i % len(pool_rows)]], k_rows)
    t = 0.0
    for i in range(args.steps):
        s, _ = oracle_decode_rows(wl, [pool_rows[i % len(pool_rows)]], k_rows)
        t += s
    value = args.steps * per_step / t
    return {
        "impl": "reference",
        "metric": "decode indexer query-rows/s @128K ctx incl. top-2048; % of HBM roofline"
        if args.workload == "long_decode" else f"{args.workload} indexer query-rows/s incl. top-2048",
        "value": round(value, 3), "unit": "rows/s", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "batch": B, "topk": wl.topk},
        "cpu_baseline": {"value": round(value, 3), "unit": "rows/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"each step one full row (of {len(pool_rows)} prepared rows)"},
        "e2e": {"value": round(value, 3), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_decode",
                    choices=["long_decode", "paged_decode"])
    ap.add_argument("--cpu-rows", type=int, default=12)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, rank)
    else:
        rank, world, local, dist = dist_setup(args.gpus)
        line = run_decode(args, rank, world, local, dist)
        if dist is not None:
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
