#!/usr/bin/env python
"""Benchmark of the FP8 lightning indexer on one GB300 (or N, one process per GPU).

Default workload: the 128K long-context decode step - batch 128, contexts
uniform in [64K, 128K] in a 1.7 GB paged k cache (block 64, 8704-byte blocks,
shuffled block tables). One step is the whole decode path: insert the new
token's k (fused quantisation), paged FP8 MQA logits over every visible
token, top-2048 per row, request-local -> physical slot conversion.
``value`` is query rows per second with every input resident in HBM; the k
cache (1.7 GB) is larger than L2, so no flush is needed between steps.

Other workloads (``--workload``): ``long_decode_mxfp4`` (the same step on the
MXFP4 indexer cache), ``paged_decode`` (batch 64, 8K-32K), ``prefill`` (8192
queries on a 32K context), ``hierarchical`` and ``hierarchical_mxfp4`` (V4.1
sparse decode at 128K), ``hierarchical_mtp`` (next_n 2, four consumer layers
per expansion), ``dcp_decode`` (four context-parallel ranks emulated on one
GPU) and ``q_prep`` (RoPE + q quantisation of an 8192-query chunk).

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


def hbm_roofline(kernel: str, alg_bytes: int, out_bytes: int, kernel_ms: float, peaks, peak_kind: str,
                 traffic=None, **extra):
    """Roofline of an HBM-bound scoring launch.

    ``frac`` counts the bytes the method has to read (the k cache records, q and
    the weights); the score write, which a fused selection would not need, is
    reported beside it (``output_bytes_per_launch``, ``frac_incl_output``).
    """
    sec = kernel_ms / 1e3
    ach = alg_bytes / sec / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": int(alg_bytes), "output_bytes_per_launch": int(out_bytes),
            "frac_incl_output": round((alg_bytes + out_bytes) / sec / 1e9 / peaks["hbm_gbs"], 4),
            "traffic": traffic, "kernel_ms": round(kernel_ms, 5), **extra}


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


def measure_mma_rate(kind: int, seconds: float, device_index: int, stream):
    """The dense tensor-core rate of this GPU, measured with the library's own diagnostic.

    ``idx_diag_mma_peak`` keeps every SM issuing 128 x 256 x K tcgen05.mma from
    shared-memory operands (kind 0: e4m3 kind::f8f6f4, 1: bf16 kind::f16). One
    launch of ~10 ms is timed alone with CUDA events (burst); then launches run
    back to back for ``seconds`` and the last half is timed (sustained), with
    nvidia-smi clock samples taken meanwhile.
    """
    import ctypes

    import sparse_attention_indexer_fp8_gb300 as idx

    lib = idx.library()
    flop = ctypes.c_double(0.0)
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def launch(iters):
        st = lib.idx_diag_mma_peak(kind, iters, 0, ctypes.byref(flop), sptr)
        if st != 0:
            raise RuntimeError(lib.idx_last_error().decode())
        return flop.value

    def timed(iters, reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        f = sum(launch(iters) for _ in range(reps))
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        return f / (ms / 1e3) / 1e12, ms

    timed(2000, 1)                                   # warm-up
    _, probe_ms = timed(20000, 1)
    iters = max(1000, int(20000 * 10.0 / max(probe_ms, 1e-3)))   # one launch of about 10 ms
    burst, _ = timed(iters, 1)
    reps = max(1, int(seconds / 2 / 0.01))
    sampler = ClockSampler(device_index)
    t0 = time.time()
    timed(iters, reps)
    sustained, _ = timed(iters, reps)
    t1 = time.time()
    sampler.stop()
    idx.idx_device_error()
    return {"burst_tflops": round(burst, 1), "sustained_tflops": round(sustained, 1),
            "clocks": sampler.summary(t0, t1),
            "how": ("own tcgen05.mma kind::" + ("f8f6f4 e4m3" if kind == 0 else "f16 bf16") +
                    ", 128x256xK from shared memory on every SM, CUDA events; burst = one ~10 ms launch, "
                    f"sustained = the second half of {seconds:.1f} s of back-to-back launches")}


def l2_stream(nbytes: int, kernel_ms: float, what: str):
    """A kernel's L2-resident read bytes per launch against the L2 read rate measured now."""
    peak = measure_l2_read()
    ach = nbytes / (kernel_ms / 1e3) / 1e9
    return {"achieved_gbs": round(ach, 1), "peak_gbs": peak["gbs"], "frac": round(ach / peak["gbs"], 4),
            "bytes_per_launch": int(nbytes), "bytes": what, "peak_source": peak["how"]}


def measure_l2_read(mb: int = 64, passes: int = 40):
    """The rate at which every SM together reads a buffer that L2 holds.

    ``idx_diag_l2_read`` (the library's own diagnostic) has one 1024-thread CTA
    per SM read one chunk of a 64 MB buffer (half of L2 at most) per pass, a
    different chunk each pass, with 16-byte loads that bypass L1; one warm-up
    launch brings the buffer into L2, then one launch of ``passes`` passes is
    timed with CUDA events.
    """
    import ctypes

    import sparse_attention_indexer_fp8_gb300 as idx

    lib = idx.library()
    stream = torch.cuda.current_stream()
    sptr = ctypes.c_void_p(stream.cuda_stream)
    buf = torch.ones(mb << 20, dtype=torch.uint8, device="cuda")

    def launch(n):
        st = lib.idx_diag_l2_read(ctypes.c_void_p(buf.data_ptr()), buf.numel(), n, 0, sptr)
        if st != 0:
            raise RuntimeError(lib.idx_last_error().decode())

    launch(2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    launch(passes)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    gbs = buf.numel() * passes / (ms / 1e3) / 1e9
    del buf
    return {"gbs": round(gbs, 1), "how": f"own diagnostic: every SM reads a different chunk of a {mb} MB buffer "
                                         f"that L2 holds in each of {passes} passes of one launch, 16-byte loads "
                                         f"past L1, CUDA events"}


def measure_cublas_fp8(device_index: int, n: int = 8192, reps: int = 10):
    """Dense e4m3 GEMM rate of the vendor library on this GPU (torch._scaled_mm, n^3, best of reps).

    A measurement only (the library GEMM is the yardstick for the FP8 tensor peak);
    clock samples are taken while it runs.
    """
    dev = torch.device("cuda", device_index)
    a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    one = torch.ones((), device=dev)
    mm = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)  # noqa: E731
    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    sampler = ClockSampler(device_index)
    t0 = time.time()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    t1 = time.time()
    sampler.stop()
    del a, b
    return {"tflops": round(2.0 * n ** 3 / (best / 1e3) / 1e12, 1), "clocks": sampler.summary(t0, t1),
            "how": f"torch._scaled_mm e4m3 x e4m3 -> bf16, {n}^3, best of {reps}, CUDA events"}


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


def rank_seed(base: int, rank: int) -> int:
    """Seed of rank `rank`'s own batch: ranks work on independent rows (weak scaling)."""
    return base + 7919 * rank


# ----------------------------------------------------------------------------- oracle side

def oracle_decode_rows(wl: W.DecodeWorkload, rows, k_rows, reps: int = 1, kv: str = "fp8"):
    """Time the oracle's decode step (new-token insert, logits, top-k, slots) on sample rows.

    ``k_rows[b]`` = (k8, kscale) of request b, or its MXFP4 k values, prepared
    beforehand (the cache is state, not per-step work). Returns (seconds, per-row results).
    """
    from oracle import indexer as O

    out = {}
    t0 = time.perf_counter()
    for _ in range(reps):
        for b in rows:
            L = int(wl.pool.ctx_lens[b])
            if kv == "mxfp4":
                O.mxfp4_quant(np.zeros((1, 128), dtype=np.float32))  # the new token's insert
                lg = O.logits_row_values(wl.q8[b], wl.w[b], k_rows[b])
            else:
                k8, ks = k_rows[b]
                O.k_quant(np.zeros((1, 128), dtype=np.float32))      # the new token's insert
                lg = O.logits_row(wl.q8[b], wl.w[b], k8, ks)
            sel = O.topk_row(lg, 0, L, wl.topk)
            sl = O.req_to_global_slots(sel[None], None, wl.pool.block_table[b:b + 1],
                                       wl.pool.block_size, wl.block_span)
            out[b] = (lg, sel, sl[0])
    return time.perf_counter() - t0, out


def oracle_k_rows(wl: W.DecodeWorkload, rows, device, kv: str = "fp8"):
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
        kf = bf16_decode(kb)
        res[b] = O.mxfp4_values(*O.mxfp4_quant(kf)) if kv == "mxfp4" else O.k_quant(kf)
    return res


# ----------------------------------------------------------------------------- workloads

def _pin(a):
    t = a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
    return t.contiguous().pin_memory()


def _nbytes(*ts):
    return int(sum(t.numel() * t.element_size() for t in ts))


def _pin_like(d):
    return torch.empty(d.shape, dtype=d.dtype).pin_memory()


class E2EPipeline:
    """End-to-end steps through the public API with host buffers, two steps in flight.

    Every step copies all of its inputs from pinned host memory to the device and
    its result back. The inputs sit back to back (256-byte aligned) in one pinned
    staging buffer and move in one host-to-device copy per step into one of two
    device buffer sets; the results move back in one device-to-host copy. The
    host-to-device copy of step i + 1 (on its own stream) and the device-to-host
    copy of step i - 1 (on a third stream) overlap step i's kernels; events order
    each copy against the kernels that read or write the same buffer set. The
    bench's own device tensors are re-pointed (``Tensor.set_``) at views of the set
    a step uses, so its ``step`` runs unchanged."""

    ALIGN = 256

    def __init__(self, bench, dev):
        self.bench = bench
        self.inputs, self.outputs = bench.e2e_io()
        self.host_in, self.in_views = self._pack(self.inputs, dev, fill=True)
        self.host_out, self.out_views = self._pack(self.outputs, dev, fill=False)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.ev = {k: [torch.cuda.Event() for _ in range(2)]
                   for k in ("in_ready", "in_free", "out_ready", "out_free")}
        self.used = [False, False]
        self.i = 0

    def _pack(self, pairs, dev, fill):
        """One pinned host buffer and two device buffers holding every tensor of
        ``pairs`` at aligned offsets; per device buffer, a view shaped like each tensor."""
        offs, total = [], 0
        for h, _ in pairs:
            offs.append(total)
            total += (h.numel() * h.element_size() + self.ALIGN - 1) // self.ALIGN * self.ALIGN
        host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        if fill:
            for (h, _), o in zip(pairs, offs):
                n = h.numel() * h.element_size()
                host[o:o + n].copy_(h.contiguous().reshape(-1).view(torch.uint8))
        sets = []
        for _ in range(2):
            buf = torch.zeros(total, dtype=torch.uint8, device=dev)
            views = [buf[o:o + d.numel() * d.element_size()].view(d.dtype).view(d.shape)
                     for (_, d), o in zip(pairs, offs)]
            sets.append((buf, views))
        return host, sets

    def bytes_per_step(self):
        return self.host_in.numel(), self.host_out.numel()

    def begin(self, stream):
        """Forks the copy streams from ``stream`` (required inside a graph capture)."""
        fork = torch.cuda.Event()
        fork.record(stream)
        self.h2d.wait_event(fork)
        self.d2h.wait_event(fork)
        self.used = [False, False]
        self.i = 0

    def step(self, stream):
        s, ev = self.i % 2, self.ev
        buf_in, views_in = self.in_views[s]
        buf_out, views_out = self.out_views[s]
        with torch.cuda.stream(self.h2d):
            if self.used[s]:
                self.h2d.wait_event(ev["in_free"][s])      # the kernels of step i - 2 are done with set s
            buf_in.copy_(self.host_in, non_blocking=True)
            ev["in_ready"][s].record(self.h2d)
        stream.wait_event(ev["in_ready"][s])
        if self.used[s]:
            stream.wait_event(ev["out_free"][s])          # step i - 2's result has left set s
        for (_, d), v in zip(self.inputs, views_in):
            d.set_(v)
        for (_, d), v in zip(self.outputs, views_out):
            d.set_(v)
        self.bench.step(stream)
        ev["in_free"][s].record(stream)
        ev["out_ready"][s].record(stream)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(ev["out_ready"][s])
            self.host_out.copy_(buf_out, non_blocking=True)
            ev["out_free"][s].record(self.d2h)
        self.used[s] = True
        self.i += 1

    def end(self, stream):
        """Joins the copy streams back into ``stream``."""
        for side in (self.h2d, self.d2h):
            j = torch.cuda.Event()
            j.record(side)
            stream.wait_event(j)


class DecodeBench:
    """Dense paged decode: k insert of the new token, logits, top-2048 with the slot conversion."""

    launches_per_step = 3

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx
        from sparse_attention_indexer_fp8_gb300.pipeline import fill_paged_cache

        self.idx, self.dev, self.name = idx, dev, name
        # the MXFP4 line runs the same long-context workload (same k) on the MXFP4 indexer cache
        self.kv = "mxfp4" if name.endswith("_mxfp4") else "fp8"
        self.wl = wl = (W.long_decode(seed=rank_seed(1003, rank)) if name.startswith("long_decode")
                        else W.paged_decode(seed=rank_seed(1001, rank)))
        pool = wl.pool
        self.B = B = wl.batch
        self.L = L = pool.ctx_lens.astype(np.int64)
        self.token_bytes = W.MXFP4_TOKEN_BYTES if self.kv == "mxfp4" else W.TOKEN_BYTES
        self.stride = W.mxfp4_block_stride_bytes() if self.kv == "mxfp4" else W.block_stride_bytes()
        self.cache = torch.zeros((pool.num_blocks, self.stride), dtype=torch.uint8, device=dev)
        fill_paged_cache(pool, wl.seed, self.cache, device_k=True, kv=self.kv)
        self.insert = idx.idx_k_quant_and_cache_mxfp4 if self.kv == "mxfp4" else idx.idx_k_quant_and_cache
        self.scorer = (idx.idx_paged_mqa_logits_decode_mxfp4 if self.kv == "mxfp4"
                       else idx.idx_paged_mqa_logits_decode)
        self.q = torch.from_numpy(wl.q8).to(dev)
        self.w = torch.from_numpy(wl.w).to(dev)
        self.bt = torch.from_numpy(pool.block_table).to(dev)
        self.ctx = torch.from_numpy(pool.ctx_lens).to(dev)
        # the new token of every request is its last position; its k comes from the same generator
        self.new_k = torch.stack([W.make_k_device(wl.seed, b, int(L[b]), dev)[-1] for b in range(B)])
        self.new_slots = torch.from_numpy(np.array([pool.slot_mapping(b)[-1] for b in range(B)])).to(dev)
        ld = (int(L.max()) + 63) // 64 * 64      # 256-byte aligned rows for the selection's vector loads
        self.logits = torch.empty((B, ld), dtype=torch.float32, device=dev)
        self.local = torch.empty((B, wl.topk), dtype=torch.int32, device=dev)
        self.slots = torch.empty((B, wl.topk), dtype=torch.int32, device=dev)
        # No selection workspace: without the first-digit histogram the scoring
        # kernel holds a fifth k stage, which saves more (128K: 265.3 -> 259.1 us)
        # than the selection's own first-digit sweep costs (step 282.3 -> 281.3 us)
        self.ws = None
        self.rows_per_step = B

    metric = property(lambda self: "decode indexer query-rows/s @128K ctx incl. top-2048; % of HBM roofline"
                      if self.name == "long_decode" else
                      ("decode indexer query-rows/s @128K ctx incl. top-2048, MXFP4 indexer cache"
                       if self.name == "long_decode_mxfp4" else "paged decode indexer query-rows/s incl. top-2048"))

    def step(self, stream, ev=None):
        idx, wl = self.idx, self.wl
        self.insert(self.new_k, self.new_slots, self.cache, wl.pool.block_size, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        self.scorer(self.q, self.w, self.cache, wl.pool.block_size, self.bt, self.ctx, self.logits, ws=self.ws,
                    stream=stream)
        if ev is not None:
            ev[1].record(stream)
        # top-2048 with the slot conversion fused into the selection's output pass
        idx.idx_topk(self.logits, None, self.ctx, wl.topk, self.local, ws=self.ws, stream=stream,
                     slots=self.slots, block_table=self.bt, block_size=wl.pool.block_size,
                     block_span=wl.block_span)

    def e2e_io(self):
        """(pinned host, device) pairs of a step's inputs and of its result."""
        inputs = [(_pin(self.wl.q8), self.q), (_pin(self.wl.w), self.w), (self.new_k.cpu().pin_memory(),
                  self.new_k), (self.new_slots.cpu().pin_memory(), self.new_slots),
                  (_pin(self.wl.pool.ctx_lens), self.ctx)]
        return inputs, [(_pin_like(self.slots), self.slots)]

    def verify_and_time_oracle(self, n_rows):
        from tests.checks import assert_logits_close, assert_topk_row

        wl, L = self.wl, self.L
        rng = np.random.default_rng(wl.seed)
        sample = sorted(rng.choice(self.B, size=min(n_rows, self.B), replace=False).tolist())
        k_rows = oracle_k_rows(wl, sample, self.dev, self.kv)
        cpu_s, ref = oracle_decode_rows(wl, sample, k_rows, kv=self.kv)
        g_logits, g_sel, g_slots = self.logits.cpu().numpy(), self.local.cpu().numpy(), self.slots.cpu().numpy()
        for b in sample:
            lg = ref[b][0]
            Lb = int(L[b])
            assert_logits_close(g_logits[b, :Lb], lg, f"bench logits row {b}")
            assert_topk_row(g_sel[b], lg, wl.topk, f"bench top-k row {b}")
            want = np.where(g_sel[b] >= 0, wl.pool.slot_mapping(b)[np.clip(g_sel[b], 0, Lb - 1)], -1)
            assert np.array_equal(g_slots[b], want), f"bench slots row {b}"
        cpu = {"value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{len(sample)} full rows of this workload (logits over every "
                                           f"visible token, top-2048, slots), cache prepared untimed"}
        return cpu, f"ok on {len(sample)} sampled rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        tok = int(self.L.sum())
        tb = self.token_bytes
        return hbm_roofline("mqa_logits_kernel<1, MXFP4 k> (paged decode)" if self.kv == "mxfp4"
                            else "mqa_logits_kernel<1> (paged decode)", tok * tb + self.B * (64 * 128 + 64 * 4),
                            tok * 4, kernel_ms, peaks, peak_kind,
                            # the committed e4m3 counters are of this launch (no workspace, five k
                            # stages); the MXFP4 ones were taken with the workspace histogram
                            traffic=(None if self.kv == "mxfp4" else
                                     profiled_traffic(f"mqa_logits_decode_{self.name}.md", "logits.cu")),
                            step_kcache_frac=round(tok * tb / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4))

    def config(self, world):
        L, pool = self.L, self.wl.pool
        return {"workload": self.wl.name + ("-mxfp4-cache" if self.kv == "mxfp4" else ""), "batch": self.B,
                "ctx_min": int(L.min()), "ctx_max": int(L.max()),
                "ctx_mean": float(L.mean()), "topk": self.wl.topk, "block_size": pool.block_size,
                "kv_cache": "MXFP4 (e2m1 + E8M0 per 32, 68 B/token)" if self.kv == "mxfp4"
                else "e4m3 + fp32 scale (132 B/token)",
                "block_stride_bytes": self.stride, "cache_gb": round(pool.num_blocks * self.stride / 1e9, 3),
                "step": "k insert + paged logits + top-2048 with the slot conversion fused",
                "l2": "inputs larger than L2 (k cache > 129 MB), no flush",
                "parallelism": f"rows sharded, {world} independent replica(s)"}

    dtype = property(lambda self: "e4m3xe2m1(mx)->f32" if self.kv == "mxfp4" else "e4m3xe4m3->f32")


class PrefillBench:
    """Prefill chunk: insert the chunk's k, gather the context, causal logits, top-2048 per row."""

    launches_per_step = 4
    dtype = "e4m3xe4m3->f32"
    metric = "prefill indexer query-rows/s incl. top-2048 (8192-query chunk of a 32K context)"

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx

        self.idx, self.dev, self.name = idx, dev, name
        self.wl = wl = W.prefill_chunk(seed=rank_seed(1002, rank))
        self.T, self.S = T, S = wl.q8.shape[0], wl.S
        self.pool = pool = W.make_pool(wl.seed, [S])
        self.stride = W.block_stride_bytes()
        self.cache = torch.zeros((pool.num_blocks, self.stride), dtype=torch.uint8, device=dev)
        k = W.make_k_device(wl.seed, 0, S, dev)
        sm = torch.from_numpy(pool.slot_mapping(0)).to(dev)
        # the context before the chunk is state; the chunk's own k is inserted every step
        idx.idx_k_quant_and_cache(k[:S - T], sm[:S - T], self.cache, pool.block_size)
        self.chunk_k, self.chunk_slots = k[S - T:].contiguous(), sm[S - T:].contiguous()
        self.bt_row = torch.from_numpy(pool.block_table[0]).to(dev)
        self.k8 = torch.empty((S, 128), dtype=torch.uint8, device=dev)
        self.kscale = torch.empty(S, dtype=torch.float32, device=dev)
        self.q = torch.from_numpy(wl.q8).to(dev)
        self.w = torch.from_numpy(wl.w.view(np.int16)).to(dev).view(torch.bfloat16)
        self.ks = torch.from_numpy(wl.row_ks).to(dev)
        self.ke = torch.from_numpy(wl.row_ke).to(dev)
        self.logits = torch.empty((T, (S + 63) // 64 * 64), dtype=torch.float32, device=dev)
        self.local = torch.empty((T, wl.topk), dtype=torch.int32, device=dev)
        self.rows_per_step = T

    def step(self, stream, ev=None):
        idx = self.idx
        idx.idx_k_quant_and_cache(self.chunk_k, self.chunk_slots, self.cache, self.pool.block_size, stream=stream)
        idx.idx_gather_k(self.cache, self.pool.block_size, self.bt_row, self.S, self.k8, self.kscale, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        idx.idx_mqa_logits_prefill(self.q, self.w, self.k8, self.kscale, self.ks, self.ke, self.logits,
                                   stream=stream)
        if ev is not None:
            ev[1].record(stream)
        idx.idx_topk(self.logits, self.ks, self.ke, self.wl.topk, self.local, stream=stream)

    def e2e_io(self):
        inputs = [(_pin(self.wl.q8), self.q), (self.w.cpu().pin_memory(), self.w),
                  (self.chunk_k.cpu().pin_memory(), self.chunk_k),
                  (self.chunk_slots.cpu().pin_memory(), self.chunk_slots)]
        return inputs, [(_pin_like(self.local), self.local)]

    def _oracle_k(self):
        from oracle import indexer as O
        from oracle.codecs import bf16_decode

        kb = W.make_k_device(self.wl.seed, 0, self.S, self.dev).view(torch.int16).cpu().numpy().view(np.uint16)
        return O.k_quant(bf16_decode(kb))

    def verify_and_time_oracle(self, n_rows):
        from oracle import indexer as O
        from oracle.codecs import bf16_decode
        from tests.checks import assert_logits_close, assert_topk_row

        wl = self.wl
        k8, ks = self._oracle_k()
        rng = np.random.default_rng(wl.seed)
        sample = sorted(set([0, self.T - 1] + rng.choice(self.T, size=max(n_rows - 2, 0), replace=False).tolist()))
        wv = bf16_decode(wl.w)
        g_logits, g_sel = self.logits.cpu().numpy(), self.local.cpu().numpy()
        t0 = time.perf_counter()
        ref = {}
        for t in sample:
            lo, hi = int(wl.row_ks[t]), int(wl.row_ke[t])
            lg = O.logits_row(wl.q8[t], wv[t], k8[lo:hi], ks[lo:hi])
            ref[t] = (lg, O.topk_row(lg, 0, hi - lo, wl.topk))
        cpu_s = time.perf_counter() - t0
        for t in sample:
            lo, hi = int(wl.row_ks[t]), int(wl.row_ke[t])
            assert_logits_close(g_logits[t, lo:hi], ref[t][0], f"bench prefill row {t}")
            assert np.all(np.isneginf(g_logits[t, hi:self.S])), f"bench prefill mask row {t}"
            assert_topk_row(g_sel[t], ref[t][0], wl.topk, f"bench prefill top-k row {t}")
        cpu = {"value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{len(sample)} full query rows of the chunk (logits over the "
                                           f"visible context, top-2048), k prepared untimed"}
        return cpu, f"ok on {len(sample)} sampled rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        pairs = int((self.wl.row_ke - self.wl.row_ks).astype(np.int64).sum())
        flop = pairs * 2 * 64 * 128
        ach = flop / (kernel_ms / 1e3) / 1e12
        derived = peaks["bf16_tflops"] * 2.0
        # the FP8 dense peak measured in this run: the vendor library's e4m3 GEMM; the
        # library's own single-CTA tcgen05 issue rate (128x256 MMAs from shared memory,
        # the shape this kernel issues) is reported beside it as the ceiling of that shape
        dev_i = torch.cuda.current_device()
        lib_fp8 = measure_cublas_fp8(dev_i)
        own_fp8 = measure_mma_rate(0, 2.0, dev_i, torch.cuda.current_stream())
        own_bf16 = measure_mma_rate(1, 1.0, dev_i, torch.cuda.current_stream())
        peak = max(lib_fp8["tflops"], own_fp8["burst_tflops"])
        return {"kernel": "mqa_logits_kernel<4> (prefill, causal)", "bound": "tensor",
                "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "peak_source": "measured in this run: the larger of the e4m3 library GEMM and the "
                               "library's own tcgen05 issue-rate diagnostic (see fp8_peak_measurements)",
                "fp8_peak_measurements": {"library_gemm": lib_fp8, "own_single_cta_mma": own_fp8,
                                          "own_single_cta_mma_bf16": own_bf16},
                "frac_of_single_cta_mma_ceiling": round(ach / own_fp8["burst_tflops"], 4),
                "frac_of_2x_measured_bf16_cublas": round(ach / derived, 4),
                "algorithmic_flop_per_launch": flop,
                "traffic": profiled_traffic("mqa_logits_prefill_prefill.md", "logits.cu"),
                "kernel_ms": round(kernel_ms, 5)}

    def config(self, world):
        return {"workload": self.wl.name, "queries": self.T, "ctx": self.S, "topk": self.wl.topk,
                "weights": "bf16", "causal_pairs": int((self.wl.row_ke - self.wl.row_ks).sum()),
                "step": "chunk k insert + gather + causal logits + top-2048",
                "l2": "logits output 1 GB > L2, no flush",
                "parallelism": f"chunks sharded, {world} independent replica(s)"}


class SparsePrefillBench:
    """V4.1 sparse prefill chunk: insert the chunk's k, gather the context, expand each row's
    candidate blocks, score the candidate sparse blocks (bf16), top-2048 + remap per row.

    The 8192-query chunk of a 32K context (the dense prefill workload), each row
    with 64 candidate 64-token blocks drawn over the context (duplicates, -1 and
    out-of-range ids included; blocks past the row's causal limit are dropped by
    the expansion). ``prefill_sparse_mxfp4`` runs it on the MXFP4 indexer cache,
    the cache of the V4.1 path (gather of the 68-byte records, fp8 x fp4 scores)."""

    launches_per_step = 5

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx

        self.idx, self.dev, self.name = idx, dev, name
        self.kv = "mxfp4" if name.endswith("_mxfp4") else "fp8"
        self.wl = wl = W.prefill_chunk(seed=rank_seed(1006, rank))
        self.T, self.S = T, S = wl.q8.shape[0], wl.S
        self.pool = pool = W.make_pool(wl.seed, [S])
        self.stride = W.mxfp4_block_stride_bytes() if self.kv == "mxfp4" else W.block_stride_bytes()
        self.cache = torch.zeros((pool.num_blocks, self.stride), dtype=torch.uint8, device=dev)
        self.insert = idx.idx_k_quant_and_cache_mxfp4 if self.kv == "mxfp4" else idx.idx_k_quant_and_cache
        k = W.make_k_device(wl.seed, 0, S, dev)
        sm = torch.from_numpy(pool.slot_mapping(0)).to(dev)
        # the context before the chunk is state; the chunk's own k is inserted every step
        self.insert(k[:S - T], sm[:S - T], self.cache, pool.block_size)
        self.chunk_k, self.chunk_slots = k[S - T:].contiguous(), sm[S - T:].contiguous()
        self.bt_row = torch.from_numpy(pool.block_table[0]).to(dev)
        if self.kv == "mxfp4":
            self.codes = torch.empty((S, 64), dtype=torch.uint8, device=dev)
            self.scales = torch.empty((S,), dtype=torch.int32, device=dev)
        else:
            self.k8 = torch.empty((S, 128), dtype=torch.uint8, device=dev)
            self.kscale = torch.empty(S, dtype=torch.float32, device=dev)
        self.q = torch.from_numpy(wl.q8).to(dev)
        self.w = torch.from_numpy(wl.w.view(np.int16)).to(dev).view(torch.bfloat16)
        self.ks = torch.from_numpy(wl.row_ks).to(dev)
        self.ke = torch.from_numpy(wl.row_ke).to(dev)
        self.h_cand = W.make_candidates(wl.seed, T, 64, S // 64)
        self.cand = torch.from_numpy(self.h_cand).to(dev)
        self.sbk = 64
        self.si = torch.empty((T, 64), dtype=torch.int32, device=dev)
        self.end = torch.empty(T, dtype=torch.int32, device=dev)
        self.logits = torch.empty((T, 64 * self.sbk), dtype=torch.bfloat16, device=dev)
        # rows this short are selected without the first-digit histogram: no workspace
        wsb = idx.idx_workspace_bytes("sparse_topk_remap", T, 64 * self.sbk, wl.topk)
        self.ws = torch.zeros((T, 1024), dtype=torch.int32, device=dev) if wsb else None
        self.pos = torch.empty((T, wl.topk), dtype=torch.int32, device=dev)
        self.cols = torch.empty((T, wl.topk), dtype=torch.int32, device=dev)
        self.rows_per_step = T

    metric = property(lambda self: "V4.1 sparse prefill indexer query-rows/s incl. top-2048 (8192-query chunk "
                      "of a 32K context, 64 candidate 64-token blocks per row" +
                      (", MXFP4 indexer cache)" if self.kv == "mxfp4" else ")"))
    dtype = property(lambda self: ("e4m3xe2m1(mx)" if self.kv == "mxfp4" else "e4m3xe4m3") + "->f32 (bf16 logits)")

    def step(self, stream, ev=None):
        idx, bs = self.idx, self.pool.block_size
        self.insert(self.chunk_k, self.chunk_slots, self.cache, bs, stream=stream)
        if self.kv == "mxfp4":
            idx.idx_gather_k_mxfp4(self.cache, bs, self.bt_row, self.S, self.codes, self.scales, stream=stream)
        else:
            idx.idx_gather_k(self.cache, bs, self.bt_row, self.S, self.k8, self.kscale, stream=stream)
        idx.idx_expand_candidates(self.cand, self.ks, self.ke, 64, self.sbk, self.si, self.end, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        if self.kv == "mxfp4":
            idx.idx_mqa_logits_prefill_mxfp4(self.q, self.w, self.codes, self.scales, self.logits, self.si,
                                             self.end, self.sbk, ws=self.ws, stream=stream)
        else:
            idx.idx_mqa_logits_prefill(self.q, self.w, self.k8, self.kscale, self.ks, self.ke, self.logits,
                                       sparse_idx=self.si, end=self.end, sbk=self.sbk, ws=self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        idx.idx_sparse_topk_remap(self.logits, self.end, self.si, self.ks, self.sbk, self.wl.topk, self.pos,
                                  col_scratch=self.cols, ws=self.ws, stream=stream)

    def e2e_io(self):
        inputs = [(_pin(self.wl.q8), self.q), (self.w.cpu().pin_memory(), self.w),
                  (self.chunk_k.cpu().pin_memory(), self.chunk_k),
                  (self.chunk_slots.cpu().pin_memory(), self.chunk_slots), (_pin(self.h_cand), self.cand)]
        return inputs, [(_pin_like(self.pos), self.pos)]

    def _oracle_k(self):
        """The context's k as the oracle quantises it: (k8, kscale), or MXFP4 (packed codes, scale codes)."""
        from oracle import indexer as O
        from oracle.codecs import bf16_decode

        kb = W.make_k_device(self.wl.seed, 0, self.S, self.dev).view(torch.int16).cpu().numpy().view(np.uint16)
        kf = bf16_decode(kb)
        if self.kv == "mxfp4":
            codes, scales = O.mxfp4_quant(kf)
            return O.mxfp4_pack(codes), scales
        return O.k_quant(kf)

    def verify_and_time_oracle(self, n_rows):
        from oracle import indexer as O
        from oracle.codecs import bf16_decode
        from tests.checks import assert_logits_close, assert_topk_row

        wl, sbk = self.wl, self.sbk
        ka, kb = self._oracle_k()
        rng = np.random.default_rng(wl.seed)
        sample = sorted(set([0, self.T - 1] + rng.choice(self.T, size=max(n_rows - 2, 0), replace=False).tolist()))
        wv = bf16_decode(wl.w)
        g_si, g_end = self.si.cpu().numpy(), self.end.cpu().numpy()
        g_lg = self.logits.float().cpu().numpy()
        g_cols, g_pos = self.cols.cpu().numpy(), self.pos.cpu().numpy()
        t0 = time.perf_counter()
        ref = {}
        for t in sample:
            osi, oend = O.expand_candidates(self.h_cand[t:t + 1], wl.row_ks[t:t + 1], wl.row_ke[t:t + 1], 64, sbk)
            if self.kv == "mxfp4":
                lg = O.sparse_logits_prefill_mxfp4(wl.q8[t:t + 1], wv[t:t + 1], ka, kb, osi, oend, sbk)[0]
            else:
                lg = O.sparse_logits_prefill(wl.q8[t:t + 1], wv[t:t + 1], ka, kb, osi, oend, sbk)[0]
            cols, pos = O.sparse_topk_remap_row(lg, int(oend[0]), osi[0], int(wl.row_ks[t]), sbk, wl.topk)
            ref[t] = (osi[0], int(oend[0]), lg, pos)
        cpu_s = time.perf_counter() - t0
        for t in sample:
            osi, e, lg, _ = ref[t]
            assert np.array_equal(g_si[t], osi) and int(g_end[t]) == e, f"bench expansion row {t}"
            assert_logits_close(g_lg[t, :e], lg[:e], f"bench sparse prefill row {t}", bf16=True)
            assert np.all(np.isneginf(g_lg[t, e:])), f"bench sparse prefill mask row {t}"
            assert_topk_row(g_cols[t], lg[:e], wl.topk, f"bench sparse prefill top-k row {t}", bf16=True)
            m = min(wl.topk, e)
            want = O.sparse_remap_columns(g_cols[t, :m], osi, int(wl.row_ks[t]), sbk)
            assert np.array_equal(g_pos[t, :m], want) and np.all(g_pos[t, m:] == -1), f"bench remap row {t}"
        self.cols_sum = int(g_end.astype(np.int64).sum())
        cpu = {"value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{len(sample)} full query rows of the chunk (expansion, candidate "
                                           f"logits, top-2048 remap), k prepared untimed"}
        return cpu, f"ok on {len(sample)} sampled rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        cols = getattr(self, "cols_sum", None)
        if cols is None:
            cols = int(self.end.sum().item())
        flop = cols * 2 * 64 * 128
        ach = flop / (kernel_ms / 1e3) / 1e12
        dev_i = torch.cuda.current_device()
        lib_fp8 = measure_cublas_fp8(dev_i)
        peak = lib_fp8["tflops"]
        kern = "mqa_logits_kernel<1%s> (sparse prefill, bf16 out)" % (", MXFP4 k" if self.kv == "mxfp4" else "")
        return {"kernel": kern, "bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "peak_source": "measured in this run: the e4m3 library GEMM (an fp8 x fp4 product runs at "
                               "the fp8 rate)",
                "algorithmic_flop_per_launch": flop,
                "traffic": profiled_traffic("launches_prefill_sparse%s.md" % ("_mxfp4" if self.kv == "mxfp4" else ""),
                                            "logits.cu"),
                "kernel_ms": round(kernel_ms, 5),
                # what actually bounds it: every visible candidate column's k record comes out of L2
                "l2": l2_stream(cols * (68 if self.kv == "mxfp4" else 132), kernel_ms,
                                "one k record (%d B) out of L2 per visible candidate column per query row"
                                % (68 if self.kv == "mxfp4" else 132))}

    def config(self, world):
        return {"workload": self.wl.name + "-sparse" + ("-mxfp4-cache" if self.kv == "mxfp4" else ""),
                "queries": self.T, "ctx": self.S, "topk": self.wl.topk, "candidates": 64,
                "cand_block_size": 64, "sbk": self.sbk, "weights": "bf16",
                "kv_cache": "MXFP4 (e2m1 + E8M0 per 32, 68 B/token)" if self.kv == "mxfp4"
                else "e4m3 + fp32 scale (132 B/token)",
                "step": "chunk k insert + gather + expand + sparse logits (bf16) + top-2048 remap",
                "l2": "the gathered k (2-4 MB) stays in L2; q (64 MB) and the scores (64 MB) stream",
                "parallelism": f"chunks sharded, {world} independent replica(s)"}


class HierBench:
    """V4.1 consumer-layer decode: expand candidates, sparse logits (bf16), top-2048 + remap + slots.

    ``hierarchical_mxfp4`` runs the same workload on the MXFP4 indexer cache, the
    cache format of the V4.1 path."""

    launches_per_step = 3

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx
        from sparse_attention_indexer_fp8_gb300.pipeline import HierarchicalStep, fill_paged_cache

        self.idx, self.dev, self.name = idx, dev, name
        self.kv = "mxfp4" if name.endswith("_mxfp4") else "fp8"
        self.wl = wl = W.hierarchical(seed=rank_seed(1004, rank))
        pool = wl.pool
        self.B = B = len(pool.ctx_lens)
        self.token_bytes = W.MXFP4_TOKEN_BYTES if self.kv == "mxfp4" else W.TOKEN_BYTES
        self.stride = W.mxfp4_block_stride_bytes() if self.kv == "mxfp4" else W.block_stride_bytes()
        self.cache = torch.zeros((pool.num_blocks, self.stride), dtype=torch.uint8, device=dev)
        fill_paged_cache(pool, wl.seed, self.cache, device_k=True, kv=self.kv)
        self.scorer = (idx.idx_paged_mqa_logits_decode_mxfp4 if self.kv == "mxfp4"
                       else idx.idx_paged_mqa_logits_decode)
        self.q = torch.from_numpy(wl.q8).to(dev)
        self.w = torch.from_numpy(wl.w).to(dev)
        self.bt = torch.from_numpy(pool.block_table).to(dev)
        self.ctx = torch.from_numpy(pool.ctx_lens).to(dev)
        self.cand = torch.from_numpy(wl.cand).to(dev)
        self.st = HierarchicalStep(B, wl.cand.shape[1], wl.cand_block_size, wl.sbk, wl.topk, pool.block_size, dev,
                                   kv=self.kv)
        self.rows_per_step = B

    metric = property(lambda self: "hierarchical sparse decode indexer query-rows/s @128K ctx incl. top-2048" +
                      (", MXFP4 indexer cache" if self.kv == "mxfp4" else ""))
    dtype = property(lambda self: ("e4m3xe2m1(mx)" if self.kv == "mxfp4" else "e4m3xe4m3") + "->f32 (bf16 logits)")

    def step(self, stream, ev=None):
        idx, st, wl = self.idx, self.st, self.wl
        idx.idx_expand_candidates(self.cand, None, self.ctx, wl.cand_block_size, wl.sbk, st.sparse_idx, st.end,
                                  stream=stream)
        if ev is not None:
            ev[0].record(stream)
        self.scorer(self.q, self.w, self.cache, wl.pool.block_size, self.bt, self.ctx, st.logits,
                    sparse_idx=st.sparse_idx, end=st.end, sbk=wl.sbk, ws=st.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        idx.idx_sparse_topk_remap(st.logits, st.end, st.sparse_idx, None, wl.sbk, wl.topk, st.positions,
                                  col_scratch=st.cols, ws=st.ws, stream=stream, slots=st.slots,
                                  block_table=self.bt, block_size=wl.pool.block_size,
                                  block_span=wl.pool.block_size)

    def e2e_io(self):
        inputs = [(_pin(self.wl.q8), self.q), (_pin(self.wl.w), self.w), (_pin(self.wl.cand), self.cand),
                  (_pin(self.wl.pool.ctx_lens), self.ctx)]
        return inputs, [(_pin_like(self.st.slots), self.st.slots)]

    def verify_and_time_oracle(self, n_rows):
        from oracle import indexer as O
        from tests.checks import assert_logits_close, assert_topk_row

        wl, st = self.wl, self.st
        g_si, g_end = st.sparse_idx.cpu().numpy(), st.end.cpu().numpy()
        o_si, o_end = O.expand_candidates(wl.cand, None, wl.pool.ctx_lens, wl.cand_block_size, wl.sbk)
        assert np.array_equal(g_si, o_si) and np.array_equal(g_end, o_end), "bench expansion differs"
        rng = np.random.default_rng(wl.seed)
        sample = sorted(rng.choice(self.B, size=min(n_rows, self.B), replace=False).tolist())
        kq = {b: oracle_sparse_k(wl, b, o_si[b], int(o_end[b]), self.dev, self.kv) for b in sample}
        g_lg = st.logits.float().cpu().numpy()
        g_cols, g_pos, g_slots = st.cols.cpu().numpy(), st.positions.cpu().numpy(), st.slots.cpu().numpy()
        t0 = time.perf_counter()
        ref = {b: oracle_hier_row(wl, b, kq[b], self.kv) for b in sample}
        cpu_s = time.perf_counter() - t0
        for b in sample:
            lg, _, _ = ref[b]
            e = int(o_end[b])
            assert_logits_close(g_lg[b, :e], lg, f"bench sparse logits row {b}", bf16=True)
            assert np.all(np.isneginf(g_lg[b, e:])), f"bench sparse mask row {b}"
            assert_topk_row(g_cols[b], lg, wl.topk, f"bench sparse top-k row {b}", bf16=True)
            m = min(wl.topk, e)
            want = [O.sparse_column_token(o_si[b], int(c), wl.sbk) for c in g_cols[b, :m]]
            assert g_pos[b, :m].tolist() == want and np.all(g_pos[b, m:] == -1), f"bench remap row {b}"
            sm = wl.pool.slot_mapping(b)
            assert np.array_equal(g_slots[b], np.where(g_pos[b] >= 0, sm[np.clip(g_pos[b], 0, None)], -1))
        self.end_sum = int(o_end.sum())
        cpu = {"value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{len(sample)} full rows (expansion, candidate logits, top-2048 "
                                           f"remap, slots), candidate k prepared untimed"}
        return cpu, f"ok on {len(sample)} sampled rows; expansion exact on all {self.B} rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        end_sum = getattr(self, "end_sum", None)
        if end_sum is None:
            end_sum = int(self.st.end.sum().item())
        ncols = self.st.logits.shape[1]
        return hbm_roofline("mqa_logits_kernel<1%s> (sparse decode, bf16 out)" % (", MXFP4 k" if self.kv == "mxfp4" else ""),
                            end_sum * self.token_bytes + self.B * (64 * 128 + 64 * 4),
                            self.B * ncols * 2, kernel_ms, peaks, peak_kind,
                            traffic=(profiled_traffic("launches_hierarchical.md", "logits.cu")
                                     if self.kv == "fp8" else None))

    def config(self, world):
        return {"workload": self.wl.name + ("-mxfp4-cache" if self.kv == "mxfp4" else ""), "batch": self.B,
                "ctx": int(self.wl.pool.ctx_lens[0]),
                "kv_cache": "MXFP4 (e2m1 + E8M0 per 32, 68 B/token)" if self.kv == "mxfp4"
                else "e4m3 + fp32 scale (132 B/token)",
                "candidates": int(self.wl.cand.shape[1]), "cand_block_size": self.wl.cand_block_size,
                "sbk": self.wl.sbk, "topk": self.wl.topk,
                "step": "expand + sparse logits (bf16) + top-2048 remap with the slot conversion fused",
                "l2": "candidate blocks scattered over a 2.2 GB cache, no flush",
                "parallelism": f"rows sharded, {world} independent replica(s)"}


def oracle_sparse_k(wl, b, si_row, end, device, kv: str = "fp8"):
    """Quantised k of the tokens one hierarchical row scores, from the GPU arm's generator
    ((k8, kscale), or MXFP4 k values)."""
    from oracle import indexer as O
    from oracle.codecs import bf16_decode

    L = int(wl.pool.ctx_lens[b])
    if device is not None:
        kall = W.make_k_device(wl.seed, b, L, device).view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        kall = W.make_k(wl.seed, b, L)
    toks = np.array([O.sparse_column_token(si_row, c, wl.sbk) for c in range(end)], dtype=np.int64)
    kf = bf16_decode(kall[toks])
    return O.mxfp4_values(*O.mxfp4_quant(kf)) if kv == "mxfp4" else O.k_quant(kf)


def oracle_hier_row(wl, b, kq, kv: str = "fp8"):
    """The oracle's hierarchical step for one row: expand, score the candidates, select, remap, slots."""
    from oracle import indexer as O

    si, end = O.expand_candidates_row(wl.cand[b], 0, int(wl.pool.ctx_lens[b]), wl.cand_block_size, wl.sbk)
    if kv == "mxfp4":
        lg = O.logits_row_values(wl.q8[b], wl.w[b], kq[:end])
    else:
        k8, ks = kq
        lg = O.logits_row(wl.q8[b], wl.w[b], k8[:end], ks[:end])
    dense = np.full(si.shape[0] * wl.sbk, -np.inf)
    dense[:end] = lg
    cols, pos = O.sparse_topk_remap_row(dense, end, si, 0, wl.sbk, wl.topk)
    sl = O.req_to_global_slots(pos[None], None, wl.pool.block_table[b:b + 1], wl.pool.block_size,
                               wl.pool.block_size)
    return lg, pos, sl[0]


class HierMtpBench:
    """V4.1 consumer layers with multi-token prediction: one expansion shared by several layers."""

    next_n, layers = 2, 4
    launches_per_step = 1 + 2 * layers
    dtype = "e4m3xe4m3->f32 (bf16 logits)"
    metric = ("hierarchical sparse decode query-row-layers/s @128K ctx incl. top-2048 "
              "(next_n 2, one expansion per step shared by 4 consumer layers)")

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx
        from sparse_attention_indexer_fp8_gb300.pipeline import HierarchicalStep, fill_paged_cache

        self.idx, self.dev, self.name = idx, dev, name
        self.wl = wl = W.hierarchical_mtp(seed=rank_seed(1005, rank), next_n=self.next_n)
        pool = wl.pool
        self.B = B = len(pool.ctx_lens)
        self.rows = rows = B * self.next_n
        self.cache = torch.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=torch.uint8, device=dev)
        fill_paged_cache(pool, wl.seed, self.cache, device_k=True)
        # layer 0 uses the workload's q / weights, later layers their own draws
        qw = [(wl.q8, wl.w)] + [W.make_q(wl.seed + 17 * i, rows) for i in range(1, self.layers)]
        self.h_qw = qw
        self.q = [torch.from_numpy(a).to(dev) for a, _ in qw]
        self.w = [torch.from_numpy(b).to(dev) for _, b in qw]
        self.bt = torch.from_numpy(pool.block_table).to(dev)
        self.ctx = torch.from_numpy(pool.ctx_lens).to(dev)
        self.h_row_ke = np.array([int(pool.ctx_lens[r // self.next_n]) - self.next_n + r % self.next_n + 1
                                  for r in range(rows)], dtype=np.int32)
        self.row_ke = torch.from_numpy(self.h_row_ke).to(dev)
        self.cand = torch.from_numpy(wl.cand).to(dev)
        self.st = HierarchicalStep(rows, wl.cand.shape[1], wl.cand_block_size, wl.sbk, wl.topk, pool.block_size,
                                   dev, next_n=self.next_n)
        self.rows_per_step = rows * self.layers

    def step(self, stream, ev=None):
        self.st.expand(self.cand, self.ctx, self.row_ke, stream=stream)
        for i in range(self.layers):
            if ev is not None and i == 0:
                ev[0].record(stream)
            idx = self.idx
            st, wl = self.st, self.wl
            idx.idx_paged_mqa_logits_decode(self.q[i], self.w[i], self.cache, wl.pool.block_size, self.bt,
                                            self.ctx, st.logits, next_n=self.next_n, sparse_idx=st.sparse_idx,
                                            end=st.end, sbk=wl.sbk, ws=st.ws, stream=stream)
            if ev is not None and i == 0:
                ev[1].record(stream)
            idx.idx_sparse_topk_remap(st.logits, st.end, st.sparse_idx, None, wl.sbk, wl.topk, st.positions,
                                      col_scratch=st.cols, ws=st.ws, stream=stream, slots=st.slots,
                                      block_table=self.bt, block_size=wl.pool.block_size,
                                      block_span=wl.pool.block_size, row_to_req=st.row_to_req)

    def e2e_io(self):
        inputs = ([(_pin(a), d) for (a, _), d in zip(self.h_qw, self.q)] +
                  [(_pin(b), d) for (_, b), d in zip(self.h_qw, self.w)] +
                  [(_pin(self.wl.cand), self.cand), (_pin(self.wl.pool.ctx_lens), self.ctx),
                   (_pin(self.h_row_ke), self.row_ke)])
        return inputs, [(_pin_like(self.st.slots), self.st.slots)]

    def verify_and_time_oracle(self, n_rows):
        from oracle import indexer as O
        from tests.checks import assert_logits_close, assert_topk_row

        wl, st, nn = self.wl, self.st, self.next_n
        g_si, g_end = st.sparse_idx.cpu().numpy(), st.end.cpu().numpy()
        o_si, o_end = O.expand_candidates(wl.cand, None, self.h_row_ke, wl.cand_block_size, wl.sbk)
        assert np.array_equal(g_si, o_si) and np.array_equal(g_end, o_end), "bench expansion differs"
        q8, w = self.h_qw[-1]          # the buffers hold the last layer's results
        rng = np.random.default_rng(wl.seed)
        sample = sorted(rng.choice(self.rows, size=min(n_rows, self.rows), replace=False).tolist())
        g_lg = st.logits.float().cpu().numpy()
        g_cols, g_pos, g_slots = st.cols.cpu().numpy(), st.positions.cpu().numpy(), st.slots.cpu().numpy()
        kq = {r: oracle_sparse_k(wl, r // nn, o_si[r], int(o_end[r]), self.dev) for r in sample}
        t0 = time.perf_counter()
        ref = {}
        for r in sample:
            k8, ks = kq[r]
            e = int(o_end[r])
            lg = O.logits_row(q8[r], w[r], k8[:e], ks[:e])
            dense = np.full(o_si.shape[1] * wl.sbk, -np.inf)
            dense[:e] = lg
            cols, pos = O.sparse_topk_remap_row(dense, e, o_si[r], 0, wl.sbk, wl.topk)
            sl = O.req_to_global_slots(pos[None], np.array([r // nn]), wl.pool.block_table, wl.pool.block_size,
                                       wl.pool.block_size)
            ref[r] = (lg, sl[0])
        cpu_s = time.perf_counter() - t0
        for r in sample:
            lg, _ = ref[r]
            e = int(o_end[r])
            assert_logits_close(g_lg[r, :e], lg, f"bench mtp sparse logits row {r}", bf16=True)
            assert_topk_row(g_cols[r], lg, wl.topk, f"bench mtp top-k row {r}", bf16=True)
            m = min(wl.topk, e)
            want = [O.sparse_column_token(o_si[r], int(c), wl.sbk) for c in g_cols[r, :m]]
            assert g_pos[r, :m].tolist() == want and np.all(g_pos[r, m:] == -1), f"bench mtp remap row {r}"
            sm = wl.pool.slot_mapping(r // nn)
            assert np.array_equal(g_slots[r], np.where(g_pos[r] >= 0, sm[np.clip(g_pos[r], 0, None)], -1))
        self.end_sum = int(o_end.sum())
        cpu = {"value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{len(sample)} query rows of the last layer (candidate logits, "
                                           f"top-2048 remap, slots), candidate k prepared untimed"}
        return cpu, f"ok on {len(sample)} sampled rows; expansion exact on all {self.rows} rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        end_sum = getattr(self, "end_sum", None)
        if end_sum is None:
            end_sum = int(self.st.end.sum().item())
        ncols = self.st.logits.shape[1]
        return hbm_roofline("mqa_logits_kernel<1> (sparse decode, bf16 out, one layer)", end_sum * W.TOKEN_BYTES + self.rows * (64 * 128 + 64 * 4),
                            self.rows * ncols * 2, kernel_ms, peaks, peak_kind)

    def config(self, world):
        return {"workload": self.wl.name, "batch": self.B, "next_n": self.next_n, "query_rows": self.rows,
                "layers_per_step": self.layers, "ctx": int(self.wl.pool.ctx_lens[0]),
                "candidates": int(self.wl.cand.shape[1]), "sbk": self.wl.sbk, "topk": self.wl.topk,
                "step": "expand once + per layer: sparse logits (bf16) + top-2048 remap with the slot conversion fused",
                "l2": "candidate blocks scattered over a 2.2 GB cache, no flush",
                "e2e_result": "the last layer's slot table",
                "parallelism": f"rows sharded, {world} independent replica(s)"}


class DcpBench:
    """Context-parallel decode of the 128K workload, four ranks emulated on one GPU.

    Rank r owns the r-th quarter of every request's blocks (its block table and
    shard lengths); each rank scores its shard and keeps its local top-2048 with
    scores, written straight into its part of the all-gather buffer (on one GPU the
    exchange is the identity), and the merge selects the global top-2048.
    """

    world = 4
    launches_per_step = 2 * world + 1
    dtype = "e4m3xe4m3->f32"
    metric = "context-parallel decode indexer query-rows/s @128K ctx incl. top-2048 (4 ranks emulated)"

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx
        from sparse_attention_indexer_fp8_gb300.pipeline import fill_paged_cache

        self.idx, self.dev, self.name = idx, dev, name
        self.wl = wl = W.long_decode(seed=rank_seed(1003, rank))
        pool = wl.pool
        self.B = B = wl.batch
        bs, W_ = pool.block_size, self.world
        self.cache = torch.zeros((pool.num_blocks, W.block_stride_bytes()), dtype=torch.uint8, device=dev)
        fill_paged_cache(pool, wl.seed, self.cache, device_k=True)
        self.q = torch.from_numpy(wl.q8).to(dev)
        self.w = torch.from_numpy(wl.w).to(dev)
        L = pool.ctx_lens.astype(np.int64)
        nblk = (L + bs - 1) // bs
        starts = np.stack([np.minimum(nblk * r // W_ * bs, L) for r in range(W_ + 1)], axis=1)
        self.starts = starts
        self.shards = []
        for r in range(W_):
            lens = (starts[:, r + 1] - starts[:, r]).astype(np.int32)
            bt = np.zeros_like(pool.block_table)
            for b in range(B):
                first, cnt = int(starts[b, r]) // bs, (int(lens[b]) + bs - 1) // bs
                bt[b, :cnt] = pool.block_table[b, first:first + cnt]
            ld = (int(lens.max()) + 63) // 64 * 64
            self.shards.append({
                "lens": torch.from_numpy(lens).to(dev), "bt": torch.from_numpy(bt).to(dev),
                "logits": torch.empty((B, ld), dtype=torch.float32, device=dev),
                "ws": torch.zeros((B, 1024), dtype=torch.int32, device=dev), "h_lens": lens})
        k = wl.topk
        self.all_vals = torch.empty((B, W_ * k), dtype=torch.float32, device=dev)
        self.all_idx = torch.empty((B, W_ * k), dtype=torch.int32, device=dev)
        self.offs = torch.from_numpy(starts[:, :W_].astype(np.int32)).to(dev)
        self.positions = torch.empty((B, k), dtype=torch.int32, device=dev)
        self.scores = torch.empty((B, k), dtype=torch.float32, device=dev)
        self.rows_per_step = B

    def step(self, stream, ev=None):
        idx, wl, k = self.idx, self.wl, self.wl.topk
        for r, sh in enumerate(self.shards):
            if ev is not None and r == 0:
                ev[0].record(stream)
            idx.idx_paged_mqa_logits_decode(self.q, self.w, self.cache, wl.pool.block_size, sh["bt"], sh["lens"],
                                            sh["logits"], ws=sh["ws"], stream=stream)
            if ev is not None and r == 0:
                ev[1].record(stream)
            idx.idx_topk(sh["logits"], None, sh["lens"], k, self.all_idx[:, r * k:(r + 1) * k],
                         vals=self.all_vals[:, r * k:(r + 1) * k], ws=sh["ws"], stream=stream)
        idx.idx_dcp_topk_merge(self.all_vals, self.all_idx, self.offs, k, k, self.positions, vals=self.scores,
                               stream=stream)

    def e2e_io(self):
        inputs = [(_pin(self.wl.q8), self.q), (_pin(self.wl.w), self.w)] + \
                 [(_pin(sh["h_lens"]), sh["lens"]) for sh in self.shards]
        return inputs, [(_pin_like(self.positions), self.positions)]

    def verify_and_time_oracle(self, n_rows):
        from tests.checks import assert_logits_close, assert_topk_row

        wl = self.wl
        rng = np.random.default_rng(wl.seed)
        rows = sorted(rng.choice(self.B, size=min(n_rows, self.B), replace=False).tolist())
        k_rows = oracle_k_rows(wl, rows, self.dev)
        cpu_s, ref = oracle_decode_rows(wl, rows, k_rows)
        pos, sc = self.positions.cpu().numpy(), self.scores.cpu().numpy()
        for b in rows:
            lg = ref[b][0]
            assert_topk_row(pos[b], lg, wl.topk, f"bench dcp top-k row {b}")
            assert_logits_close(sc[b], lg[pos[b]], f"bench dcp scores row {b}")
        cpu = {"value": round(len(rows) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{len(rows)} full rows of this workload (logits over the whole context, top-2048), "
                         f"cache prepared untimed"}
        return cpu, f"merged top-2048 and scores ok on {len(rows)} sampled rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        lens = self.shards[0]["h_lens"].astype(np.int64)
        tok = int(lens.sum())
        return hbm_roofline("mqa_logits_kernel<1> (rank 0's quarter of every context)",
                            tok * W.TOKEN_BYTES + self.B * (8192 + 256), tok * 4, kernel_ms, peaks, peak_kind)

    def config(self, world):
        return {"workload": self.wl.name + "-dcp4", "batch": self.B, "ranks_emulated": self.world,
                "sharding": "contiguous block-aligned quarters of every context", "topk": self.wl.topk,
                "step": "per rank: paged logits + local top-2048 with scores; merge of the 4 lists",
                "l2": "inputs larger than L2 (k cache > 129 MB), no flush",
                "parallelism": f"ranks emulated on one GPU, {world} independent replica(s)"}


class QPrepBench:
    """q preparation of the prefill chunk: partial RoPE, per-head e4m3 quantisation, folded bf16 weights."""

    launches_per_step = 1
    dtype = "bf16->e4m3 (f32 arithmetic)"
    metric = "indexer q preparation query-rows/s (RoPE + e4m3 quant + weight folding, 8192-query chunk)"
    # per query row: bf16 q in, e4m3 q out, fp32 weights in, bf16 weights out, position, cos/sin row
    row_bytes = 64 * 128 * 2 + 64 * 128 + 64 * 4 + 64 * 2 + 4 + 64 * 4

    def __init__(self, name, rank, dev):
        import sparse_attention_indexer_fp8_gb300 as idx

        self.idx, self.dev, self.name = idx, dev, name
        self.wl = wl = W.q_prep_chunk(seed=rank_seed(1006, rank))
        self.T = wl.T
        self.q = W.make_q_raw_device(wl.seed, wl.T, dev)
        self.pos = torch.from_numpy(wl.positions).to(dev)
        self.cs = torch.from_numpy(wl.cos_sin).to(dev)
        self.w = torch.from_numpy(wl.w).to(dev)
        self.q8 = torch.empty((wl.T, 64 * 128), dtype=torch.uint8, device=dev)
        self.w_out = torch.empty((wl.T, 64), dtype=torch.bfloat16, device=dev)
        self.rows_per_step = wl.T

    def step(self, stream, ev=None):
        if ev is not None:
            ev[0].record(stream)
        self.idx.idx_q_rope_quant(self.q, self.pos, self.cs, self.w, self.q8, self.w_out, 128 ** -0.5,
                                  64 ** -0.5, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def e2e_io(self):
        inputs = [(self.q.cpu().pin_memory(), self.q), (_pin(self.wl.positions), self.pos), (_pin(self.wl.w), self.w)]
        return inputs, [(_pin_like(self.q8), self.q8), (_pin_like(self.w_out), self.w_out)]

    def verify_and_time_oracle(self, n_rows):
        from oracle import indexer as O
        from oracle.codecs import bf16_decode, bf16_encode

        wl = self.wl
        rng = np.random.default_rng(wl.seed)
        sample = sorted(rng.choice(wl.T, size=min(max(n_rows, 1) * 64, wl.T), replace=False).tolist())
        qs = bf16_decode(self.q[sample].view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float32)
        g8 = self.q8[sample].cpu().numpy()
        gw = self.w_out[sample].view(torch.int16).cpu().numpy().view(np.uint16)
        t0 = time.perf_counter()
        o8, ow, _ = O.q_rope_quant(qs.reshape(-1, 64, 128), wl.positions[sample], wl.cos_sin, wl.w[sample],
                                   128 ** -0.5, 64 ** -0.5)
        cpu_s = time.perf_counter() - t0
        assert np.array_equal(g8.reshape(-1, 64, 128), o8), "bench q8 bytes differ from the oracle"
        assert np.array_equal(gw, bf16_encode(ow)), "bench bf16 weights differ from the oracle"
        cpu = {"value": round(len(sample) / cpu_s, 3), "unit": "rows/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{len(sample)} query rows of the chunk (RoPE, quantisation, "
                                           f"weights), inputs prepared untimed"}
        return cpu, f"q8 and bf16 weights bit-exact on {len(sample)} sampled rows"

    def roofline(self, kernel_ms, step_ms, peaks, peak_kind):
        byt = self.T * self.row_bytes
        ach = byt / (kernel_ms / 1e3) / 1e9
        return {"kernel": "q_rope_quant_kernel", "bound": "hbm", "achieved": round(ach, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                "peak_source": peak_kind, "algorithmic_bytes_per_launch": byt, "traffic": None,
                "kernel_ms": round(kernel_ms, 5)}

    def config(self, world):
        return {"workload": self.wl.name, "queries": self.T, "heads": 64, "head_dim": 128, "rope_dims": 64,
                "rope": "neox", "weights_out": "bf16",
                "step": "partial RoPE + per-head e4m3 quantisation + folded weights",
                "l2": "q in (128 MB) + q8 out (64 MB) > L2, no flush",
                "parallelism": f"rows sharded, {world} independent replica(s)"}


BENCHES = {"long_decode": DecodeBench, "long_decode_mxfp4": DecodeBench, "paged_decode": DecodeBench,
           "prefill": PrefillBench, "hierarchical_mxfp4": HierBench,
           "hierarchical": HierBench, "hierarchical_mtp": HierMtpBench, "q_prep": QPrepBench,
           "dcp_decode": DcpBench, "prefill_sparse": SparsePrefillBench,
           "prefill_sparse_mxfp4": SparsePrefillBench}


# ----------------------------------------------------------------------------- harness

GRAPH_STEPS = 10


def run_ours(args, rank, world, local, dist):
    import sparse_attention_indexer_fp8_gb300 as idx

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    bench = BENCHES[args.workload](args.workload, rank, dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        bench.step(stream)
    idx.idx_device_error(stream)
    # keep the GPU busy for a moment so the clock sampler sees it under load
    t_soak = time.time()
    while time.time() - t_soak < 1.0:
        for _ in range(5):
            bench.step(stream)
        torch.cuda.synchronize(dev)
    # the dominant kernel's own duration, from events around it in plain launches;
    # a sleep kernel holds the GPU while the host queues every one of these steps,
    # so no host launch time falls between a pair of events
    n_kev = min(args.steps, 100)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_kev)]
    torch.cuda.synchronize(dev)
    h0 = time.perf_counter()
    for _ in range(3):
        bench.step(stream)
    host_s = (time.perf_counter() - h0) / 3
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(int(min(0.2, 2.0 * n_kev * host_s) * 2.2e9))
    for i in range(n_kev):
        bench.step(stream, kev[i])
    torch.cuda.synchronize(dev)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    # the timed steps: replays of a CUDA graph holding GRAPH_STEPS steps (the
    # launches of a step are captured once; a replay costs one launch)
    graph = None
    if args.graphs:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream(dev)
            for _ in range(GRAPH_STEPS):
                bench.step(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e0.record(stream)
    done = 0
    if graph is not None:
        for _ in range(args.steps // GRAPH_STEPS):
            graph.replay()
        done = args.steps // GRAPH_STEPS * GRAPH_STEPS
    for _ in range(args.steps - done):
        bench.step(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t1 = time.time()
    ms_total = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    idx.idx_device_error(stream)

    # end to end through the public API with host buffers: every step copies its
    # inputs in from pinned memory and its result table out; two steps are in
    # flight, so step i + 1's inputs and step i - 1's result move during step i
    pipe = E2EPipeline(bench, dev)
    h2d, d2h = pipe.bytes_per_step()
    pipe.begin(stream)
    for _ in range(args.warmup):
        pipe.step(stream)
    pipe.end(stream)
    e2e_graph = None
    if args.graphs:
        # the copies from and to pinned host memory are captured with the kernels
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            cap = torch.cuda.current_stream(dev)
            pipe.begin(cap)
            for _ in range(GRAPH_STEPS):
                pipe.step(cap)
            pipe.end(cap)
        e2e_graph.replay()
    barrier(dist)
    torch.cuda.synchronize(dev)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    done = 0
    if e2e_graph is not None:
        for _ in range(args.steps // GRAPH_STEPS):
            e2e_graph.replay()
        done = args.steps // GRAPH_STEPS * GRAPH_STEPS
    if args.steps > done:
        pipe.begin(stream)
        for _ in range(args.steps - done):
            pipe.step(stream)
        pipe.end(stream)
    a1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2e_ms = max_over_ranks(dist, a0.elapsed_time(a1), dev)
    if sampler:
        sampler.stop()
    # the buffers now hold the last e2e step's results: re-run one plain step for the checks
    bench.step(stream)
    torch.cuda.synchronize(dev)
    if rank != 0:
        return None
    # the CPU baseline is taken at N = 1 only; with N > 1 rank 0 still checks a few rows
    if world == 1:
        cpu, parity = bench.verify_and_time_oracle(args.cpu_rows)
    else:
        cpu, (_, parity) = None, bench.verify_and_time_oracle(2)
    peaks, peak_kind = measured_peaks()
    rows_total = bench.rows_per_step * world
    step_ms = ms_total / args.steps
    return {
        "metric": bench.metric, "value": round(rows_total / (step_ms / 1e3), 1), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": bench.dtype,
        "data": "synthetic", "config": bench.config(world),
        "roofline": bench.roofline(kernel_ms, step_ms, peaks, peak_kind),
        "cpu_baseline": cpu,
        "e2e": {"value": round(rows_total / (e2e_ms / 1e3 / args.steps), 1), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "every step: all inputs in from one pinned host staging buffer (one copy), the "
                          "result out (one copy); two steps in flight (step i+1's inputs and step "
                          "i-1's result move during step i)"},
        "gpu_launches": bench.launches_per_step * args.steps,
        "launch": (f"CUDA graph of {GRAPH_STEPS} steps, replayed" if args.graphs else "direct launches"),
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "parity": parity,
    }


def run_reference(args, rank):
    """The oracle on the host cores: same workload, metric and unit, one row per step."""
    if rank != 0:
        return None
    name = args.workload
    rows_per_call = 1
    if name in ("long_decode", "long_decode_mxfp4", "paged_decode", "dcp_decode"):
        wl = W.paged_decode() if name == "paged_decode" else W.long_decode()
        kv = "mxfp4" if name == "long_decode_mxfp4" else "fp8"
        rng = np.random.default_rng(wl.seed)
        rows = sorted(rng.choice(wl.batch, size=min(4, wl.batch), replace=False).tolist())
        k_rows = oracle_k_rows(wl, rows, None, kv)
        one = lambda i: oracle_decode_rows(wl, [rows[i % len(rows)]], k_rows, kv=kv)[0]  # noqa: E731
        metric = (DcpBench.metric if name == "dcp_decode"
                  else DecodeBench.metric.fget(type("X", (), {"name": name})()))
        cfg = {"workload": wl.name, "batch": wl.batch, "topk": wl.topk}
    elif name == "prefill":
        from oracle import indexer as O
        from oracle.codecs import bf16_decode

        wl = W.prefill_chunk()
        k8, ks = O.k_quant(bf16_decode(W.make_k(wl.seed, 0, wl.S)))
        wv = bf16_decode(wl.w)
        T = wl.q8.shape[0]

        def one(i):
            t = (i * 997) % T
            lo, hi = int(wl.row_ks[t]), int(wl.row_ke[t])
            t0 = time.perf_counter()
            lg = O.logits_row(wl.q8[t], wv[t], k8[lo:hi], ks[lo:hi])
            O.topk_row(lg, 0, hi - lo, wl.topk)
            return time.perf_counter() - t0
        metric, cfg = PrefillBench.metric, {"workload": wl.name, "queries": T, "ctx": wl.S, "topk": wl.topk}
    elif name in ("prefill_sparse", "prefill_sparse_mxfp4"):
        from oracle import indexer as O
        from oracle.codecs import bf16_decode

        wl = W.prefill_chunk(seed=rank_seed(1006, 0))
        kv = "mxfp4" if name.endswith("_mxfp4") else "fp8"
        kf = bf16_decode(W.make_k(wl.seed, 0, wl.S))
        if kv == "mxfp4":
            codes, scales = O.mxfp4_quant(kf)
            ka, kb = O.mxfp4_pack(codes), scales
        else:
            ka, kb = O.k_quant(kf)
        wv = bf16_decode(wl.w)
        T = wl.q8.shape[0]
        cand = W.make_candidates(wl.seed, T, 64, wl.S // 64)

        def one(i):
            t = (i * 997) % T
            t0 = time.perf_counter()
            si, end = O.expand_candidates(cand[t:t + 1], wl.row_ks[t:t + 1], wl.row_ke[t:t + 1], 64, 64)
            score = O.sparse_logits_prefill_mxfp4 if kv == "mxfp4" else O.sparse_logits_prefill
            lg = score(wl.q8[t:t + 1], wv[t:t + 1], ka, kb, si, end, 64)[0]
            O.sparse_topk_remap_row(lg, int(end[0]), si[0], int(wl.row_ks[t]), 64, wl.topk)
            return time.perf_counter() - t0
        metric = SparsePrefillBench.metric.fget(type("X", (), {"kv": kv})())
        cfg = {"workload": wl.name + "-sparse" + ("-mxfp4-cache" if kv == "mxfp4" else ""), "queries": T,
               "ctx": wl.S, "topk": wl.topk}
    elif name == "q_prep":
        from oracle import indexer as O

        wl = W.q_prep_chunk()
        g = np.random.default_rng(wl.seed)
        rows = np.arange(64)
        qh = g.standard_normal((64, 64, 128)).astype(np.float32)

        def one(i):
            t0 = time.perf_counter()
            O.q_rope_quant(qh, wl.positions[rows], wl.cos_sin, wl.w[rows], 128 ** -0.5, 64 ** -0.5)
            return time.perf_counter() - t0
        metric, cfg = QPrepBench.metric, {"workload": wl.name, "queries": wl.T}
        rows_per_call = 64
    elif name == "hierarchical_mtp":
        from oracle import indexer as O

        wl = W.hierarchical_mtp()
        nn = wl.next_n
        rows = [0, 1, 2, 3]
        prep = {}
        for r in rows:
            ke = int(wl.pool.ctx_lens[r // nn]) - nn + r % nn + 1
            si, end = O.expand_candidates_row(wl.cand[r], 0, ke, 64, 64)
            prep[r] = (si, end, oracle_sparse_k(wl, r // nn, si, end, None))

        def one(i):
            r = rows[i % 4]
            si, end, (k8, ks) = prep[r]
            t0 = time.perf_counter()
            lg = O.logits_row(wl.q8[r], wl.w[r], k8[:end], ks[:end])
            dense = np.full(si.shape[0] * wl.sbk, -np.inf)
            dense[:end] = lg
            _, pos = O.sparse_topk_remap_row(dense, end, si, 0, wl.sbk, wl.topk)
            O.req_to_global_slots(pos[None], np.array([r // nn]), wl.pool.block_table, 64, 64)
            return time.perf_counter() - t0
        metric, cfg = HierMtpBench.metric, {"workload": wl.name, "batch": len(wl.pool.ctx_lens),
                                           "next_n": nn, "topk": wl.topk}
    else:
        from oracle import indexer as O

        wl = W.hierarchical()
        kv = "mxfp4" if name == "hierarchical_mxfp4" else "fp8"
        rows = [0, 1, 2, 3]
        kq = {}
        for b in rows:
            si, end = O.expand_candidates_row(wl.cand[b], 0, int(wl.pool.ctx_lens[b]), 64, 64)
            kq[b] = oracle_sparse_k(wl, b, si, end, None, kv)

        def one(i):
            t0 = time.perf_counter()
            oracle_hier_row(wl, rows[i % 4], kq[rows[i % 4]], kv)
            return time.perf_counter() - t0
        metric = ("hierarchical sparse decode indexer query-rows/s @128K ctx incl. top-2048" +
                  (", MXFP4 indexer cache" if kv == "mxfp4" else ""))
        cfg = {"workload": wl.name + ("-mxfp4-cache" if kv == "mxfp4" else ""), "batch": len(wl.pool.ctx_lens),
               "topk": wl.topk}
    for i in range(args.warmup):
        one(i)
    t = sum(one(i) for i in range(args.steps))
    value = args.steps * rows_per_call / t
    return {
        "impl": "reference", "metric": metric, "value": round(value, 3), "unit": "rows/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if name == "q_prep" else "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": round(value, 3), "unit": "rows/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "each step one full row of the workload (64 query rows of N(0,1) q for "
                                   "q_prep), cache prepared untimed"},
        "e2e": {"value": round(value, 3), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_decode", choices=sorted(BENCHES))
    ap.add_argument("--cpu-rows", type=int, default=12)
    ap.add_argument("--no-graphs", dest="graphs", action="store_false",
                    help="launch every step's kernels directly instead of replaying a CUDA graph")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        line = run_reference(args, int(os.environ.get("RANK", "0")))
    else:
        rank, world, local, dist = dist_setup(args.gpus)
        line = run_ours(args, rank, world, local, dist)
        if dist is not None:
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
