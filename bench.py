"""Benchmark of the sink-attention hot path on GB300.

One step = one pass of the whole path over the gpt-oss-shaped workloads:
  1. ragged causal prefill, 4 sequences with lengths U[2048, 8192], 64/8 heads,
     head_dim 64 (the headline: prefill attention TFLOP/s);
  2. the same prefill with a 128-token sliding window;
  3. paged split-KV decode, batch 64, contexts U[1024, 8192], 64/8 heads, head_dim 64,
     page size 16, shuffled page table, chunks of 1024 (+ the merge kernel):
     decode KV-read HBM GB/s.
Inputs are seeded synthetic tensors resident in HBM; the L2 is flushed before every
timed kernel (a 512 MB write, then a 512 MB read of another buffer, so that no dirty
line of the flush or of the previous kernel is written back inside a timed region);
every kernel is timed with CUDA events on the stream it is launched on. `e2e` repeats the headline through the public API from
pinned host buffers (sink_attn_prefill_from_host: per group of sequences the host->device
copies of q, k, v, the kernel and the device->host copy of the output, overlapped on three
streams), every copy inside the timed region.

Beside the step, timed the same way and reported in their own keys: the Qwen3-235B-style
prefill and decode (64/4 heads, head_dim 128), the gpt-oss decode replayed from one CUDA
graph, a chunked prefill over the paged cache (KV append + paged prefill), and the long
decode (batch 128 x 32768 tokens) full, with a 128-token window, and the two alternating.

--impl reference times the fp64 CPU oracle (the only other implementation of this
path) on bounded samples of the same workload on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       python bench.py --profile CASE [--reps R]   (small driver for ncu captures)
With N > 1 (torchrun) every rank runs an independent replica (the op has no
exchange step); value = units of all ranks / max-over-ranks time.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "prefill attn TFLOP/s and decode KV-read HBM GB/s, as % of GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch from an ncu capture (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by the SHA-256 of the kernel source it was taken on; stale entries are ignored.
NCU_TRAFFIC = {
    # prefill_kernel<64,0,0,0,1>, gpt-oss causal: 195.5 MB read + 116.5 MB written
    "prefill_tc.cu:1a4ec468a4219454": 312.1e6,
    # prefill_band_kernel, gpt-oss window 128: 193.2 MB read + 108.6 MB written
    "prefill_band.cu:64112c8817f75910": 301.8e6,
    # decode_split_kernel<64,1,false,8>, gpt-oss decode: 691.5 MB read + 7.3 MB written
    "decode_split.cu:25b6e31ebae3f2fc": 698.8e6,
}


def kernel_source_sha(name):
    path = os.path.join(ROOT, "gqa_attention_head_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(values, device=None):
    """Element-wise maximum of floats over every rank of the default process group; the
    values themselves when there is no group or it has one rank."""
    import torch.distributed as dist
    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate(units_per_rank, world_size, max_ms):
    """Whole-job throughput (units per second): what every rank processed, over the slowest
    rank's time. Ranks are independent replicas of the same workload."""
    return units_per_rank * world_size / (max_ms * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"sink_attn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


def prefill_flops(case):
    """Algorithmic FLOPs: two GEMMs x 2 flop per MAC over the visible (q, k) pairs."""
    return 4.0 * case.head_dim * case.num_q_heads * case.visible_pairs()


def decode_bytes(dc, fp8=False):
    """Algorithmic bytes: visible K + V (FP8 cache: codes + one fp32 scale per row), q, out,
    page-table entries read, sinks."""
    row = dc.head_dim + 4 if fp8 else dc.head_dim * 2
    kv = 2.0 * dc.visible_tokens() * dc.num_kv_heads * row
    qo = 2.0 * dc.batch * dc.num_q_heads * dc.head_dim * 2
    L = dc.seq_lens.to(torch.int64)
    lo = torch.clamp(L - dc.window, min=0) if dc.window > 0 else torch.zeros_like(L)
    pages = ((L - 1) // 16 - lo // 16 + 1).clamp(min=0) * dc.num_kv_heads
    return kv + qo + 4.0 * float(pages.sum()) + 4.0 * dc.num_q_heads + 4.0 * dc.batch


def run_ours(args):
    import gqa_attention_head_gb300 as sa
    from gqa_attention_head_gb300 import _build
    from gqa_attention_head_gb300 import workloads as wl

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or ws > 1:
        _build.build()
    sa.load_library()

    pc = wl.gptoss_prefill(seed=0, window=0)
    pw = wl.gptoss_prefill(seed=0, window=128)
    dc = wl.gptoss_decode(seed=0)
    q, k, v = pc.q.to(dev), pc.k.to(dev), pc.v.to(dev)
    sinks, cu = pc.sinks.to(dev), pc.cu_seqlens.to(dev)
    out_p = torch.empty_like(q)
    out_w = torch.empty_like(q)
    dq, dk, dv = dc.q.to(dev), dc.k_cache.to(dev), dc.v_cache.to(dev)
    dpt, dsl, dsk = dc.page_table.to(dev), dc.seq_lens.to(dev), dc.sinks.to(dev)
    need = sa.sink_attn_decode_workspace_bytes(dc.batch, dc.num_q_heads, dc.head_dim,
                                               dc.max_seq_len, dc.kv_chunk)
    dws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    dout = torch.empty_like(dq)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(i):
        """Empty the L2 (129 MB) of everything a kernel could reuse: write 512 MB, then read
        another 512 MB, so that the write's dirty lines (and those a previous kernel left) are
        written back here and not inside the next timed region."""
        flush.fill_(float(i))
        flush_rd.amax()

    def k_prefill():
        sa.sink_attn_prefill(q, k, v, sinks, cu, pc.max_seqlen, window=0, scale=pc.scale,
                             out=out_p, stream=stream)

    def k_prefill_w():
        sa.sink_attn_prefill(q, k, v, sinks, cu, pw.max_seqlen, window=128, scale=pw.scale,
                             out=out_w, stream=stream)

    def k_decode():
        sa.sink_attn_decode(dq, dk, dv, dpt, dsl, dsk, dc.max_seq_len, window=0,
                            scale=dc.scale, kv_chunk=dc.kv_chunk, workspace=dws, out=dout,
                            stream=stream)

    kernels = [("prefill", k_prefill), ("prefill_w128", k_prefill_w), ("decode", k_decode)]
    launches_per_step = 2 + 1 + (1 if need > 0 else 0)

    for _ in range(args.warmup):
        for _, fn in kernels:
            flush_l2(1)
            fn()
    torch.cuda.synchronize()
    st, bits = sa.sink_attn_read_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {bits:#x} after warm-up")

    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for n, _ in kernels}
    if ws > 1:
        torch.distributed.barrier()
    clocks = Clocks(local)
    clocks.start()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        for n, fn in kernels:
            a, b = ev[n][i]
            flush_l2(i)
            a.record(stream)
            fn()
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    # The timed steps last tens of milliseconds, less than the sampling interval: keep the
    # GPU on the same steps, untimed, while the sampler records the clocks under this load.
    t_load = time.perf_counter() + 0.6
    while time.perf_counter() < t_load:
        for i in range(args.steps):
            for _, fn in kernels:
                flush_l2(i)
                fn()
        torch.cuda.synchronize()
    clk = clocks.stop()
    clk["window"] = "the timed steps, then 0.6 s of the same steps untimed"
    if ws > 1:
        torch.distributed.barrier()
    st, bits = sa.sink_attn_read_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {bits:#x} after timing")

    ms = {n: [a.elapsed_time(b) for a, b in ev[n]] for n, _ in kernels}
    mean = {n: sum(x) / len(x) for n, x in ms.items()}
    step_ms = sum(mean.values())
    red = max_over_ranks([step_ms] + [mean[n] for n, _ in kernels], dev)
    step_ms = red[0]
    for i, (n, _) in enumerate(kernels):
        mean[n] = red[i + 1]

    # ---------------- e2e: host buffers through the public API ----------------
    # sink_attn_prefill_from_host: per group of sequences, the inputs' host->device copies,
    # the prefill kernel and the output's device->host copy, overlapped on three streams.
    hq_ = pc.q.pin_memory()
    hk_, hv_ = pc.k.pin_memory(), pc.v.pin_memory()
    hs_, hc_ = pc.sinks.pin_memory(), pc.cu_seqlens.pin_memory()
    hout = torch.empty(pc.q.shape, dtype=torch.bfloat16).pin_memory()
    e2e_ms = []
    for i in range(max(args.steps, 3) + 2):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        sa.sink_attn_prefill_from_host(hq_, hk_, hv_, hs_, hc_, pc.max_seqlen, window=0,
                                       scale=pc.scale, out=hout, device=dev, q_dev=q, k_dev=k,
                                       v_dev=v, out_dev=out_p)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            e2e_ms.append(a.elapsed_time(b))
    e2e_mean = max_over_ranks([sum(e2e_ms) / len(e2e_ms)], dev)[0]
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_, hs_, hc_))
    d2h = hout.numel() * hout.element_size()

    # ---------------- the Qwen3-235B-style workloads (not part of the step) ----------------
    # Timed the same way (L2 flushed, CUDA events on the launching stream), reported beside
    # the step so that every configuration's rate is measured on each run.
    qp = wl.qwen_prefill(seed=0, sinks="normal")
    qq, qk, qv = qp.q.to(dev), qp.k.to(dev), qp.v.to(dev)
    qs, qcu = qp.sinks.to(dev), qp.cu_seqlens.to(dev)
    qout = torch.empty_like(qq)
    # the same tensors with sinks -inf (standard softmax attention): the q, k and v draws
    # come before the sinks, so both sink settings share them
    qp_ninf = wl.qwen_prefill(seed=0, sinks="-inf")
    assert torch.equal(qp_ninf.q, qp.q) and torch.equal(qp_ninf.k, qp.k)
    qs_ninf = qp_ninf.sinks.to(dev)
    qd = wl.qwen_decode(seed=0)
    qdq, qdk, qdv = qd.q.to(dev), qd.k_cache.to(dev), qd.v_cache.to(dev)
    qdpt, qdsl, qdsk = qd.page_table.to(dev), qd.seq_lens.to(dev), qd.sinks.to(dev)
    qneed = sa.sink_attn_decode_workspace_bytes(qd.batch, qd.num_q_heads, qd.head_dim,
                                                qd.max_seq_len, qd.kv_chunk)
    qdws = torch.empty(max(qneed, 16), dtype=torch.uint8, device=dev)
    qdout = torch.empty_like(qdq)

    def q_prefill():
        sa.sink_attn_prefill(qq, qk, qv, qs, qcu, qp.max_seqlen, window=0, scale=qp.scale,
                             out=qout, stream=stream)

    def q_prefill_ninf():
        sa.sink_attn_prefill(qq, qk, qv, qs_ninf, qcu, qp.max_seqlen, window=0, scale=qp.scale,
                             out=qout, stream=stream)

    def q_decode():
        sa.sink_attn_decode(qdq, qdk, qdv, qdpt, qdsl, qdsk, qd.max_seq_len, window=0,
                            scale=qd.scale, kv_chunk=qd.kv_chunk, workspace=qdws, out=qdout,
                            stream=stream)

    def timed_mean(fn, reps):
        for _ in range(3):
            flush_l2(1)
            fn()
        ts = []
        for i in range(reps):
            flush_l2(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return sum(ts) / len(ts)

    q_prefill_ms = timed_mean(q_prefill, max(args.steps, 3))
    q_prefill_ninf_ms = timed_mean(q_prefill_ninf, max(args.steps, 3))
    q_decode_ms = timed_mean(q_decode, max(args.steps, 3))
    qfkc, qfks = sa.sink_attn_quantize_fp8(qdk)
    qfvc, qfvs = sa.sink_attn_quantize_fp8(qdv)

    def q_decode_fp8():
        sa.sink_attn_decode_fp8(qdq, qfkc, qfvc, qfks, qfvs, qdpt, qdsl, qdsk, qd.max_seq_len,
                                window=0, scale=qd.scale, kv_chunk=qd.kv_chunk, workspace=qdws,
                                out=qdout, stream=stream)

    q_decode_fp8_ms = timed_mean(q_decode_fp8, max(args.steps, 3))
    del qfkc, qfvc, qfks, qfvs

    # ---------------- decode as one CUDA graph (split + merge kernels) ----------------
    def decode_on(s):
        sa.sink_attn_decode(dq, dk, dv, dpt, dsl, dsk, dc.max_seq_len, window=0,
                            scale=dc.scale, kv_chunk=dc.kv_chunk, workspace=dws, out=dout,
                            stream=s)

    k_decode()
    direct = dout.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_on(torch.cuda.current_stream(dev))
    dout.zero_()
    graph.replay()
    torch.cuda.synchronize()
    if not torch.equal(dout, direct):
        raise RuntimeError("graph-replayed decode differs from the direct call")
    decode_graph_ms = timed_mean(graph.replay, max(args.steps, 3))
    del graph, direct

    # ---------------- gpt-oss decode over an FP8 cache ----------------
    fkc, fks = sa.sink_attn_quantize_fp8(dk)
    fvc, fvs = sa.sink_attn_quantize_fp8(dv)

    def f_decode():
        sa.sink_attn_decode_fp8(dq, fkc, fvc, fks, fvs, dpt, dsl, dsk, dc.max_seq_len, window=0,
                                scale=dc.scale, kv_chunk=dc.kv_chunk, workspace=dws, out=dout,
                                stream=stream)

    f_decode_ms = timed_mean(f_decode, max(args.steps, 3))
    f_bytes = decode_bytes(dc, fp8=True)
    del fkc, fvc, fks, fvs

    # ---------------- chunked prefill over the paged cache (append + prefill) ----------------
    cp = wl.gptoss_chunked_prefill(seed=0)
    cq, ckn, cvn = cp.q.to(dev), cp.k_new.to(dev), cp.v_new.to(dev)
    ckc, cvc = cp.k_cache.to(dev), cp.v_cache.to(dev)
    cpt, ccu, csl, csk = (cp.page_table.to(dev), cp.cu_seqlens.to(dev), cp.seq_lens.to(dev),
                          cp.sinks.to(dev))
    cout = torch.empty_like(cq)

    def c_prefill():
        # the append writes the same rows into the same slots on every call
        sa.sink_attn_prefill_paged(cq, ckn, cvn, ckc, cvc, cpt, ccu, csl, csk, cp.max_q_len,
                                   cp.max_seq_len, window=0, scale=cp.scale, out=cout,
                                   stream=stream)

    c_prefill_ms = timed_mean(c_prefill, max(args.steps, 3))
    c_flops = 4.0 * cp.q.shape[2] * cp.q.shape[1] * cp.visible_pairs()
    del ckc, cvc

    # ---------------- long decode: 128 x 32768, full and window 128 ----------------
    # The 8.6 GB cache is filled on the device; the full call reads more than the L2 holds,
    # the window-128 call (33.5 MB) is timed after the same flush.
    ld = wl.long_decode(0, window=0, cache_device=str(dev), only_seqs=[0])
    ldw = dataclasses.replace(ld, window=128)
    lq, lpt, lsl, lsk = ld.q.to(dev), ld.page_table.to(dev), ld.seq_lens.to(dev), ld.sinks.to(dev)
    lneed = sa.sink_attn_decode_workspace_bytes(ld.batch, ld.num_q_heads, ld.head_dim,
                                                ld.max_seq_len, ld.kv_chunk)
    lws = torch.empty(max(lneed, 16), dtype=torch.uint8, device=dev)
    lout = torch.empty_like(lq)

    def l_decode(w):
        sa.sink_attn_decode(lq, ld.k_cache, ld.v_cache, lpt, lsl, lsk, ld.max_seq_len, window=w,
                            scale=ld.scale, kv_chunk=ld.kv_chunk, workspace=lws, out=lout,
                            stream=stream)

    # the same cache as FP8 (e4m3 codes + row scales, quantised on the device)
    lkc, lks = sa.sink_attn_quantize_fp8(ld.k_cache)
    lvc, lvs = sa.sink_attn_quantize_fp8(ld.v_cache)

    def l_decode_fp8():
        sa.sink_attn_decode_fp8(lq, lkc, lvc, lks, lvs, lpt, lsl, lsk, ld.max_seq_len, window=0,
                                scale=ld.scale, kv_chunk=ld.kv_chunk, workspace=lws, out=lout,
                                stream=stream)

    l_fp8_ms = timed_mean(l_decode_fp8, max(args.steps, 3))
    l_fp8_bytes = decode_bytes(ld, fp8=True)
    del lkc, lvc, lks, lvs
    l_full_ms = timed_mean(lambda: l_decode(0), max(args.steps, 3))
    l_w_ms = timed_mean(lambda: l_decode(128), max(args.steps, 3))
    l_pair_ms = timed_mean(lambda: (l_decode(0), l_decode(128)), max(args.steps, 3))
    l_bytes, lw_bytes = decode_bytes(ld), decode_bytes(ldw)
    del ld, ldw, lws
    torch.cuda.empty_cache()
    st, bits = sa.sink_attn_read_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {bits:#x} after the side measurements")

    peaks, peak_src = load_peaks()
    pf = prefill_flops(pc)
    pwf = prefill_flops(pw)
    # algorithmic bytes of a prefill: Q, K, V read once, the output written once
    pw_bytes = float(sum(t.numel() * t.element_size() for t in (pw.q, pw.k, pw.v, pw.q)))
    db = decode_bytes(dc)
    tflops = pf / (mean["prefill"] * 1e-3) / 1e12  # per replica
    tflops_w = pwf / (mean["prefill_w128"] * 1e-3) / 1e12
    gbs = db / (mean["decode"] * 1e-3) / 1e9
    peak_tc = float(peaks["bf16_tflops"])
    peak_hbm = float(peaks["hbm_gbs"])

    def traffic(src):
        return NCU_TRAFFIC.get(f"{src}:{kernel_source_sha(src)}")

    result = {
        "metric": METRIC,
        "value": round(job_rate(pf, ws, mean["prefill"]) / 1e12, 3),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs of the gpt-oss attention shapes)",
        "config": step_config(pc, dc.name, dc.batch, dc.visible_tokens(), {
            "l2": "flushed before every timed kernel (512 MB write, then 512 MB read)",
            "parallelism": f"replicas x{ws}",
        }),
        "impl": "ours",
        "gpu_launches": launches_per_step * args.steps,
        "kernel_ms": {n: round(x, 4) for n, x in mean.items()},
        "kernel_ms_p10_p50_p90": {n: [round(float(np.percentile(x, q)), 4) for q in (10, 50, 90)]
                                  for n, x in ms.items()},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak_tc,
                     "unit": "TFLOP/s", "frac": round(tflops / peak_tc, 4),
                     "traffic": traffic("prefill_tc.cu"),
                     "kernel": "prefill_kernel<64,0,0,0,1> (gpt-oss causal)",
                     "peak_source": f"bf16_tflops burst, {peak_src}"},
        "prefill_window128": {"value": round(tflops_w, 3), "unit": "TFLOP/s",
                              "frac": round(tflops_w / peak_tc, 4),
                              "kernel": "prefill_band_kernel (32 queries x 8 heads per unit)",
                              "hbm": {"algorithmic_bytes": pw_bytes,
                                      "achieved_gbs": round(pw_bytes / (mean["prefill_w128"] * 1e-3) / 1e9, 1),
                                      "frac": round(pw_bytes / (mean["prefill_w128"] * 1e-3) / 1e9
                                                    / peak_hbm, 4),
                                      "traffic": traffic("prefill_band.cu")},
                              "note": "about 4e10 flop against 346 MB of Q, K, V and output: "
                                      "the HBM time of its bytes (51 us) is the floor"},
        "decode": {"value": round(job_rate(db, ws, mean["decode"]) / 1e9, 2), "unit": "GB/s",
                   "frac": round(gbs / peak_hbm, 4),
                   "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_hbm,
                                "unit": "GB/s", "frac": round(gbs / peak_hbm, 4),
                                "traffic": traffic("decode_split.cu"),
                                "peak_source": f"hbm_gbs, {peak_src}"},
                   "algorithmic_bytes": db},
        "prefill_qwen": {"value": round(prefill_flops(qp) / (q_prefill_ms * 1e-3) / 1e12, 3),
                         "unit": "TFLOP/s",
                         "frac": round(prefill_flops(qp) / (q_prefill_ms * 1e-3) / 1e12 / peak_tc, 4),
                         "ms": round(q_prefill_ms, 4), "workload": qp.name,
                         "note": "measured beside the step (not part of it)"},
        "prefill_qwen_sinks_ninf": {
            "value": round(prefill_flops(qp_ninf) / (q_prefill_ninf_ms * 1e-3) / 1e12, 3),
            "unit": "TFLOP/s",
            "frac": round(prefill_flops(qp_ninf) / (q_prefill_ninf_ms * 1e-3) / 1e12 / peak_tc, 4),
            "ms": round(q_prefill_ninf_ms, 4), "workload": qp_ninf.name,
            "note": "measured beside the step (not part of it)"},
        "decode_qwen": {"value": round(decode_bytes(qd) / (q_decode_ms * 1e-3) / 1e9, 2),
                        "unit": "GB/s",
                        "frac": round(decode_bytes(qd) / (q_decode_ms * 1e-3) / 1e9 / peak_hbm, 4),
                        "ms": round(q_decode_ms, 4), "workload": qd.name,
                        "algorithmic_bytes": decode_bytes(qd),
                        "note": "measured beside the step (not part of it)"},
        "decode_qwen_fp8": {"value": round(decode_bytes(qd, fp8=True) / (q_decode_fp8_ms * 1e-3) / 1e9, 2),
                            "unit": "GB/s",
                            "frac": round(decode_bytes(qd, fp8=True) / (q_decode_fp8_ms * 1e-3) / 1e9
                                          / peak_hbm, 4),
                            "ms": round(q_decode_fp8_ms, 4), "workload": qd.name + ", FP8 cache",
                            "algorithmic_bytes": decode_bytes(qd, fp8=True),
                            "note": f"speedup over the bf16 decode: {q_decode_ms / q_decode_fp8_ms:.2f}x"},
        "decode_graph": {"value": round(db / (decode_graph_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                         "frac": round(db / (decode_graph_ms * 1e-3) / 1e9 / peak_hbm, 4),
                         "ms": round(decode_graph_ms, 4), "workload": dc.name,
                         "note": "split + merge captured in one CUDA graph, replayed"},
        "prefill_paged": {"value": round(c_flops / (c_prefill_ms * 1e-3) / 1e12, 3),
                          "unit": "TFLOP/s",
                          "frac": round(c_flops / (c_prefill_ms * 1e-3) / 1e12 / peak_tc, 4),
                          "ms": round(c_prefill_ms, 4), "workload": cp.name,
                          "note": "KV append + paged prefill kernels, measured beside the step"},
        "decode_fp8": {"value": round(f_bytes / (f_decode_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "frac": round(f_bytes / (f_decode_ms * 1e-3) / 1e9 / peak_hbm, 4),
                       "ms": round(f_decode_ms, 4), "algorithmic_bytes": f_bytes,
                       "workload": dc.name + ", FP8 cache (e4m3 + fp32 row scales)",
                       "note": "speedup over the bf16 decode: "
                               f"{mean['decode'] / f_decode_ms:.2f}x"},
        "decode_long_fp8": {"value": round(l_fp8_bytes / (l_fp8_ms * 1e-3) / 1e9, 2),
                            "unit": "GB/s",
                            "frac": round(l_fp8_bytes / (l_fp8_ms * 1e-3) / 1e9 / peak_hbm, 4),
                            "ms": round(l_fp8_ms, 4), "algorithmic_bytes": l_fp8_bytes,
                            "workload": "long decode B128 ctx32768 Hq64/Hkv8 D64 full, FP8 cache"},
        "decode_long": {"value": round(l_bytes / (l_full_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                        "frac": round(l_bytes / (l_full_ms * 1e-3) / 1e9 / peak_hbm, 4),
                        "ms": round(l_full_ms, 4), "algorithmic_bytes": l_bytes,
                        "workload": "long decode B128 ctx32768 Hq64/Hkv8 D64 full"},
        "decode_long_w128": {"value": round(lw_bytes / (l_w_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                             "frac": round(lw_bytes / (l_w_ms * 1e-3) / 1e9 / peak_hbm, 4),
                             "ms": round(l_w_ms, 4), "algorithmic_bytes": lw_bytes,
                             "note": "latency-dominated (33.5 MB visible)"},
        "decode_long_pair": {"value": round((l_bytes + lw_bytes) / (l_pair_ms * 1e-3) / 1e9, 2),
                             "unit": "GB/s",
                             "frac": round((l_bytes + lw_bytes) / (l_pair_ms * 1e-3) / 1e9
                                           / peak_hbm, 4),
                             "ms": round(l_pair_ms, 4),
                             "note": "full then window-128 call on the same cache, combined"},
        "e2e": {"value": round(job_rate(pf, ws, e2e_mean) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_mean, 4)},
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(pc, args.cpu_seconds)
        result["cpu_baseline"]["decode"] = cpu_baseline_decode(dc)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline(pc, seconds):
    """The fp64 oracle, as it stands, on a bounded sample of the headline workload:
    random (token, head) rows of the causal gpt-oss prefill, timed on all host cores."""
    import oracle
    from gqa_attention_head_gb300 import workloads as wl
    rng = np.random.default_rng(0)
    qb, kb, vb = wl.bf16_bits(pc.q), wl.bf16_bits(pc.k), wl.bf16_bits(pc.v)
    sk, cu = pc.sinks.numpy(), pc.cu_seqlens.numpy()
    starts = np.repeat(cu[:-1], np.diff(cu))
    done_flops, done_rows, t_total = 0.0, 0, 0.0
    batch = 256
    while t_total < seconds:
        toks = rng.integers(0, pc.total_tokens, batch)
        heads = rng.integers(0, pc.num_q_heads, batch).astype(np.int32)
        t0 = time.perf_counter()
        oracle.prefill_rows(qb, kb, vb, sk, cu, toks, heads, window=0, scale=pc.scale)
        t_total += time.perf_counter() - t0
        keys = toks - starts[toks] + 1
        done_flops += 4.0 * pc.head_dim * float(keys.sum())
        done_rows += batch
    return {"value": round(done_flops / t_total / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done_rows} random (token, head) rows of the causal gpt-oss prefill, "
                      f"{t_total:.1f} s"}


def cpu_baseline_decode(dc):
    """The fp64 oracle on the whole gpt-oss decode (every output), timed once on all host
    cores; reported in the decode's own unit (algorithmic bytes per second)."""
    import oracle
    from gqa_attention_head_gb300 import workloads as wl
    args = (wl.bf16_bits(dc.q), wl.bf16_bits(dc.k_cache), wl.bf16_bits(dc.v_cache),
            dc.page_table.numpy(), dc.seq_lens.numpy(), dc.sinks.numpy())
    oracle.decode(*args, window=dc.window, scale=dc.scale)  # untimed: loads and warms up
    t0 = time.perf_counter()
    oracle.decode(*args, window=dc.window, scale=dc.scale)
    dt = time.perf_counter() - t0
    return {"value": round(decode_bytes(dc) / dt / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle", "seconds": round(dt, 4),
            "sample": f"every output of the {dc.name} ({dc.batch} sequences), once"}


def step_config(pc, decode_name, decode_batch, decode_tokens, extra):
    """The `config` of both arms' JSON lines: the timed step's workloads and their sizes."""
    cfg = {"workload": pc.name + " | same with window 128 | " + decode_name,
           "prefill_tokens": pc.total_tokens, "prefill_lengths": pc.lengths,
           "decode_batch": decode_batch, "decode_context_tokens": decode_tokens}
    cfg.update(extra)
    return cfg


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores. Each step
    runs the step's three workloads, the causal prefill on a bounded sample of random
    (token, head) rows (its whole would take about 20 s) and the windowed prefill and the
    decode whole; `value` is the causal prefill's rate on its sample (the same metric and
    unit as the GPU arm's headline), `ms_per_step` the measured wall time of one such
    step, and `extrapolated_full_step_ms` the time the whole step would take at the
    measured rates."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    from gqa_attention_head_gb300 import workloads as wl
    import oracle
    oracle.build.build()
    pc = wl.gptoss_prefill(seed=0, window=0)
    pw = wl.gptoss_prefill(seed=0, window=128)
    dc = wl.gptoss_decode(seed=0)
    qb, kb, vb = wl.bf16_bits(pc.q), wl.bf16_bits(pc.k), wl.bf16_bits(pc.v)
    dargs = (wl.bf16_bits(dc.q), wl.bf16_bits(dc.k_cache), wl.bf16_bits(dc.v_cache),
             dc.page_table.numpy(), dc.seq_lens.numpy(), dc.sinks.numpy())
    # seconds of causal-prefill rows per step, so that the whole run stays within minutes
    per_step = max(1.0, min(8.0, 100.0 / max(1, args.steps + args.warmup)))

    def step():
        t0 = time.perf_counter()
        cb = cpu_baseline(pc, per_step)
        t1 = time.perf_counter()
        oracle.prefill(qb, kb, vb, pw.sinks.numpy(), pw.cu_seqlens.numpy(), window=pw.window,
                       scale=pw.scale)
        t2 = time.perf_counter()
        oracle.decode(*dargs, window=dc.window, scale=dc.scale)
        t3 = time.perf_counter()
        return cb, (t3 - t0) * 1e3, (t2 - t1) * 1e3, (t3 - t2) * 1e3

    for _ in range(args.warmup):
        step()
    runs = [step() for _ in range(args.steps)]
    value = sum(r[0]["value"] for r in runs) / len(runs)
    ms_per_step = sum(r[1] for r in runs) / len(runs)
    w_ms = sum(r[2] for r in runs) / len(runs)
    d_ms = sum(r[3] for r in runs) / len(runs)
    full_causal_ms = prefill_flops(pc) / (value * 1e12) * 1e3
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs of the gpt-oss attention shapes)",
        "config": step_config(pc, dc.name, dc.batch, dc.visible_tokens(), {
            "parallelism": "host cores (OpenMP)",
            "timed": "per step: the causal prefill on sampled rows (the headline value), the "
                     "window-128 prefill and the decode whole",
        }),
        "impl": "reference",
        "extrapolated_full_step_ms": round(full_causal_ms + w_ms + d_ms, 1),
        "part_ms": {"prefill_causal_sampled": round(ms_per_step - w_ms - d_ms, 1),
                    "prefill_w128": round(w_ms, 1), "decode": round(d_ms, 1)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                         "cores": runs[0][0]["cores"],
                         "sample": f"each step: random (token, head) rows of the causal "
                                   f"prefill for ~{per_step:.0f} s, then the window-128 "
                                   f"prefill and the decode whole"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PROFILE_CASES = ("prefill_gptoss", "prefill_gptoss_w128", "prefill_qwen", "prefill_qwen_ninf",
                 "prefill_paged", "decode_gptoss", "decode_gptoss_fp8", "decode_qwen",
                 "decode_qwen_fp8")


def run_profile(args):
    """A small driver for ncu captures: one workload's inputs on the device and nothing else
    (no L2 flush buffers, no other workload), the kernel launched `--reps` times. Prints
    one line with the last launch's time; that time is not a bench value."""
    import gqa_attention_head_gb300 as sa
    from gqa_attention_head_gb300 import _build
    from gqa_attention_head_gb300 import workloads as wl
    _build.build()
    sa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    name = args.profile
    if name.startswith("prefill") and name != "prefill_paged":
        pc = {"prefill_gptoss": lambda: wl.gptoss_prefill(0, window=0),
              "prefill_gptoss_w128": lambda: wl.gptoss_prefill(0, window=128),
              "prefill_qwen": lambda: wl.qwen_prefill(0, sinks="normal"),
              "prefill_qwen_ninf": lambda: wl.qwen_prefill(0, sinks="-inf")}[name]()
        q, k, v = pc.q.to(dev), pc.k.to(dev), pc.v.to(dev)
        sk, cu = pc.sinks.to(dev), pc.cu_seqlens.to(dev)
        out = torch.empty_like(q)
        work, unit = prefill_flops(pc), "flop"

        def fn():
            sa.sink_attn_prefill(q, k, v, sk, cu, pc.max_seqlen, window=pc.window,
                                 scale=pc.scale, out=out, stream=stream)
    elif name == "prefill_paged":
        cp = wl.gptoss_chunked_prefill(seed=0)
        cq, ckn, cvn = cp.q.to(dev), cp.k_new.to(dev), cp.v_new.to(dev)
        ckc, cvc = cp.k_cache.to(dev), cp.v_cache.to(dev)
        cpt, ccu, csl, csk = (cp.page_table.to(dev), cp.cu_seqlens.to(dev),
                              cp.seq_lens.to(dev), cp.sinks.to(dev))
        out = torch.empty_like(cq)
        work, unit = 4.0 * cp.q.shape[2] * cp.q.shape[1] * cp.visible_pairs(), "flop"

        def fn():
            sa.sink_attn_prefill_paged(cq, ckn, cvn, ckc, cvc, cpt, ccu, csl, csk, cp.max_q_len,
                                       cp.max_seq_len, window=0, scale=cp.scale, out=out,
                                       stream=stream)
    else:
        fp8 = name.endswith("_fp8")
        if name.startswith("decode_qwen"):
            dc = wl.qwen_decode(seed=0)
        else:
            dc = wl.gptoss_decode(seed=0)
        dq, dk, dv = dc.q.to(dev), dc.k_cache.to(dev), dc.v_cache.to(dev)
        dpt, dsl, dsk = dc.page_table.to(dev), dc.seq_lens.to(dev), dc.sinks.to(dev)
        need = sa.sink_attn_decode_workspace_bytes(dc.batch, dc.num_q_heads, dc.head_dim,
                                                   dc.max_seq_len, dc.kv_chunk)
        ws_ = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        out = torch.empty_like(dq)
        if fp8:
            kc, ks = sa.sink_attn_quantize_fp8(dk)
            vc, vs = sa.sink_attn_quantize_fp8(dv)
            del dk, dv

            def fn():
                sa.sink_attn_decode_fp8(dq, kc, vc, ks, vs, dpt, dsl, dsk, dc.max_seq_len,
                                        window=dc.window, scale=dc.scale, kv_chunk=dc.kv_chunk,
                                        workspace=ws_, out=out, stream=stream)
        else:
            def fn():
                sa.sink_attn_decode(dq, dk, dv, dpt, dsl, dsk, dc.max_seq_len, window=dc.window,
                                    scale=dc.scale, kv_chunk=dc.kv_chunk, workspace=ws_, out=out,
                                    stream=stream)
        work, unit = decode_bytes(dc, fp8=fp8), "byte"
    ms = 0.0
    for _ in range(args.reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
    st, bits = sa.sink_attn_read_device_error()
    if st != 0:
        raise RuntimeError(f"device error word {bits:#x}")
    print(json.dumps({"profile": name, "reps": args.reps, "algorithmic": work, "unit": unit,
                      "last_ms": round(ms, 4),
                      "note": "small-driver run for ncu; not a bench value"}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=PROFILE_CASES, default=None,
                    help="small driver for ncu: only this workload's kernel, --reps launches")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
