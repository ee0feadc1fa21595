"""Benchmark: paged KV-cache decode on one GB300 (plus replicas for N > 1).

One step = one serving decode step of the paged path: append the new token's
k/v into its page and attend over the paged cache (page resolution, fused
append, device split plan, split-KV decode and, when splits are used, the
combine) for a batch of 256 sequences at context 4096 with 32 query / 32 kv
heads, head_dim 128, fp16, 16-token pages and a block table that is a random
permutation of the pool.  The cache (17.2 GB) is far larger than L2 (129 MB),
so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is the whole-job algorithmic HBM
throughput in GB/s; `roofline` compares the decode kernel's achieved GB/s with
the measured HBM copy bandwidth; `cpu_baseline` is the CPU oracle timed on a
bounded sample of the same workload.  `--impl reference` times the CPU oracle
itself as the reference arm.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(workload="paged decode step with fused 1-token append", batch=256, ctx=4096,
                num_q_heads=32, num_kv_heads=32, head_dim=128, page_size=16, dtype="f16",
                lnew=1, block_table="random permutation of the pool", values="N(0,1)",
                l2="inputs (17.2 GB of K/V) larger than L2; no flush")
METRIC = "paged decode HBM GB/s (% of peak) and prefill TFLOPS (% tensor peak) vs µs/call"
HBM_NOMINAL_GBS = 7900.0  # GB300 HBM3e, nominal


def algorithmic_bytes(B, lk, lnew, lq, hq, hkv, d, elt=2):
    """Bytes the step must move at minimum: every key/value of the context once
    (cached ones from HBM, new ones from k_new/v_new), the appended k/v write,
    q, out, lse and the block-table entries."""
    kv_read = B * lk * hkv * d * elt * 2
    append_write = B * lnew * hkv * d * elt * 2
    q_out = B * lq * hq * d * elt * 2
    lse = B * lq * hq * 4
    table = B * math.ceil(lk / 16) * 4
    return kv_read + append_write + q_out + lse + table


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def read_tensor_peak():
    """Dense 16-bit tensor peak in TFLOP/s (fp16 and bf16 run at the same rate):
    the burst figure for a kernel timed alone."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


def attention_flops(q_lens, k_lens, heads, d, causal):
    """4*D flops (QK^T and PV) per visible (query, key) pair, summed exactly."""
    total = 0
    for lq, lk in zip(q_lens, k_lens):
        if causal:
            pairs = sum(max(0, min(lk, i + lk - lq + 1)) for i in range(lq))
        else:
            pairs = lq * lk
        total += pairs
    return 4 * d * heads * total


class L2Flush:
    """Cold-L2 preparation between timed calls: a 512 MB write (four times
    the 129 MB L2), then a 512 MB read, so that the dirty lines the write
    leaves are written back before the timed call rather than during it
    (a write-only flush costs the call that follows 2-4 us of write-backs it
    did not cause)."""

    def __init__(self, device):
        import torch

        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(128 << 20, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def time_calls(fn, steps, warmup, stream, graph=True, flush=False):
    """Device time per call in us.  With `graph`, `steps` calls are captured in
    one CUDA graph and replayed, so host launch overhead does not show up as
    idle device time for short kernels (the library never synchronises or
    reads lengths on the host, so its calls capture as they are).  With
    `flush`, every call is preceded by an L2 flush (L2Flush) outside its own
    event pair: for workloads whose inputs would otherwise stay in L2 between
    calls; the call's launches are queued behind the flush, so no host gap
    shows up inside the pair, and the figure is the mean over the pairs."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if flush:
        l2flush = L2Flush(stream.device)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)]
        for a, b in pairs:
            l2flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        # the mean, not the median: event timestamps on this part step in
        # 4.096 us, so a single call's time is a multiple of that and the
        # median of such samples snaps to one of the multiples; calls that
        # start at random phases against the step average to the true time
        return sum(a.elapsed_time(b) for a, b in pairs) / steps * 1e3
    if graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
            with torch.cuda.graph(g, stream=side):
                for _ in range(steps):
                    fn()
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    else:
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps * 1e3


def sweep_point(dev, ctx, B, peak):
    """One point of the paged decode sweep: 32 q = 32 kv heads, D 128, fp16,
    one appended token per sequence, automatic splits.  Inputs under 4x L2
    are timed cold (L2 flushed before every call), larger ones back to back.
    Returns (us, GB/s, frac of peak, timing mode, graded)."""
    import torch

    import paged_kv_cache_page_gb300 as pa
    from paged_kv_cache_page_gb300 import workloads as wl

    stream = torch.cuda.current_stream(dev)
    w = wl.paged_decode(B, ctx, lnew=1, seed=1002, device=dev)
    out = torch.empty((B, 1, 32, 128), dtype=torch.float16, device=dev)
    lse = torch.empty((B, 32, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, pa.fwd_kvcache_workspace_size(B, 1, 32, 32, 128, ctx, 0)),
                     dtype=torch.uint8, device=dev)
    fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"],  # noqa: E731
                                   w["cache_seqlens"], w["block_table"], k=w["k_new"],
                                   v=w["v_new"], out=out, lse=lse, workspace=ws,
                                   max_seqlen_k=ctx)
    steps = max(5, min(200, int(2e9 / max(1, B * ctx * 16384))))
    by = algorithmic_bytes(B, ctx, 1, 1, 32, 32, 128)
    if by < 4 * 129e6:
        l2flush = L2Flush(dev)
        ts = []
        steps = max(steps, 60)  # enough calls to average out the timestamp step
        for i in range(steps + 3):
            l2flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        us = sum(ts) / len(ts)  # mean: see time_calls on the 4.096 us timestamp step
        mode = "cold (L2 flushed per call)"
        del l2flush
    else:
        us = time_calls(fn, steps, 3, stream, graph=False)
        mode = "inputs > 4x L2"
    gbs = by / us / 1e3
    ideal_us = by / (peak * 1e3)
    del w, out, lse, ws
    torch.cuda.empty_cache()
    return us, gbs, gbs / peak, mode, ideal_us >= 20.0


def decode_sweep(dev):
    """The paged decode sweep: ctx {512..4096} x batch {1..256}.  One JSON
    line per point with us per call, algorithmic GB/s and the fraction of the
    HBM copy peak; points whose ideal time is under 20 us are launch-latency
    bound and marked `graded: false`."""
    peak, src = read_peaks()
    for ctx in (512, 1024, 2048, 4096):
        for B in (1, 2, 4, 8, 16, 32, 64, 128, 256):
            us, gbs, frac, mode, graded = sweep_point(dev, ctx, B, peak)
            print(json.dumps({"sweep": "paged decode", "ctx": ctx, "batch": B, "us": round(us, 2),
                              "gbs": round(gbs, 1), "frac_hbm": round(frac, 4),
                              "peak": peak, "peak_source": src, "timing": mode,
                              "graded": graded}), flush=True)


def graded_sweep(dev):
    """The graded points of the decode sweep (context >= 2048, ideal time at
    the peak >= 20 us): ctx 2048 x B 8..256 and ctx 4096 x B 4..256; the bar
    is 0.70 of the measured HBM peak."""
    peak, src = read_peaks()
    pts = []
    for ctx, batches in ((2048, (8, 16, 32, 64, 128, 256)), (4096, (4, 8, 16, 32, 64, 128, 256))):
        for B in batches:
            us, gbs, frac, mode, _ = sweep_point(dev, ctx, B, peak)
            pts.append({"ctx": ctx, "batch": B, "us": round(us, 2), "gbs": round(gbs, 1),
                        "frac": round(frac, 4), "timing": mode})
    return {"points": pts, "passing": sum(p["frac"] >= 0.70 for p in pts), "graded": len(pts),
            "bar": 0.70, "peak": peak, "peak_source": src,
            "workload": "paged decode, 32/32 heads, D 128, fp16, 16-token pages, 1 appended token"}


def secondary_measurements(dev, only=None):
    """Other configurations of the path, each timed alone with CUDA events
    (median-free mean over the timed calls, after warm-up)."""
    import torch

    import paged_kv_cache_page_gb300 as pa
    from paged_kv_cache_page_gb300 import workloads as wl

    stream = torch.cuda.current_stream(dev)
    tpeak, tsrc = read_tensor_peak()
    hpeak, hsrc = read_peaks()
    res = {}
    if only == "prefill" or only is None:
        # causal prefill large enough for the tensor-core roofline to matter:
        # 16 sequences x 4096 new tokens, 32 heads, D 128, fp16, appended in-call
        w = wl.prefill_append(batch=16, lnew=4096, num_heads=32, head_dim=128, old_lo=0,
                              old_hi=0, pool=16 * 256, dtype="f16", dist="normal", seed=1006,
                              device=dev)
        out = torch.empty_like(w["q"])
        fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                       w["block_table"], k=w["k_new"], v=w["v_new"], causal=True,
                                       out=out, return_lse=False)
        us_append = time_calls(fn, 5 if only is None else 2, 2, stream)
        # the same attention with the 4096 tokens already cached: the prefill
        # kernel alone (one launch per call)
        full = (w["cache_seqlens"] + 4096).contiguous()
        fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], full,  # noqa: E731
                                       w["block_table"], causal=True, out=out, return_lse=False)
        us = time_calls(fn, 10 if only is None else 3, 3, stream)
        fl = attention_flops([4096] * 16, [4096] * 16, 32, 128, True)
        res["prefill_causal_16x4096"] = {
            "us": round(us, 1), "tflops": round(fl / us / 1e6, 1),
            "roofline": {"bound": "tensor", "achieved": round(fl / us / 1e6, 1), "peak": tpeak,
                         "unit": "TFLOP/s", "frac": round(fl / us / 1e6 / tpeak, 4),
                         "peak_source": tsrc, "kernel": "prefill_kernel<128, __half>"},
            "flops": fl, "us_with_append": round(us_append, 1),
            "note": "fp16, 32 heads x D 128, causal, keys read through 16-token pages"}
        if only == "prefill":
            return res
    if only is None:
        # the small-page reproduction shapes: 4 x 170 new tokens over a cached prefix
        w = wl.prefill_append(device=dev, seed=1004)
        out = torch.empty_like(w["q"])
        fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                       w["block_table"], k=w["k_new"], v=w["v_new"], causal=True,
                                       out=out, return_lse=False)
        us = time_calls(fn, 50, 5, stream, flush=True)
        old = w["cache_seqlens"].cpu().tolist()
        fl = attention_flops([170] * 4, [o + 170 for o in old], 32, 128, True)
        res["prefill_append_4x170"] = {"us": round(us, 1), "tflops": round(fl / us / 1e6, 2),
                                       "frac_tensor_peak": round(fl / us / 1e6 / tpeak, 4),
                                       "l2": "flushed between calls"}
    if only in (None, "gqa"):
        gqa_leg(dev, stream, only, hpeak, res)
        if only == "gqa":
            return res
    if only in (None, "unified"):
        unified_leg(dev, stream, only, hpeak, tpeak, res)
        if only == "unified":
            return res
    rest_legs(dev, stream, hpeak, res, only)
    if only == "spec":
        return res
    res["decode_sweep_graded"] = graded_sweep(dev)
    return res


def gqa_leg(dev, stream, only, hpeak, res):
    import torch

    import paged_kv_cache_page_gb300 as pa
    from paged_kv_cache_page_gb300 import workloads as wl

    # GQA split-KV decode on a contiguous 131072-token cache, lengths U[1024, 8192]
    w = wl.gqa_contiguous(device=dev)
    kc = torch.empty((8, w["capacity"], 8, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    n = w["k_rows"].shape[1]
    kc[:, :n] = w["k_rows"]
    vc[:, :n] = w["v_rows"]
    del w["k_rows"], w["v_rows"]
    out = torch.empty_like(w["q"])
    lse = torch.empty((8, 32, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, pa.fwd_kvcache_workspace_size(8, 1, 32, 8, 128, w["capacity"], 0)),
                     dtype=torch.uint8, device=dev)
    fn = lambda: pa.pa_fwd_kvcache(w["q"], kc, vc, w["cache_seqlens"], None, out=out, lse=lse,  # noqa: E731
                                   workspace=ws)
    # 132 MB of K/V against a 129 MB L2 (loaded evict-last): flush between calls
    us = time_calls(fn, 50 if only is None else 3, 10 if only is None else 3, stream, flush=True)
    us_warm = time_calls(fn, 100, 10, stream) if only is None else None
    lens = w["cache_seqlens"].cpu().tolist()
    by = sum(lens) * 8 * 128 * 2 * 2 + 8 * 32 * 128 * 2 * 2
    res["gqa_contiguous_split_kv"] = {"us": round(us, 1), "gbs": round(by / us / 1e3, 1),
                                      "frac_hbm_peak": round(by / us / 1e3 / hpeak, 4),
                                      "mean_len": sum(lens) / len(lens),
                                      "l2": "flushed between calls",
                                      "us_l2_warm": None if us_warm is None else round(us_warm, 1)}
    del kc, vc


def unified_leg(dev, stream, only, hpeak, tpeak, res):
    import torch

    import paged_kv_cache_page_gb300 as pa
    from paged_kv_cache_page_gb300 import workloads as wl

    # unified mixed batch in one launch: prefills of 100/500/1000 query tokens
    # over cached prefixes U[0, 2048] + 64 decodes with contexts U[1024, 4096],
    # bf16, causal; heads x head_dim 32 x 128 (the reported leg), then
    # 12 x 64 and 64 x 128
    for heads, hd in ((32, 128), (12, 64), (64, 128)):
        w = wl.unified_mixed(num_heads=heads, head_dim=hd, device=dev, seed=1005)
        out = torch.empty_like(w["q"])
        ws = torch.empty(max(1, pa.load_library().pa_fwd_varlen_workspace_size(
            67, w["q"].shape[0], w["max_seqlen_q"], heads, heads, hd, w["max_seqlen_k"])),
            dtype=torch.uint8, device=dev)
        fn = lambda: pa.pa_fwd_varlen_unified(w["q"], w["k_cache"], w["v_cache"],  # noqa: E731
                                              w["cu_seqlens_q"], w["seqlens_k"], w["block_table"],
                                              w["max_seqlen_q"], w["max_seqlen_k"], out=out,
                                              workspace=ws, return_lse=False)
        us = time_calls(fn, 20 if only is None else 3, 5 if only is None else 3, stream)
        cu = w["cu_seqlens_q"].cpu().tolist()
        kl = w["seqlens_k"].cpu().tolist()
        ql = [cu[i + 1] - cu[i] for i in range(len(kl))]
        by = sum(kl) * heads * hd * 2 * 2 + sum(ql) * heads * hd * 2 * 2
        fl = attention_flops(ql, kl, heads, hd, True)
        res[f"unified_mixed_{heads}x{hd}"] = {"us": round(us, 1), "gbs": round(by / us / 1e3, 1),
                                              "tflops": round(fl / us / 1e6, 1),
                                              "frac_hbm_peak": round(by / us / 1e3 / hpeak, 4),
                                              "frac_tensor_peak": round(fl / us / 1e6 / tpeak, 4)}
        del w, out, ws


def rest_legs(dev, stream, hpeak, res, only=None):
    import torch

    import paged_kv_cache_page_gb300 as pa
    from paged_kv_cache_page_gb300 import workloads as wl

    # multi-query (speculative) decode: 6 new tokens per sequence appended in the
    # call, causal among themselves, 64 sequences x ctx 4096, GQA 32/8, D 128, bf16
    w = wl.paged_decode(batch=64, ctx=4096, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        dtype="bf16", lnew=6, seed=1010, device=dev)
    out = torch.empty_like(w["q"])
    fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                   w["block_table"], k=w["k_new"], v=w["v_new"], causal=True,
                                   out=out, return_lse=False)
    us = time_calls(fn, 50 if only is None else 3, 5 if only is None else 3, stream)
    by = algorithmic_bytes(64, 4096, 6, 6, 32, 8, 128)
    res["spec_decode_lq6_b64_ctx4096"] = {"us": round(us, 1), "gbs": round(by / us / 1e3, 1),
                                          "frac_hbm_peak": round(by / us / 1e3 / hpeak, 4)}
    del w, out
    if only == "spec":
        return
    # rotary embedding of the new token (inside the decode launch): the same
    # paged decode step with and without it, B64 x ctx 4096, 32x128, fp16
    w = wl.paged_decode(batch=64, ctx=4096, lnew=1, seed=1011, device=dev)
    out = torch.empty_like(w["q"])
    ang = torch.arange(4096, dtype=torch.float64, device=dev)[:, None] * (
        10000.0 ** (-2.0 * torch.arange(64, dtype=torch.float64, device=dev) / 128))[None, :]
    cos, sin = ang.cos().half(), ang.sin().half()
    plain = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                      w["block_table"], k=w["k_new"], v=w["v_new"], out=out,
                                      return_lse=False)
    rotary = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                       w["block_table"], k=w["k_new"], v=w["v_new"], out=out,
                                       return_lse=False, rotary_cos=cos, rotary_sin=sin)
    us_plain = time_calls(plain, 50, 5, stream)
    us_rot = time_calls(rotary, 50, 5, stream)
    res["rotary_decode_b64_ctx4096"] = {"us": round(us_rot, 1), "us_without_rotary": round(us_plain, 1)}
    del w, out
    # page size 16 vs 256 (the block sizes compared on the flash-attn
    # integration page): writing a prompt's k/v into the cache (B64 x ctx
    # 512 / 1024 new tokens, 32 heads x D 128, fp16) and a decode step over
    # B64 x ctx 4096
    ps = {}
    for ctx in (512, 1024):
        row = []
        for page in (16, 256):
            w = wl.prefill_append(batch=64, lnew=ctx, num_heads=32, head_dim=128, old_lo=0,
                                  old_hi=0, pool=0, dtype="f16", seed=1012, device=dev,
                                  page_size=page)
            fn = lambda: pa.pa_append_kv(w["k_cache"], w["v_cache"], w["k_new"], w["v_new"],  # noqa: E731
                                         w["cache_seqlens"], w["block_table"])
            row.append(round(time_calls(fn, 30, 5, stream), 1))
            del w
        ps[f"append_b64_ctx{ctx}_us"] = {"page16": row[0], "page256": row[1]}
    row = []
    for page in (16, 256):
        w = wl.paged_decode(batch=64, ctx=4096, lnew=1, seed=1013, device=dev, page_size=page)
        out = torch.empty_like(w["q"])
        fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                       w["block_table"], k=w["k_new"], v=w["v_new"], out=out,
                                       return_lse=False)
        row.append(round(time_calls(fn, 50, 5, stream), 1))
        del w, out
    ps["decode_b64_ctx4096_us"] = {"page16": row[0], "page256": row[1]}
    res["page_size_16_vs_256"] = ps
    # tiny paged decode (launch-latency bound)
    w = wl.tiny_decode(device=dev)
    fn = lambda: pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],  # noqa: E731
                                   w["block_table"], scale=w["scale"])
    res["tiny_decode"] = {"us": round(time_calls(fn, 200, 20, stream), 2)}
    return res


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("decode.cu", "pa_common.cuh", "pa_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_page_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, or None if
    the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "decode_paged_b256_ctx4096.txt")
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256_16") != kernel_source_hash():
            return None
        return float(fields["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0:  # first sample before timing
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_seed(rank):
    """Seed of a rank's batch: every rank is an independent replica with its
    own sequences (weak scaling; no data crosses ranks)."""
    return 1002 + rank


def max_over_ranks(x, world, device=None):
    """The largest `x` over all ranks (the slowest rank's time), `x` itself on
    one rank; on whatever backend the process group was created with."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes, steps, world, elapsed_ms):
    """Whole-job throughput in GB/s: the bytes all ranks processed over the
    slowest rank's time."""
    return step_bytes * steps * world / (elapsed_ms * 1e-3) / 1e9


def cpu_oracle_rate(w_cpu, seqs, lnew):
    """Time the CPU oracle on sequences `seqs` of the workload; returns
    (GB/s-equivalent, wall seconds, process CPU seconds)."""
    import numpy as np

    import oracle

    q = w_cpu["q"]
    t0, c0 = time.perf_counter(), time.process_time()
    nbytes = 0
    for b in seqs:
        old = int(w_cpu["cache_seqlens"][b])
        oracle.fwd_kvcache(q[b:b + 1], w_cpu["k_pages"][b], w_cpu["v_pages"][b], [old],
                           np.arange(w_cpu["k_pages"][b].shape[0])[None],
                           k_new=w_cpu["k_new"][b:b + 1], v_new=w_cpu["v_new"][b:b + 1],
                           scale=w_cpu["scale"], causal=False)
        nbytes += algorithmic_bytes(1, old + lnew, lnew, q.shape[1], q.shape[2],
                                    w_cpu["k_new"].shape[2], q.shape[3])
    dt, ct = time.perf_counter() - t0, time.process_time() - c0
    return nbytes / dt / 1e9, dt, ct


_BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                     "BLIS_NUM_THREADS", "NUMEXPR_NUM_THREADS")


def cpu_single_thread(budget_s=3.0):
    """The oracle on one host thread: a child process with every BLAS/OpenMP
    thread count pinned to 1, on a host-drawn sample of the same shape (two
    sequences of ctx 4096, 32x128 heads); returns its GB/s-equivalent or None."""
    env = dict(os.environ)
    for k in _BLAS_THREAD_VARS:
        env[k] = "1"
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-single-thread",
                            str(budget_s)], env=env, capture_output=True, text=True, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])["gbs"]
    except Exception:
        return None


def run_cpu_single_thread(budget_s):
    from paged_kv_cache_page_gb300 import workloads as wl

    w = wl.paged_decode(2, WORKLOAD["ctx"], lnew=WORKLOAD["lnew"], seed=1002, device="cpu")
    hs = host_sample(w, [0, 1])
    total_b, total_s = 0.0, 0.0
    while total_s < budget_s:
        rate, dt, _ = cpu_oracle_rate(hs, [0, 1], WORKLOAD["lnew"])
        total_b += rate * dt * 1e9
        total_s += dt
    print(json.dumps({"gbs": round(total_b / total_s / 1e9, 4), "seconds": round(total_s, 2)}))


def host_sample(w, seqs):
    """Copy the pages of `seqs` to the host as float64 arrays for the oracle."""
    table = w["block_table"]
    out = {"q": w["q"].double().cpu().numpy(), "k_new": w["k_new"].double().cpu().numpy(),
           "v_new": w["v_new"].double().cpu().numpy(), "cache_seqlens": w["cache_seqlens"].cpu(),
           "scale": w["scale"], "k_pages": {}, "v_pages": {}}
    for b in seqs:
        npg = -(-int(w["cache_seqlens"][b]) // 16)
        pages = table[b, :npg].long()
        out["k_pages"][b] = w["k_cache"][pages].double().cpu().numpy()
        out["v_pages"][b] = w["v_cache"][pages].double().cpu().numpy()
    return out


def cpu_baseline(w, budget_s=10.0, max_seqs=8):
    """Oracle throughput on a bounded sample: up to `max_seqs` sequences of the
    workload (held on the host in float64), passed repeatedly until about
    `budget_s` seconds of CPU work have been timed.  `threads` is the number
    the run actually kept busy (process CPU time / wall time); `single_thread`
    the same oracle with every BLAS/OpenMP thread count pinned to 1."""
    lnew = WORKLOAD["lnew"]
    seqs = list(range(min(max_seqs, w["q"].shape[0])))
    hs = host_sample(w, seqs)
    total_bytes, total_s, total_cpu, passes = 0.0, 0.0, 0.0, 0
    while total_s < budget_s and passes < 1000:
        rate, dt, ct = cpu_oracle_rate(hs, seqs, lnew)
        total_bytes += rate * dt * 1e9
        total_s += dt
        total_cpu += ct
        passes += 1
    rate = total_bytes / total_s / 1e9
    threads = round(total_cpu / total_s, 1)
    single = cpu_single_thread()
    return {"value": round(rate, 3), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "threads": threads, "single_thread": single,
            "sample": f"{len(seqs)} of {WORKLOAD['batch']} sequences (ctx {WORKLOAD['ctx']}, "
                      f"32x128 heads, fp16 values widened to float64) through the numpy oracle, "
                      f"{passes} passes, {total_s:.1f} s on {os.cpu_count()} host cores; "
                      f"threads = process CPU time / wall time ({threads}); single_thread = the "
                      f"same oracle with BLAS/OpenMP pinned to one thread, 2 sequences"}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, on rank 0 only."""
    if rank != 0:
        return
    import numpy as np

    import oracle  # noqa: F401
    from paged_kv_cache_page_gb300 import workloads as wl

    B = WORKLOAD["batch"]
    # Draw the workload on the GPU when there is one (drawing 17 GB on the host
    # takes minutes), else a smaller host draw of the same shape per sequence.
    import torch
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    if dev == "cpu":
        w = wl.paged_decode(8, WORKLOAD["ctx"], lnew=WORKLOAD["lnew"], seed=1002, device="cpu")
    else:
        w = wl.paged_decode(B, WORKLOAD["ctx"], lnew=WORKLOAD["lnew"], seed=1002, device=dev)
    seqs_per_step = 2
    total = args.warmup + args.steps
    seqs = [i % w["q"].shape[0] for i in range(total * seqs_per_step)]
    hs = host_sample(w, sorted(set(seqs)))
    lnew = WORKLOAD["lnew"]
    for i in range(args.warmup):
        cpu_oracle_rate(hs, seqs[i * seqs_per_step:(i + 1) * seqs_per_step], lnew)
    t0, c0 = time.perf_counter(), time.process_time()
    nbytes = 0
    for i in range(args.warmup, total):
        s = seqs[i * seqs_per_step:(i + 1) * seqs_per_step]
        cpu_oracle_rate(hs, s, lnew)
        nbytes += algorithmic_bytes(len(s), WORKLOAD["ctx"], lnew, lnew, 32, 32, 128)
    dt = time.perf_counter() - t0
    threads = round((time.process_time() - c0) / dt, 1)
    value = nbytes / dt / 1e9
    line = {"metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": dict(WORKLOAD, sample=f"{seqs_per_step} sequences per step"),
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": os.cpu_count(),
                             "kind": "oracle", "threads": threads,
                             "sample": f"{seqs_per_step} of {B} sequences per step; threads = "
                                       f"process CPU time / wall time"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    del np
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-single-thread", type=float, default=None,
                    help=argparse.SUPPRESS)
    ap.add_argument("--batch", type=int, default=WORKLOAD["batch"],
                    help="smaller batches are for profiling runs only")
    ap.add_argument("--ctx", type=int, default=WORKLOAD["ctx"])
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other configurations (prefill, GQA split-KV, tiny decode)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the paged decode sweep (ctx 512..4096 x batch 1..256) instead")
    ap.add_argument("--only", choices=["prefill", "gqa", "unified", "spec", "graded"],
                    help="time only this secondary leg (for profiling runs)")
    args = ap.parse_args()
    WORKLOAD["batch"], WORKLOAD["ctx"] = args.batch, args.ctx
    kv_gb = args.batch * args.ctx * 32 * 128 * 2 * 2 / 1e9
    WORKLOAD["l2"] = (f"inputs ({kv_gb:.1f} GB of K/V) larger than L2; no flush" if kv_gb > 4 * 0.129
                      else f"inputs ({kv_gb:.2f} GB of K/V) within 4x L2")
    args.warmup = max(3, args.warmup)
    if args.cpu_single_thread is not None:
        run_cpu_single_thread(args.cpu_single_thread)
        return
    rank, world, local = dist_env()

    import torch
    import torch.distributed as dist

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            dist.destroy_process_group()
        return

    import paged_kv_cache_page_gb300 as pa
    from paged_kv_cache_page_gb300 import workloads as wl

    pa.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.only == "graded":
        print(json.dumps(graded_sweep(dev)), flush=True)
        return
    if args.only:
        print(json.dumps(secondary_measurements(dev, only=args.only)), flush=True)
        return
    if args.sweep:
        decode_sweep(dev)
        return
    B, ctx, lnew = WORKLOAD["batch"], WORKLOAD["ctx"], WORKLOAD["lnew"]
    hq, hkv, d = WORKLOAD["num_q_heads"], WORKLOAD["num_kv_heads"], WORKLOAD["head_dim"]
    # each rank is an independent replica with its own sequences (weak scaling)
    w = wl.paged_decode(B, ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, lnew=lnew,
                        seed=replica_seed(rank), device=dev)
    out = torch.empty((B, lnew, hq, d), dtype=torch.float16, device=dev)
    lse = torch.empty((B, hq, lnew), dtype=torch.float32, device=dev)
    ws_bytes = pa.fwd_kvcache_workspace_size(B, lnew, hq, hkv, d, ctx, 0)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    launches_per_step = 1 + (1 if ws_bytes > 0 else 0)
    stream = torch.cuda.current_stream(dev)

    def step():
        pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                          w["block_table"], k=w["k_new"], v=w["v_new"], scale=w["scale"],
                          out=out, lse=lse, workspace=ws, max_seqlen_k=ctx)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_all1.record(stream)
        barrier()
    elapsed_ms = t_all0.elapsed_time(t_all1)
    per_launch_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    step_bytes = algorithmic_bytes(B, ctx, lnew, lnew, hq, hkv, d)
    value = whole_job_gbs(step_bytes, args.steps, world, elapsed_ms)

    # end-to-end through the public API with host buffers: inputs of the step
    # (q, new k/v, lengths, block table) copied from pinned host memory, output
    # and lse read back, every step.
    h_q = w["q"].cpu().pin_memory()
    h_k = w["k_new"].cpu().pin_memory()
    h_v = w["v_new"].cpu().pin_memory()
    h_sl = w["cache_seqlens"].cpu().pin_memory()
    h_bt = w["block_table"].cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d_q, d_k, d_v = torch.empty_like(w["q"]), torch.empty_like(w["k_new"]), torch.empty_like(w["v_new"])
    d_sl, d_bt = torch.empty_like(w["cache_seqlens"]), torch.empty_like(w["block_table"])
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_sl, h_bt))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    def e2e_step():
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_sl.copy_(h_sl, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        pa.pa_fwd_kvcache(d_q, w["k_cache"], w["v_cache"], d_sl, d_bt, k=d_k, v=d_v,
                          scale=w["scale"], out=out, lse=lse, workspace=ws, max_seqlen_k=ctx)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = whole_job_gbs(step_bytes, args.steps, world, e2e_ms)

    if rank == 0:
        peak, peak_src = read_peaks()
        achieved = step_bytes / (per_launch_ms * 1e-3) / 1e9
        traffic = profiled_traffic()
        cpu = None
        if not args.no_cpu_baseline and world >= 1:
            cpu = cpu_baseline(w)
        secondary = None
        if not args.no_secondary:
            del w
            torch.cuda.empty_cache()
            secondary = secondary_measurements(dev)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": dict(WORKLOAD, parallelism=f"replicas x{world}",
                           us_per_call=round(elapsed_ms / args.steps * 1e3, 2),
                           algorithmic_bytes_per_step=step_bytes),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "peak_source": f"{peak_src} (copy bandwidth)",
                         "kernel": "decode_kernel<128, half, 1>",
                         # the copy peak counts a read and a write stream; a
                         # read-only stream can run slightly above it, so the
                         # nominal HBM3e rate is given beside it
                         "peak_nominal": HBM_NOMINAL_GBS,
                         "frac_nominal": round(achieved / HBM_NOMINAL_GBS, 4)},
            "clocks": clk.summary(),
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "cpu_baseline": cpu,
            "secondary": secondary,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
