"""CUDA-graph replay of the fixed-capacity launches.

The unified launch's grid depends only on host-known capacities (the batch
entry count, max_seqlen_q, max_seqlen_k, total_q); every length, split count
and page lives on the device.  So one captured graph serves any batch that
fits the capacities, padding entries included -- vLLM #6052 "Unify the
kernel used in flash attention backend", the comment on CUDA graphs padding
the batch to the captured size with empty entries.  These tests
capture once, then rewrite lengths, tables and inputs in place and replay: the
replay must match the oracle on the new batch and be bit-identical to an eager
call on the same buffers."""

import numpy as np
import pytest
import torch

import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import OUT_TOL, np64, oracle_kvcache
from test_gpu_varlen import check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def capture(fn):
    """One eager warm-up call on a side stream, then capture fn in a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def load_batch(static, w, page_offset):
    """Write batch w into the static capacity buffers: its q rows at the start
    of q, its pages at page_offset in the shared pool, padding entries (empty
    sequences) after its own."""
    B = w["cu_seqlens_q"].numel() - 1
    cap_b = static["seqlens_k"].numel()
    total = int(w["cu_seqlens_q"][-1])
    static["q"][:total].copy_(w["q"])
    static["q"][total:].normal_()
    cu = torch.full((cap_b + 1,), total, dtype=torch.int32, device=DEV)
    cu[:B + 1] = w["cu_seqlens_q"]
    static["cu_seqlens_q"].copy_(cu)
    lens = torch.zeros(cap_b, dtype=torch.int32, device=DEV)
    lens[:B] = w["seqlens_k"]
    static["seqlens_k"].copy_(lens)
    table = torch.zeros_like(static["block_table"])
    npg = w["block_table"].shape[1]
    table[:B, :npg] = w["block_table"] + page_offset
    static["block_table"].copy_(table)
    pool = w["k_cache"].shape[0]
    static["k_cache"][page_offset:page_offset + pool].copy_(w["k_cache"])
    static["v_cache"][page_offset:page_offset + pool].copy_(w["v_cache"])


def test_unified_graph_replay_with_new_lengths():
    kw = dict(num_heads=16, num_kv_heads=4, head_dim=128, device=DEV)
    wa = wl.unified_mixed(prefill_lens=(7, 300), prefix_hi=600, num_decode=9, ctx_lo=1,
                          ctx_hi=900, seed=501, **kw)
    wb = wl.unified_mixed(prefill_lens=(120, 33, 5), prefix_hi=500, num_decode=4, ctx_lo=100,
                          ctx_hi=1000, seed=502, **kw)
    cap_b, cap_q, cap_seq_q, cap_seq_k = 16, 512, 320, 1100
    pool = wa["k_cache"].shape[0] + wb["k_cache"].shape[0]
    npg = -(-cap_seq_k // 16)
    hq, hkv, d = 16, 4, 128
    static = dict(
        q=torch.zeros((cap_q, hq, d), dtype=torch.bfloat16, device=DEV),
        k_cache=torch.zeros((pool, 16, hkv, d), dtype=torch.bfloat16, device=DEV),
        v_cache=torch.zeros((pool, 16, hkv, d), dtype=torch.bfloat16, device=DEV),
        cu_seqlens_q=torch.zeros(cap_b + 1, dtype=torch.int32, device=DEV),
        seqlens_k=torch.zeros(cap_b, dtype=torch.int32, device=DEV),
        block_table=torch.zeros((cap_b, npg), dtype=torch.int32, device=DEV),
        scale=wa["scale"], causal=True)
    out = torch.full((cap_q, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((hq, cap_q), float("nan"), device=DEV)
    err = pa.new_err_word(DEV)

    def call(o=out, l=lse):
        pa.pa_fwd_varlen_unified(static["q"], static["k_cache"], static["v_cache"],
                                 static["cu_seqlens_q"], static["seqlens_k"],
                                 static["block_table"], cap_seq_q, cap_seq_k, scale=static["scale"],
                                 causal=True, out=o, lse=l, err=err)

    load_batch(static, wa, 0)
    g = capture(call)
    for w, off in ((wa, 0), (wb, wa["k_cache"].shape[0]), (wa, 0)):
        load_batch(static, w, off)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert err[0].item() == 0
        B = w["cu_seqlens_q"].numel() - 1
        check(static, out, lse, "bf16", seqs=list(range(B)))
        # an eager call on the same buffers gives the same bits
        out_e = torch.full_like(out, float("nan"))
        lse_e = torch.full_like(lse, float("nan"))
        call(out_e, lse_e)
        torch.cuda.synchronize()
        total = int(w["cu_seqlens_q"][-1])
        assert torch.equal(out[:total], out_e[:total])
        assert torch.equal(lse[:, :total], lse_e[:, :total])


def test_decode_graph_replay_with_new_lengths():
    """Paged decode (MHA: the fused decode kernel; GQA: the engine) captured at
    a capacity of 1024 keys, replayed after the cache lengths change in place
    (an empty sequence included)."""
    for hq, hkv in ((8, 8), (16, 4)):
        w = wl.paged_decode(batch=6, ctx=1024, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                            dtype="f16", device=DEV, seed=600 + hq)
        lens = w["cache_seqlens"]  # the captured buffer; rewritten in place below
        out = torch.empty((6, 1, hq, 128), dtype=torch.float16, device=DEV)
        lse = torch.empty((6, hq, 1), dtype=torch.float32, device=DEV)

        def call(o=out, l=lse):
            pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], lens, w["block_table"],
                              out=o, lse=l, max_seqlen_k=1024)

        g = capture(call)
        gen = torch.Generator().manual_seed(hq)
        for trial in range(3):
            new = torch.randint(1, 1025, (6,), generator=gen, dtype=torch.int32)
            if trial == 1:
                new[2] = 0
            lens.copy_(new.to(DEV))
            out.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            ref_o, ref_l = oracle_kvcache(w)
            e = np.abs(np64(out) - ref_o).max()
            assert e <= OUT_TOL["f16"], (hq, trial, e)
            out_e = torch.empty_like(out)
            lse_e = torch.empty_like(lse)
            call(out_e, lse_e)
            torch.cuda.synchronize()
            assert torch.equal(out, out_e)
            assert torch.equal(lse, lse_e)
