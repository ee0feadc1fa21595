"""GPU parity of the split-KV decode path (pa_fwd_kvcache with Lq*G <= 16)
against the CPU oracle, plus the standalone combine and the device-side error
word.  Calls go through the C ABI (ctypes binding)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import LSE_TOL, OUT_TOL, assert_close, bits, np64, oracle_kvcache

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(w, **kw):
    err = pa.new_err_word(DEV)
    out, lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                 w["block_table"], k=w.get("k_new"), v=w.get("v_new"),
                                 scale=w["scale"], causal=w["causal"], err=err, **kw)
    torch.cuda.synchronize()
    assert err[0].item() == 0, f"device error word {err.tolist()}"
    return out, lse


def test_tiny_paged_decode_gqa():
    w = wl.tiny_decode(device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "f16")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("batch,ctx", [(1, 512), (3, 1024), (8, 2048), (2, 4096)])
def test_paged_decode_with_append(dtype, batch, ctx):
    w = wl.paged_decode(batch, ctx, dtype=dtype, lnew=1, seed=7 + batch + ctx, device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    kc0 = w["k_cache"].clone()
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, dtype)
    # the appended token landed in its page slot, bit for bit, and nothing else changed
    kn, table = bits(w["k_new"]), w["block_table"].cpu().numpy()
    expect, _ = oracle.append_kv(bits(kc0), bits(kc0), kn, kn, w["cache_seqlens"].cpu().numpy(),
                                 table)
    assert np.array_equal(bits(w["k_cache"]), expect)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 0])
def test_split_count_does_not_change_result(splits):
    lens = [1000, 37, 700, 16, 1]
    w = wl.paged_decode(5, 0, num_q_heads=8, num_kv_heads=2, head_dim=128, lens=lens, seed=11,
                        device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w, num_splits=splits)
    assert_close(out, lse, ref_o, ref_l, "f16")


@pytest.mark.parametrize("hq,hkv,lq", [(8, 8, 1), (16, 2, 1), (8, 2, 4)])
def test_stale_workspace_bytes(hq, hkv, lq):
    """A workspace holding other bytes (split counts of 0x01010101, finite
    partials) gives the same result: the CUDA-core decode (Lq*G <= 2) and the
    packed tensor-core items (Lq*G > 2) rewrite every sequence's split count."""
    lens = [900, 5, 2000, 4, 17, 600]
    w = wl.paged_decode(len(lens), 0, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                        lens=lens, lnew=lq, seed=21 + hq + lq, device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    cap = w["block_table"].shape[1] * 16
    nbytes = pa.fwd_kvcache_workspace_size(len(lens), lq, hq, hkv, 128, cap, 0)
    assert nbytes > 0
    ws = torch.full((nbytes,), 0x01, dtype=torch.uint8, device=DEV)
    out, lse = run(w, workspace=ws)
    assert_close(out, lse, ref_o, ref_l, "f16")


def test_split_matches_unsplit_closely():
    w = wl.paged_decode(3, 2048, num_q_heads=4, num_kv_heads=4, seed=12, device=DEV)
    o1, l1 = run(w, num_splits=1)
    o4, l4 = run(w, num_splits=4)
    assert (np64(o1) - np64(o4)).__abs__().max() <= OUT_TOL["f16"]
    assert (np64(l1) - np64(l4)).__abs__().max() <= 1e-5


@pytest.mark.parametrize("lq,hq,hkv,causal", [(2, 4, 2, True), (4, 8, 4, True), (8, 4, 4, True),
                                              (3, 2, 2, False), (2, 8, 2, True)])
def test_multi_query_decode(lq, hq, hkv, causal):
    lens = [100, 333, 17]
    w = wl.paged_decode(3, 0, num_q_heads=hq, num_kv_heads=hkv, head_dim=64, lens=lens,
                        lnew=lq, seed=13 + lq, device=DEV, dtype="bf16")
    w["causal"] = causal
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "bf16")


def test_page_placement_is_bit_invariant():
    w = wl.paged_decode(4, 1024, num_q_heads=8, num_kv_heads=8, seed=14, device=DEV)
    out1, lse1 = run(w)
    # move every page to a new physical slot (random permutation of the pool)
    pool = w["k_cache"].shape[0]
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(5)).to(DEV)
    w2 = dict(w)
    k2 = torch.empty_like(w["k_cache"])
    v2 = torch.empty_like(w["v_cache"])
    k2[perm] = w["k_cache"]
    v2[perm] = w["v_cache"]
    w2["k_cache"], w2["v_cache"] = k2, v2
    w2["block_table"] = perm.to(torch.int32)[w["block_table"].long()]
    out2, lse2 = run(w2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_contiguous_gqa_split_kv_cache():
    """B8, 32 q / 8 kv heads, D 128, bf16, lengths U[1024, 8192] in a
    131072-token contiguous cache: the launch the benchmark times, every row."""
    w = wl.gqa_contiguous(device=DEV)
    B, cap = 8, w["capacity"]
    hkv, d = w["num_kv_heads"], w["head_dim"]
    kc = torch.zeros((B, cap, hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    n = w["k_rows"].shape[1]
    kc[:, :n] = w["k_rows"]
    vc[:, :n] = w["v_rows"]
    ww = dict(w, k_cache=kc, v_cache=vc)
    ref_o, ref_l = oracle_kvcache(ww)
    out, lse = run(ww)
    assert_close(out, lse, ref_o, ref_l, "bf16")


def test_empty_and_single_key_sequences():
    w = wl.paged_decode(3, 0, num_q_heads=4, num_kv_heads=2, head_dim=128, lens=[0, 1, 5],
                        seed=15, device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    # a single key returns its value exactly
    v0 = w["v_cache"][w["block_table"][1, 0].long(), 0]  # [Hkv, D]
    assert torch.equal(out[1, 0, 0], v0[0]) and torch.equal(out[1, 0, 3], v0[1])
    assert_close(out, lse, ref_o, ref_l, "f16")


@pytest.mark.parametrize("S,D", [(5, 128), (32, 128), (32, 64), (45, 128), (70, 64)])
def test_split_combine_entry_point(S, D):
    """Up to 32 splits take the lane-per-split path, more take the serial one;
    both skip empty splits (LSE -inf) without reading their partials."""
    g = torch.Generator().manual_seed(16 + S)
    B, Lq, Hq = 4, 2, 4
    o = torch.randn((S, B, Lq, Hq, D), generator=g).float()
    l = torch.randn((S, B, Lq, Hq), generator=g).float() * 3
    l[2, 1] = float("-inf")  # an empty split
    o[2, 1] = float("nan")   # whose partial must not be read
    l[S - 1, 0] = float("-inf")
    o[S - 1, 0] = float("nan")
    l[:, 3, 1] = float("-inf")  # a query row with no keys at all
    nsp = torch.tensor([S, 3, 0, S], dtype=torch.int32)
    out = torch.full((B, Lq, Hq, D), 7.0, dtype=torch.float16, device=DEV)
    lse = torch.full((B, Hq, Lq), 7.0, dtype=torch.float32, device=DEV)
    pa.pa_split_combine(o.to(DEV), l.to(DEV), out, lse, nsp.to(DEV))
    torch.cuda.synchronize()
    for b in range(B):
        n = int(nsp[b])
        if n == 0:
            assert torch.all(out[b] == 7.0) and torch.all(lse[b] == 7.0)
            continue
        ref_o, ref_l = oracle.combine_splits(o[:n, b].double().numpy(), l[:n, b].double().numpy())
        got_o, got_l = np64(out[b]), np64(lse[b]).transpose(1, 0)
        empty = np.isneginf(ref_l)
        assert np.all(got_o[empty] == 0) and np.all(np.isneginf(got_l[empty]))
        assert np.abs(got_o[~empty] - ref_o[~empty]).max() <= OUT_TOL["f16"]
        assert np.abs(got_l[~empty] - ref_l[~empty]).max() <= LSE_TOL


def test_out_of_range_pages_report_and_do_not_fault():
    w = wl.paged_decode(2, 64, num_q_heads=2, num_kv_heads=2, head_dim=64, lnew=1, seed=17,
                        device=DEV)
    pool = w["k_cache"].shape[0]
    w["block_table"][1, 2] = pool + 1000  # outside the pool
    kc0, vc0 = w["k_cache"].clone(), w["v_cache"].clone()
    err = pa.new_err_word(DEV)
    pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"], w["block_table"],
                      k=w["k_new"], v=w["v_new"], err=err)
    torch.cuda.synchronize()
    assert err[0].item() == pa.PA_DEVERR_PAGE_OOB and err[1].item() == 1
    # sequence 0's append still happened; nothing was written through the bad entry
    assert not torch.equal(w["k_cache"], kc0)
    pg = w["block_table"][0, 3].long()
    assert torch.equal(w["k_cache"][pg, 15], w["k_new"][0, 0])


def test_lengths_beyond_table_report():
    w = wl.paged_decode(2, 64, num_q_heads=2, num_kv_heads=2, head_dim=64, seed=18, device=DEV)
    w["cache_seqlens"][0] = 65  # table holds 4 pages = 64 tokens
    err = pa.new_err_word(DEV)
    out, lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                 w["block_table"], err=err, max_seqlen_k=64)
    torch.cuda.synchronize()
    assert err[0].item() == pa.PA_DEVERR_LENGTH and err[1].item() == 0
    ref_o, ref_l = oracle_kvcache(w, rows=[1])
    assert_close(out[1:], lse[1:], ref_o, ref_l, "f16")


def test_full_size_decode_sweep_point_sampled():
    """ctx 4096 x batch 256, 32/32 heads, D 128, fp16 with one appended token:
    the launch configuration the benchmark times; the first and the last 8
    sequences (the first and the last work items the persistent grid deals)
    and two in between are checked."""
    w = wl.paged_decode(256, 4096, lnew=1, seed=1002, device=DEV)
    rows = list(range(8)) + [77, 128] + list(range(248, 256))
    ref_o, ref_l = oracle_kvcache(w, rows=rows)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "f16", rows=rows)


@pytest.mark.parametrize("batch,ctx", [(4, 4096), (8, 4096), (16, 2048)])
def test_graded_sweep_split_points_sampled(batch, ctx):
    """Graded points of the decode sweep that run the balanced split
    schedule at their benchmarked size (32/32 heads, D 128, fp16, one
    appended token, automatic splits): ctx 4096 x B4 by the whole-split cost
    test, ctx 4096 x B8 and ctx 2048 x B16 by the idle-last-round test of the
    host gate.  The first and the last two sequences are checked."""
    w = wl.paged_decode(batch, ctx, lnew=1, seed=1002 + batch, device=DEV)
    rows = [0, 1, batch - 2, batch - 1]
    ref_o, ref_l = oracle_kvcache(w, rows=rows)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "f16", rows=rows)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv,lq,splits", [(32, 8, 1, 0), (64, 8, 1, 0), (16, 4, 2, 3),
                                              (12, 4, 1, 5), (8, 1, 1, 0), (6, 2, 2, 0),
                                              (32, 8, 6, 0), (16, 2, 4, 3), (12, 4, 7, 0)])
def test_gqa_rows_share_each_key(dtype, d, hq, hkv, lq, splits):
    """3-32 query rows per kv head (GQA decode, multi-query decode with a
    causal in-call append): up to 16 rows the decode kernel's warp-level
    tensor-core consumer (8 rows per MMA tile; padded row counts 3 and 6),
    past 16 the tcgen05 engine's packed items (21, 24 and 32 rows); ragged
    lengths whose last page is partial, and forced split counts."""
    lens = [1000, 37, 700, 16, 8, 513]
    w = wl.paged_decode(len(lens), 0, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, lens=lens,
                        lnew=lq, seed=31 + hq + lq + d, device=DEV, dtype=dtype)
    w["causal"] = lq > 1
    ref_o, ref_l = oracle_kvcache(w)
    kc0 = w["k_cache"].clone()
    out, lse = run(w, num_splits=splits)
    assert_close(out, lse, ref_o, ref_l, dtype)
    kn, table = bits(w["k_new"]), w["block_table"].cpu().numpy()
    expect, _ = oracle.append_kv(bits(kc0), bits(kc0), kn, kn, w["cache_seqlens"].cpu().numpy(),
                                 table)
    assert np.array_equal(bits(w["k_cache"]), expect)


def test_speculative_decode_bench_shape_sampled():
    """The multi-query (speculative) decode the benchmark times: 64 sequences
    at ctx 4096, 6 new tokens appended in the call and attended causally, GQA
    32/8, D 128, bf16 (query blocks of 24 rows per kv head: the tensor-core
    engine).  The first and the last 4 sequences are checked against the
    oracle, and their appended slots bit for bit."""
    w = wl.paged_decode(batch=64, ctx=4096, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        dtype="bf16", lnew=6, seed=1010, device=DEV)
    w["causal"] = True
    rows = [0, 1, 2, 3, 60, 61, 62, 63]
    ref_o, ref_l = oracle_kvcache(w, rows=rows)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", rows=rows)
    table = w["block_table"]
    for b in rows:
        old = int(w["cache_seqlens"][b])
        for i in range(6):
            pos = old + i
            page = table[b, pos // 16].long()
            assert torch.equal(w["k_cache"][page, pos % 16], w["k_new"][b, i])
            assert torch.equal(w["v_cache"][page, pos % 16], w["v_new"][b, i])
