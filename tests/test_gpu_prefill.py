"""GPU parity of the tensor-core (tcgen05) prefill path of pa_fwd_kvcache
(query blocks of more than 8 rows per kv head) against the CPU oracle."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import assert_close, bits, np64, oracle_kvcache

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


def test_causal_prefill_with_append_config():
    """B 4, 170 new tokens, 32 heads, D 128, fp16 U[0,1), cached prefix
    U[0,512], distinct pages from a 1000-page pool (the small-page
    reproduction's shapes)."""
    w = wl.prefill_append(device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    kc0, vc0 = bits(w["k_cache"]), bits(w["v_cache"])
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "f16")
    table = w["block_table"].cpu().numpy()
    ek, ev = oracle.append_kv(kc0, vc0, bits(w["k_new"]), bits(w["v_new"]),
                              w["cache_seqlens"].cpu().numpy(), table)
    assert np.array_equal(bits(w["k_cache"]), ek) and np.array_equal(bits(w["v_cache"]), ev)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d,hq,hkv,lnew,causal", [(64, 8, 2, 300, True), (128, 4, 4, 129, False),
                                                  (64, 4, 1, 257, True), (128, 6, 3, 40, True)])
def test_prefill_shapes(dtype, d, hq, hkv, lnew, causal):
    w = wl.prefill_append(batch=3, lnew=lnew, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                          dtype=dtype, dist="normal", seed=31 + lnew + d, device=DEV)
    w["causal"] = causal
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, dtype)


def test_prefill_contiguous_cache():
    g = torch.Generator(device=DEV).manual_seed(41)
    B, cap, hkv, hq, d, lq = 2, 1000, 2, 4, 128, 200
    kc = torch.randn((B, cap, hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    vc = torch.randn((B, cap, hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn((B, lq, hq, d), generator=g, device=DEV).to(torch.bfloat16)
    w = dict(q=q, k_cache=kc, v_cache=vc, k_new=None, v_new=None,
             cache_seqlens=torch.tensor([700, 233], dtype=torch.int32, device=DEV),
             block_table=None, scale=d ** -0.5, causal=True)
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, "bf16")


def test_causal_rows_without_visible_keys():
    """Lq > Lk: the first Lq - Lk rows see no key (O = 0, LSE = -inf)."""
    w = wl.paged_decode(2, 0, num_q_heads=4, num_kv_heads=4, head_dim=64, lens=[10, 150],
                        seed=42, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(43)
    w["q"] = torch.randn((2, 20, 4, 64), generator=g, device=DEV).half()
    w["causal"] = True
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert torch.all(out[0, :10] == 0) and torch.all(torch.isneginf(lse[0, :, :10]))
    assert_close(out, lse, ref_o, ref_l, "f16")


def test_small_page_reproduction_loop_does_not_fault():
    """The flash-attention small-page reproduction: B 4, 170 new tokens appended
    at position 0 through randint block tables (duplicates allowed), repeated.
    Page aliasing makes the cache contents racy, so only the absence of faults,
    of device errors and of non-finite outputs is checked."""
    gen = torch.Generator(device=DEV).manual_seed(44)
    num_blocks, bs, seq, heads, d = 1000, 4, 170, 32, 128
    kc = torch.rand((num_blocks, 16, heads, d), generator=gen, device=DEV).half()
    vc = torch.rand((num_blocks, 16, heads, d), generator=gen, device=DEV).half()
    seql = torch.zeros(bs, dtype=torch.int32, device=DEV)
    err = pa.new_err_word(DEV)
    for _ in range(50):
        q = torch.rand((bs, seq, heads, d), generator=gen, device=DEV).half()
        k = torch.rand((bs, seq, heads, d), generator=gen, device=DEV).half()
        v = torch.rand((bs, seq, heads, d), generator=gen, device=DEV).half()
        table = torch.randint(0, num_blocks, (bs, (seq + 15) // 16), generator=gen, device=DEV,
                              dtype=torch.int32)
        out, _ = pa.pa_fwd_kvcache(q, kc, vc, seql, table, k=k, v=v, causal=True, err=err)
    torch.cuda.synchronize()
    assert err[0].item() == 0
    assert torch.isfinite(out).all()


def test_long_causal_prefill_sampled():
    """16 x 2048 new tokens, 32 heads, D 128, bf16: 16 query tiles per head;
    two sequences checked at four heads each against the oracle."""
    w = wl.prefill_append(batch=16, lnew=2048, num_heads=32, head_dim=128, old_lo=0, old_hi=0,
                          pool=16 * 128, dtype="bf16", dist="normal", seed=45, device=DEV)
    ref = {}
    for b in (0, 9):
        for h in (0, 7, 21, 31):
            wb = dict(w)
            wb["q"] = w["q"][:, :, h:h + 1]
            wb["k_new"] = w["k_new"][:, :, h:h + 1]
            wb["v_new"] = w["v_new"][:, :, h:h + 1]
            wb["k_cache"] = w["k_cache"][:, :, h:h + 1]
            wb["v_cache"] = w["v_cache"][:, :, h:h + 1]
            ref[(b, h)] = oracle_kvcache(wb, rows=[b])
    out, lse = run(w)
    for (b, h), (ro, rl) in ref.items():
        assert_close(out[b:b + 1, :, h:h + 1], lse[b:b + 1, h:h + 1], ro, rl, "bf16")


@pytest.mark.parametrize("lnew,d,hq,hkv,causal,dtype", [
    (600, 128, 8, 1, True, "bf16"),   # 5 query tiles: pairs 2 + 0 (tile 5 past the queries), pair 1 alone
    (768, 64, 16, 2, True, "f16"),    # 6 full query tiles
    (1025, 128, 4, 4, False, "f16"),  # 9 query tiles, the last holding one row; all keys visible
])
def test_prefill_query_tile_pairs(lnew, d, hq, hkv, causal, dtype):
    """Query blocks of several 128-row tiles, run two tiles of one head per
    CTA: a unit's heavier and lighter pair, an odd middle pair, a pair whose
    second tile lies past the queries, GQA up to 8 query heads per kv head,
    over cached prefixes of different lengths."""
    w = wl.prefill_append(batch=2, lnew=lnew, num_heads=hq, num_kv_heads=hkv, head_dim=d,
                          old_lo=0, old_hi=600, dtype=dtype, dist="normal", seed=50 + lnew,
                          device=DEV)
    w["causal"] = causal
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run(w)
    assert_close(out, lse, ref_o, ref_l, dtype)


def test_prefill_lengths_beyond_table_report():
    """A sequence whose length exceeds its block table: the call reports
    PA_DEVERR_LENGTH for it and writes O = 0, LSE = -inf for its rows; the
    other sequence is unaffected."""
    w = wl.prefill_append(batch=2, lnew=200, num_heads=4, head_dim=64, old_lo=50, old_hi=300,
                          dtype="f16", dist="normal", seed=47, device=DEV)
    lens = w["cache_seqlens"] + 200  # the new tokens taken as already cached
    w.update(k_new=None, v_new=None, cache_seqlens=lens)
    width = w["block_table"].shape[1]
    w["cache_seqlens"][0] = width * 16 + 1
    err = pa.new_err_word(DEV)
    out, lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                 w["block_table"], scale=w["scale"], causal=True, err=err)
    torch.cuda.synchronize()
    assert err[0].item() == pa.PA_DEVERR_LENGTH and err[1].item() == 0, err.tolist()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ref_o, ref_l = oracle_kvcache(w, rows=[1])
    assert_close(out[1:], lse[1:], ref_o, ref_l, "f16")
