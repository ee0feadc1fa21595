"""GPU parity at page sizes other than 16: the block size 16 vs 256 of vLLM
#3010 "Introduce flash-attn" (flash-attention then required pages divisible
by 256).  The kernels move 16-token boxes; a page of P tokens holds P / 16 of
them.  Every path -- fused decode append, standalone append, GQA split-KV
engine items, prefill tiles, the unified launch -- against the oracle (which
reads the page size from the cache's second dimension)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import assert_close, bits, oracle_kvcache
from test_gpu_varlen import check, run as run_varlen

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_kvcache(w, **kw):
    err = pa.new_err_word(DEV)
    out, lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                 w["block_table"], k=w.get("k_new"), v=w.get("v_new"),
                                 causal=w["causal"], err=err, **kw)
    torch.cuda.synchronize()
    assert err[0].item() == 0, err.tolist()
    return out, lse


@pytest.mark.parametrize("page", [32, 64, 256])
def test_mha_decode_with_fused_append(page):
    w = wl.paged_decode(batch=6, ctx=0, num_q_heads=8, num_kv_heads=8, head_dim=128, dtype="f16",
                        lnew=1, seed=700 + page, device=DEV, lens=[1, 16, 17, 255, 257, 3000],
                        page_size=page)
    kc0, vc0 = bits(w["k_cache"]), bits(w["v_cache"])
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run_kvcache(w)
    assert_close(out, lse, ref_o, ref_l, "f16")
    # the new token landed in its slot of its P-token page, bit for bit
    ek, ev = oracle.append_kv(kc0, vc0, bits(w["k_new"]), bits(w["v_new"]),
                              w["cache_seqlens"].cpu().numpy(), w["block_table"].cpu().numpy())
    assert np.array_equal(bits(w["k_cache"]), ek) and np.array_equal(bits(w["v_cache"]), ev)


@pytest.mark.parametrize("page", [128, 256])
def test_gqa_split_decode(page):
    w = wl.paged_decode(batch=5, ctx=0, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        dtype="bf16", lnew=1, seed=710 + page, device=DEV,
                        lens=[3, 600, 2048, 4096, 5000], page_size=page)
    ref_o, ref_l = oracle_kvcache(w)
    for splits in (0, 3):
        out, lse = run_kvcache(w, num_splits=splits)
        assert_close(out, lse, ref_o, ref_l, "bf16")


@pytest.mark.parametrize("page", [64, 256])
def test_causal_prefill_with_append(page):
    w = wl.prefill_append(batch=3, lnew=300, num_heads=8, head_dim=128, old_lo=0, old_hi=700,
                          dtype="f16", seed=720 + page, device=DEV, page_size=page)
    ref_o, ref_l = oracle_kvcache(w)
    out, lse = run_kvcache(w)
    assert_close(out, lse, ref_o, ref_l, "f16")


@pytest.mark.parametrize("page", [32, 256])
def test_unified_mixed_batch(page):
    w = wl.unified_mixed(num_heads=16, num_kv_heads=4, head_dim=128, prefill_lens=(7, 300),
                         prefix_hi=900, num_decode=6, ctx_lo=1, ctx_hi=1500, pad_to=10,
                         device=DEV, seed=730 + page, page_size=page)
    out, lse = run_varlen(w)
    check(w, out, lse, "bf16")


@pytest.mark.parametrize("lnew", [1, 17, 300])
def test_standalone_append_bit_exact(lnew):
    w = wl.prefill_append(batch=4, lnew=lnew, num_heads=4, head_dim=64, dtype="bf16",
                          seed=740 + lnew, device=DEV, page_size=256)
    kc0, vc0 = bits(w["k_cache"]), bits(w["v_cache"])
    ek, ev = oracle.append_kv(kc0, vc0, bits(w["k_new"]), bits(w["v_new"]),
                              w["cache_seqlens"].cpu().numpy(), w["block_table"].cpu().numpy())
    err = pa.new_err_word(DEV)
    pa.pa_append_kv(w["k_cache"], w["v_cache"], w["k_new"], w["v_new"], w["cache_seqlens"],
                    w["block_table"], err=err)
    torch.cuda.synchronize()
    assert err[0].item() == 0
    assert np.array_equal(bits(w["k_cache"]), ek) and np.array_equal(bits(w["v_cache"]), ev)


@pytest.mark.parametrize("page", [64, 256])
@pytest.mark.parametrize("d,hq,hkv,lq,dtype", [(64, 32, 4, 1, "f16"), (128, 16, 1, 1, "bf16"),
                                               (64, 16, 4, 2, "bf16")])
def test_tensor_core_decode_consumer(page, d, hq, hkv, lq, dtype):
    """The decode kernel's warp-level tensor-core consumer (8 and 16 query rows
    per kv head; 64-column 128-byte-swizzled boxes) at pages of 64 and 256
    tokens: head dims 64 and 128, a causal two-token append, automatic and
    forced splits."""
    w = wl.paged_decode(batch=5, ctx=0, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                        dtype=dtype, lnew=lq, seed=950 + page + d + hq + lq, device=DEV,
                        lens=[lq + 1, 300, 1000, 2500, 4100], page_size=page)
    w["causal"] = lq > 1
    ref_o, ref_l = oracle_kvcache(w)
    for splits in (0, 4):
        out, lse = run_kvcache(w, num_splits=splits)
        assert_close(out, lse, ref_o, ref_l, dtype)


def test_rotary_in_decode_launch_large_pages():
    """Rotary embedding inside the decode launch (q staged rotated, k rotated
    where the fused append stores it) with 256-token pages."""
    from test_gpu_rotary import run_case
    w = wl.paged_decode(batch=4, ctx=0, num_q_heads=16, num_kv_heads=4, head_dim=128,
                        dtype="bf16", lnew=2, seed=960, device=DEV, lens=[2, 45, 1500, 3000],
                        page_size=256)
    run_case(w, 64, False, causal=True)
