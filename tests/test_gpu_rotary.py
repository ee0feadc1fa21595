"""GPU parity of the rotary-embedded kvcache forward (pa_fwd_kvcache_rotary):
the new tokens' q and k rotated at their positions, k stored rotated in the
cache, attention over the rotated keys -- against the oracle's rotation
(rounded once to the dtype) and attention."""

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import LSE_TOL, OUT_TOL, np64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def tables(n_pos, rotary_dim, dtype, base=10000.0):
    p = torch.arange(rotary_dim // 2, dtype=torch.float64)
    theta = base ** (-2.0 * p / rotary_dim)
    ang = torch.arange(n_pos, dtype=torch.float64)[:, None] * theta[None, :]
    return (ang.cos().to(TORCH_DT[dtype]).to(DEV), ang.sin().to(TORCH_DT[dtype]).to(DEV))


def ulps(a, b, dtype):
    """Distance in units in the last place between two arrays of dtype values."""
    ia = torch.from_numpy(a).to(TORCH_DT[dtype]).view(torch.int16).numpy().astype(np.int32)
    ib = torch.from_numpy(b).to(TORCH_DT[dtype]).view(torch.int16).numpy().astype(np.int32)
    # sign-magnitude -> ordered integers
    ia = np.where(ia < 0, -32768 - ia, ia)
    ib = np.where(ib < 0, -32768 - ib, ib)
    return np.abs(ia - ib)


def run_case(w, rotary_dim, interleaved, causal, n_pos=None):
    dtype = w["dtype"]
    lens = w["cache_seqlens"].cpu().tolist()
    lnew = w["k_new"].shape[1]
    n_pos = n_pos or (max(lens) + lnew + 3)
    cos, sin = tables(n_pos, rotary_dim, dtype)
    k_before = w["k_cache"].clone()
    err = pa.new_err_word(DEV)
    out, lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                 w["block_table"], k=w["k_new"], v=w["v_new"], causal=causal,
                                 rotary_cos=cos, rotary_sin=sin, rotary_interleaved=interleaved,
                                 err=err)
    torch.cuda.synchronize()
    assert err[0].item() == 0, err.tolist()
    q_rot, k_rot = oracle.rotate_new_tokens(np64(w["q"]), np64(w["k_new"]), np64(cos), np64(sin),
                                            lens, interleaved, dtype)
    table = w["block_table"]
    for b in range(w["q"].shape[0]):
        old = lens[b]
        npg = -(-(old + lnew) // w["k_cache"].shape[1])
        pages = table[b, :npg].long()
        # the cache now holds the rotated new keys: within one unit in the last
        # place of the oracle's once-rounded rotation
        kc_after = np64(w["k_cache"][pages]).reshape(-1, *w["k_cache"].shape[2:])
        got = kc_after[old:old + lnew]
        assert ulps(got, k_rot[b], dtype).max() <= 1, b
        # attention over the old keys and the rotated new keys
        kc = np64(k_before[pages])
        vc = np64(w["v_cache"][pages])
        o, l = oracle.fwd_kvcache(q_rot[b:b + 1], kc, vc, [old], np.arange(npg)[None],
                                  k_new=k_rot[b:b + 1], v_new=np64(w["v_new"][b:b + 1]),
                                  scale=w["scale"], causal=causal)
        e = np.abs(np64(out[b]) - o[0]).max()
        assert e <= OUT_TOL[dtype], (b, e)
        assert np.abs(np64(lse[b]) - l[0]).max() <= LSE_TOL, b


@pytest.mark.parametrize("dtype,hq,hkv,rotary_dim,interleaved", [
    ("f16", 8, 8, 128, False),    # MHA decode: rotated inside the decode launch
    ("bf16", 16, 4, 64, True),    # GQA decode, partial rotary_dim: tensor-core decode consumer
])
def test_rotary_decode(dtype, hq, hkv, rotary_dim, interleaved):
    w = wl.paged_decode(batch=5, ctx=0, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                        dtype=dtype, lnew=1, seed=900 + hq, device=DEV,
                        lens=[1, 17, 300, 1024, 2049])
    run_case(w, rotary_dim, interleaved, causal=True)


def test_rotary_multi_query_decode():
    w = wl.paged_decode(batch=4, ctx=0, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        dtype="bf16", lnew=6, seed=911, device=DEV, lens=[6, 40, 777, 1500])
    run_case(w, 128, False, causal=True)


def test_rotary_prefill_with_append():
    w = wl.prefill_append(batch=2, lnew=170, num_heads=8, head_dim=128, old_lo=0, old_hi=300,
                          dtype="f16", seed=912, device=DEV)
    run_case(w, 96, True, causal=True)


def test_rotary_position_beyond_table_reports():
    w = wl.paged_decode(batch=2, ctx=0, num_q_heads=4, num_kv_heads=4, head_dim=64, dtype="f16",
                        lnew=1, seed=913, device=DEV, lens=[10, 200])
    cos, sin = tables(50, 64, "f16")  # sequence 1's position 199 is past the table
    err = pa.new_err_word(DEV)
    pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"], w["block_table"],
                      k=w["k_new"], v=w["v_new"], rotary_cos=cos, rotary_sin=sin, err=err)
    torch.cuda.synchronize()
    e = err.tolist()
    assert e[0] == 2 and e[1] == 1 and e[2] == 199, e


@pytest.mark.parametrize("lq,hq,hkv,d,dtype,interleaved", [(2, 32, 8, 128, "bf16", False),
                                                           (4, 16, 4, 64, "f16", True)])
def test_rotary_short_multi_query_decode_in_launch(lq, hq, hkv, d, dtype, interleaved):
    """Up to 16 query rows per kv head: rotated inside the decode launch (q as
    the producer stages it, k where the append stores it), causal among the
    new tokens, ragged lengths that split."""
    w = wl.paged_decode(batch=4, ctx=0, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                        dtype=dtype, lnew=lq, seed=920 + lq, device=DEV,
                        lens=[lq, 45, 1500, 3000])
    run_case(w, d if interleaved else d // 2, interleaved, causal=True)
