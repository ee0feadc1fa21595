"""GPU parity of the standalone KV append (pa_append_kv): bit-exact against
the oracle's append on integer bit views, paged and contiguous."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("lnew", [1, 15, 16, 17, 170])
def test_paged_append_bit_exact(dtype, lnew):
    w = wl.prefill_append(batch=4, lnew=lnew, num_heads=8, head_dim=128, dtype=dtype,
                          seed=100 + lnew, device=DEV)
    kc0, vc0 = bits(w["k_cache"]), bits(w["v_cache"])
    table = w["block_table"].cpu().numpy()
    seql = w["cache_seqlens"].cpu().numpy()
    ek, ev = oracle.append_kv(kc0, vc0, bits(w["k_new"]), bits(w["v_new"]), seql, table)
    err = pa.new_err_word(DEV)
    pa.pa_append_kv(w["k_cache"], w["v_cache"], w["k_new"], w["v_new"], w["cache_seqlens"],
                    w["block_table"], err=err)
    torch.cuda.synchronize()
    assert err[0].item() == 0
    assert np.array_equal(bits(w["k_cache"]), ek)
    assert np.array_equal(bits(w["v_cache"]), ev)


def test_contiguous_append_bit_exact_and_strided_view():
    g = torch.Generator(device=DEV).manual_seed(3)
    B, cap, hkv, d = 3, 300, 4, 64
    base = torch.randn((B, cap, hkv + 2, d), generator=g, device=DEV).half()
    kc = base[:, :, 1:1 + hkv]  # a strided view: heads 1..4 of 6
    vc = torch.randn((B, cap, hkv, d), generator=g, device=DEV).half()
    kn = torch.randn((B, 7, hkv, d), generator=g, device=DEV).half()
    vn = torch.randn((B, 7, hkv, d), generator=g, device=DEV).half()
    seql = torch.tensor([0, 100, 293], dtype=torch.int32, device=DEV)
    base0, vc0 = bits(base), bits(vc)
    ek, ev = oracle.append_kv(base0[:, :, 1:1 + hkv], vc0, bits(kn), bits(vn), [0, 100, 293])
    pa.pa_append_kv(kc, vc, kn, vn, seql)
    torch.cuda.synchronize()
    got = bits(base)
    assert np.array_equal(got[:, :, 1:1 + hkv], ek)
    assert np.array_equal(got[:, :, 0], base0[:, :, 0]) and np.array_equal(got[:, :, 5], base0[:, :, 5])
    assert np.array_equal(bits(vc), ev)


def test_append_outside_table_is_skipped_and_reported():
    w = wl.prefill_append(batch=2, lnew=20, num_heads=2, head_dim=64, seed=5, device=DEV)
    table = w["block_table"][:, :1].contiguous()  # one page per sequence: too narrow
    kc0 = w["k_cache"].clone()
    err = pa.new_err_word(DEV)
    seql = torch.zeros(2, dtype=torch.int32, device=DEV)
    pa.pa_append_kv(w["k_cache"], w["v_cache"], w["k_new"], w["v_new"], seql, table, err=err)
    torch.cuda.synchronize()
    assert err[0].item() == pa.PA_DEVERR_LENGTH
    # the first 16 tokens of each sequence were written, the rest skipped
    for b in range(2):
        pg = table[b, 0].long()
        assert torch.equal(w["k_cache"][pg], w["k_new"][b, :16])
    changed = (w["k_cache"] != kc0).flatten(1).any(1).nonzero().flatten().tolist()
    assert sorted(changed) == sorted(table[:, 0].tolist())
