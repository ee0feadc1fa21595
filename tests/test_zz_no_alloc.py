"""pa_fwd_kvcache_noalloc: the forward for callers that cannot allocate.

Callers that run inside another library's allocator or stream callback, or in
a serving process whose device memory pool is owned and capped by the
framework, cannot hand the library a workspace.  This entry point uses the
library's own fixed split scratch instead.  The test calls it through the C
ABI (ctypes, raw arguments) on workloads that do split the keys -- the
tensor-core decode consumer on a contiguous cache, 4 and 1 rows per kv head
on paged caches with forced split counts -- twice, with a different workload
run through the same scratch in between (so the second call starts from
another call's leftovers), and checks each result against pa_fwd_kvcache
with a caller workspace, within the parity tolerances of the other GPU
tests.  It also calls the binding's wrapper.  It lives in its own file,
named to be collected last.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import LSE_TOL, OUT_TOL, np64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _raw_noalloc(w, out, lse, err, num_splits):
    lib = pa.load_library()
    q, kc, vc = w["q"], w["k_cache"], w["v_cache"]
    B, lq, hq, d = q.shape
    hkv = kc.shape[2]
    table = w["block_table"]
    if table is not None:
        extent, max_pages, bt_stride = kc.shape[0], table.shape[1], table.stride(0)
        max_k = max_pages * 16
    else:
        extent, max_pages, bt_stride = kc.shape[1], 0, 0
        max_k = extent
    kn, vn = w.get("k_new"), w.get("v_new")
    lnew = 0 if kn is None else kn.shape[1]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    t4 = lambda t: pa.pa_tensor4(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pa_fwd_kvcache_noalloc(
        p(q), q.stride(0), q.stride(1), q.stride(2), t4(kc), t4(vc), p(kn), p(vn), lnew,
        p(w["cache_seqlens"]), p(table), bt_stride, max_pages, 16, B, lq, hq, hkv, d, extent,
        max_k,
        float(w["scale"]), int(bool(w["causal"])), num_splits, p(out), p(lse), p(err),
        pa.PA_BF16 if q.dtype == torch.bfloat16 else pa.PA_F16, stream)


def _contiguous_gqa():
    w = wl.gqa_contiguous(capacity=16384, device=DEV)
    B, hkv, d = 8, w["num_kv_heads"], w["head_dim"]
    kc = torch.zeros((B, w["capacity"], hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    n = w["k_rows"].shape[1]
    kc[:, :n] = w["k_rows"]
    vc[:, :n] = w["v_rows"]
    return dict(w, k_cache=kc, v_cache=vc), "bf16"


def _paged_forced_splits():
    w = wl.paged_decode(5, 0, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        lens=[1000, 37, 700, 16, 1], lnew=1, seed=21, device=DEV)
    return w, "f16"


def _paged_mha_forced_splits():
    # one query row per kv head: the CUDA-core decode consumer
    w = wl.paged_decode(4, 0, num_q_heads=8, num_kv_heads=8, head_dim=64,
                        lens=[513, 2000, 48, 1200], lnew=1, seed=23, device=DEV, dtype="bf16")
    return w, "bf16"


def _interloper():
    """A different workload (other lengths, heads and split count) run through
    the same scratch between the two compared calls, so the second one starts
    from another call's leftovers."""
    w = wl.paged_decode(3, 0, num_q_heads=16, num_kv_heads=4, head_dim=128,
                        lens=[3000, 77, 1500], lnew=1, seed=29, device=DEV)
    out = torch.empty_like(w["q"])
    lse = torch.empty((3, 16, 1), dtype=torch.float32, device=DEV)
    err = pa.new_err_word(DEV)
    assert _raw_noalloc(w, out, lse, err, 5) == pa.PA_OK
    torch.cuda.synchronize()
    assert err[0].item() == 0


@pytest.mark.parametrize("make,num_splits", [(_contiguous_gqa, 0), (_paged_forced_splits, 7),
                                             (_paged_mha_forced_splits, 6)])
def test_noalloc_matches_workspace_entry_point_twice(make, num_splits):
    w, dt = make()
    B, lq, hq, d = w["q"].shape
    hkv = w["k_cache"].shape[2]
    # the case must actually use split scratch
    max_k = (w["block_table"].shape[1] * 16 if w["block_table"] is not None
             else w["k_cache"].shape[1])
    assert pa.fwd_kvcache_workspace_size(B, lq, hq, hkv, d, max_k, num_splits) > 0
    kc0, vc0 = w["k_cache"].clone(), w["v_cache"].clone()
    ref_out, ref_lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"],
                                         w["cache_seqlens"], w["block_table"],
                                         k=w.get("k_new"), v=w.get("v_new"), scale=w["scale"],
                                         causal=w["causal"], num_splits=num_splits)
    torch.cuda.synchronize()
    for call in range(2):
        if call == 1:
            _interloper()
        # the same cache image before every call (the append writes the same
        # bytes again)
        w["k_cache"].copy_(kc0)
        w["v_cache"].copy_(vc0)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = pa.new_err_word(DEV)
        rc = _raw_noalloc(w, out, lse, err, num_splits)
        torch.cuda.synchronize()
        assert rc == pa.PA_OK, pa.load_library().pa_last_error_string()
        assert err[0].item() == 0, err.tolist()
        o_err = float(np.abs(np64(out) - np64(ref_out)).max())
        assert o_err <= OUT_TOL[dt], (call, o_err)
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        l_err = float((lse[fin] - ref_lse[fin]).abs().max())
        assert l_err <= LSE_TOL, (call, l_err)


def test_noalloc_python_wrapper():
    """The binding's wrapper passes the caller's tensors through unchanged and
    refuses a strided k it could only copy by allocating."""
    w, dt = _paged_forced_splits()
    out = torch.empty_like(w["q"])
    lse = torch.empty((w["q"].shape[0], w["q"].shape[2], 1), dtype=torch.float32, device=DEV)
    kc0, vc0 = w["k_cache"].clone(), w["v_cache"].clone()
    ref_out, ref_lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                         w["block_table"], k=w["k_new"], v=w["v_new"],
                                         num_splits=7)
    w["k_cache"].copy_(kc0)
    w["v_cache"].copy_(vc0)
    pa.pa_fwd_kvcache_noalloc(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"], out,
                              block_table=w["block_table"], k=w["k_new"], v=w["v_new"], lse=lse,
                              num_splits=7)
    torch.cuda.synchronize()
    assert float(np.abs(np64(out) - np64(ref_out)).max()) <= OUT_TOL[dt]
    assert float((lse - ref_lse).abs().max()) <= LSE_TOL
    strided = torch.empty((w["k_new"].shape[0], w["k_new"].shape[1], w["k_new"].shape[2],
                           2 * w["k_new"].shape[3]), dtype=w["k_new"].dtype, device=DEV)
    k_view = strided[..., :w["k_new"].shape[3]]
    assert not k_view.is_contiguous()
    with pytest.raises(ValueError):
        pa.pa_fwd_kvcache_noalloc(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"], out,
                                  block_table=w["block_table"], k=k_view, v=w["v_new"], lse=lse)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = pa.load_library()
    # 256 sequences x 64 q heads at D 128 with 128 forced splits need about
    # 1 GB of split scratch, far beyond the fixed array: rejected with a clear
    # error before any work is queued.  Every pointer is NULL, so that even if
    # the size check came later the call would stop at argument validation.
    need = lib.pa_fwd_kvcache_workspace_size(256, 1, 64, 8, 128, 131072, 128)
    assert need > pa.PA_NOALLOC_SCRATCH_BYTES
    t4 = pa.pa_tensor4(None, 1 << 20, 1024, 128)
    rc = lib.pa_fwd_kvcache_noalloc(None, 64 * 128, 64 * 128, 128, t4, t4, None, None, 0, None,
                                    None, 8192, 8192, 16, 256, 1, 64, 8, 128, 1 << 16, 131072,
                                    1.0 / math.sqrt(128), 0, 128, None, None, None, pa.PA_F16,
                                    None)
    assert rc == pa.PA_ERR_WORKSPACE
    assert "scratch" in lib.pa_last_error_string().decode()
