"""Failure detection without a GPU fault: a pipeline wait on a barrier that
no thread arrives at gives up after its time limit, the kernel reports
PA_DEVERR_TIMEOUT in the error word and returns, and the context still runs
attention correctly afterwards."""

import ctypes

import pytest
import torch

import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import build as pabuild
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import assert_close, oracle_kvcache

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_bounded_wait_times_out_reports_and_leaves_the_context_usable():
    pabuild.build()
    lib = ctypes.CDLL(pabuild.lib_path(pabuild.SELFTEST_LIB))
    err = pa.new_err_word(DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    stream = torch.cuda.current_stream(DEV)
    rc = lib.pa_selftest_wait_timeout(ctypes.c_void_p(err.data_ptr()),
                                      ctypes.c_void_p(elapsed.data_ptr()),
                                      ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert err[0].item() == pa.PA_DEVERR_TIMEOUT and err[2].item() == 99, err.tolist()
    assert 1.5e9 < elapsed.item() < 20e9  # the 2 s limit, measured on the device clock
    w = wl.paged_decode(3, 300, num_q_heads=8, num_kv_heads=8, head_dim=128, lnew=1, seed=60,
                        device=DEV)
    ref_o, ref_l = oracle_kvcache(w)
    err2 = pa.new_err_word(DEV)
    out, lse = pa.pa_fwd_kvcache(w["q"], w["k_cache"], w["v_cache"], w["cache_seqlens"],
                                 w["block_table"], k=w["k_new"], v=w["v_new"], err=err2)
    torch.cuda.synchronize()
    assert err2[0].item() == 0
    assert_close(out, lse, ref_o, ref_l, "f16")
