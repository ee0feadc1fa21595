"""Encoding self-test of the tcgen05 operand layouts the prefill kernel uses
(one CTA, one 128x128 tile) against a plain PyTorch fp32 matmul:
C1 = A B1^T with both operands K-major and 128-byte swizzled (A written by
threads like the P tile, B1 fetched by TMA like a K tile), C2 = A B2 with
B2 an MN-major operand (like a V tile), and C3 = A B2 with A read from tensor
memory (like the P tile)."""

import ctypes

import pytest
import torch

import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import build as pabuild

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("a_col", [384, 448])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
def test_tcgen05_operand_layouts(dtype, d, a_col):
    pabuild.build()
    lib = ctypes.CDLL(pabuild.lib_path(pabuild.SELFTEST_LIB))
    g = torch.Generator(device=DEV).manual_seed(d)
    A = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    B1 = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    B2 = torch.randn((128, d), generator=g, device=DEV).to(dtype)
    C1 = torch.full((128, 128), float("nan"), device=DEV)
    C2 = torch.full((128, d), float("nan"), device=DEV)
    C3 = torch.full((128, d), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.pa_selftest_tcgen05_gemm(p(A), p(B1), p(B2), p(C1), p(C2), p(C3), d,
                                      pa.PA_BF16 if dtype == torch.bfloat16 else pa.PA_F16,
                                      p(status), a_col,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and status.item() == 0
    ref1 = A.float() @ B1.float().T
    ref2 = A.float() @ B2.float()
    torch.testing.assert_close(C1, ref1, rtol=1e-4, atol=1e-3)
    torch.testing.assert_close(C2, ref2, rtol=1e-4, atol=1e-3)
    torch.testing.assert_close(C3, ref2, rtol=1e-4, atol=1e-3)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_tcgen05_transposed_decode_shapes(dtype):
    """The transposed decode-tile shapes: C4 = K Q^T with N = 16 query rows
    (both operands K-major, fetched by TMA) and C5 = V^T P^T with the V tile
    read as an MN-major A operand and a 16-row P tile written by threads."""
    pabuild.build()
    lib = ctypes.CDLL(pabuild.lib_path(pabuild.SELFTEST_LIB))
    g = torch.Generator(device=DEV).manual_seed(7)
    K = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    Q = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    V = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    P = torch.randn((16, 128), generator=g, device=DEV).to(dtype)
    C4 = torch.full((128, 16), float("nan"), device=DEV)
    C5 = torch.full((128, 16), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.pa_selftest_tcgen05_transposed(p(K), p(Q), p(V), p(P), p(C4), p(C5),
                                            pa.PA_BF16 if dtype == torch.bfloat16 else pa.PA_F16,
                                            p(status),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and status.item() == 0
    torch.testing.assert_close(C4, K.float() @ Q[:16].float().T, rtol=1e-4, atol=1e-3)
    torch.testing.assert_close(C5, V.float().T @ P.float().T, rtol=1e-4, atol=1e-3)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_tcgen05_cp_places_an_a_operand_in_tmem(dtype):
    """tcgen05.cp of the 128-byte-swizzled Q tile (eight 128x256b blocks, one
    per k-step) into TMEM gives the A operand the TMEM-A MMA reads: Q K^T with
    Q from TMEM equals Q K^T with Q from shared memory and the reference."""
    pabuild.build()
    lib = ctypes.CDLL(pabuild.lib_path(pabuild.SELFTEST_LIB))
    g = torch.Generator(device=DEV).manual_seed(11)
    Q = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    K = torch.randn((128, 128), generator=g, device=DEV).to(dtype)
    C1 = torch.full((128, 128), float("nan"), device=DEV)
    C2 = torch.full((128, 128), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.pa_selftest_tcgen05_cpq(p(Q), p(K), p(C1), p(C2),
                                     pa.PA_BF16 if dtype == torch.bfloat16 else pa.PA_F16,
                                     p(status),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and status.item() == 0
    ref = Q.float() @ K.float().T
    torch.testing.assert_close(C1, ref, rtol=1e-4, atol=1e-3)
    torch.testing.assert_close(C2, ref, rtol=1e-4, atol=1e-3)
