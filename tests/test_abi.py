"""The C-ABI library loads and exports what include/pagedattn.h declares (CPU).

Only host-side paths run here: symbol lookup, workspace sizing and argument
validation that rejects a call before any CUDA API is touched.
"""

import ctypes
import os
import re

import pytest

import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import build as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    pabuild.build()
    return pa.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    for n in ["pa_append_kv", "pa_fwd_kvcache", "pa_fwd_varlen_unified", "pa_split_combine",
              "pa_fwd_kvcache_workspace_size", "pa_fwd_varlen_workspace_size",
              "pa_last_error_string", "pa_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(pabuild.lib_path())
    for name in declared_symbols():
        assert hasattr(raw, name), name
    assert lib.pa_version() >= 100


def test_binding_signatures_cover_header(lib):
    assert set(declared_symbols()) == set(pa._SIGNATURES)


def declared_prototypes():
    """name -> list of parameter declarations, from the header's PA_API
    prototypes (comments removed)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    out = {}
    for m in re.finditer(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [x.strip() for x in m.group(2).split(",") if x.strip()]
        out[m.group(1)] = [] if params == ["void"] else params
    return out


def test_binding_argument_counts_and_kinds_match_header(lib):
    """Every binding signature has the header's parameter count, with each
    pointer / 64-bit / 32-bit / float / struct parameter marshalled as one."""
    protos = declared_prototypes()
    assert set(protos) == set(pa._SIGNATURES)
    for name, params in protos.items():
        argtypes = pa._SIGNATURES[name][1]
        assert len(argtypes) == len(params), (name, len(argtypes), len(params))
        for decl, at in zip(params, argtypes):
            if "*" in decl or decl.startswith("pa_stream_t"):
                assert at in (ctypes.c_void_p, ctypes.c_char_p), (name, decl, at)
            elif decl.startswith("pa_tensor4"):
                assert at is pa.pa_tensor4, (name, decl, at)
            elif decl.split()[0] in ("int64_t", "size_t"):
                assert ctypes.sizeof(at) == 8, (name, decl, at)
            elif decl.split()[0] == "float":
                assert at is ctypes.c_float, (name, decl, at)
            else:
                assert decl.split()[0] in ("int", "int32_t") and ctypes.sizeof(at) == 4, (name, decl, at)


def _t4(stride_b=16 * 2 * 64, stride_t=2 * 64, stride_h=64, ptr=4096):
    return pa.pa_tensor4(ptr, stride_b, stride_t, stride_h)


def _kvcache_call(lib, **kw):
    args = dict(q=4096, q_sb=256, q_st=256, q_sh=64, k=_t4(), v=_t4(), k_new=None, v_new=None,
                lnew=0, seqlens=4096, table=4096, bt_stride=4, max_pages=4, page_size=16, B=2,
                Lq=1, Hq=4,
                Hkv=2, D=64, extent=8, max_k=64, scale=0.125, causal=0, splits=0, out=4096,
                lse=None, ws=None, ws_bytes=0, err=None, dtype=pa.PA_F16)
    args.update(kw)
    a = args
    return lib.pa_fwd_kvcache(a["q"], a["q_sb"], a["q_st"], a["q_sh"], a["k"], a["v"],
                              a["k_new"], a["v_new"], a["lnew"], a["seqlens"], a["table"],
                              a["bt_stride"], a["max_pages"], a["page_size"], a["B"], a["Lq"],
                              a["Hq"], a["Hkv"],
                              a["D"], a["extent"], a["max_k"], a["scale"], a["causal"],
                              a["splits"], a["out"], a["lse"], a["ws"], a["ws_bytes"], a["err"],
                              a["dtype"], None)


def test_validation_rejects_before_any_cuda_call(lib):
    assert _kvcache_call(lib, dtype=7) == pa.PA_ERR_UNSUPPORTED
    assert _kvcache_call(lib, D=96) == pa.PA_ERR_UNSUPPORTED
    assert _kvcache_call(lib, Hq=3, Hkv=2) == pa.PA_ERR_UNSUPPORTED
    assert _kvcache_call(lib, B=-1) == pa.PA_ERR_INVALID_ARG
    assert _kvcache_call(lib, k=_t4(ptr=0)) == pa.PA_ERR_INVALID_ARG
    assert _kvcache_call(lib, k=_t4(ptr=4100)) == pa.PA_ERR_INVALID_ARG      # misaligned
    assert _kvcache_call(lib, v=_t4(stride_h=60)) == pa.PA_ERR_INVALID_ARG   # TMA stride rule
    assert _kvcache_call(lib, seqlens=None) == pa.PA_ERR_INVALID_ARG
    assert _kvcache_call(lib, lnew=3) == pa.PA_ERR_INVALID_ARG               # Lnew without k/v
    assert _kvcache_call(lib, max_pages=0) == pa.PA_ERR_INVALID_ARG
    assert _kvcache_call(lib, bt_stride=2) == pa.PA_ERR_INVALID_ARG
    assert _kvcache_call(lib, scale=float("nan")) == pa.PA_ERR_INVALID_ARG
    for bad_page in (0, 8, 24, 48, 512):  # 16 << s, s in [0, 4], only
        assert _kvcache_call(lib, page_size=bad_page) == pa.PA_ERR_UNSUPPORTED
    assert _kvcache_call(lib, q_sh=7) == pa.PA_ERR_INVALID_ARG
    # a split plan that needs workspace but gets none
    assert _kvcache_call(lib, max_k=4096, table=4096, max_pages=256, bt_stride=256,
                         splits=4) == pa.PA_ERR_WORKSPACE
    assert "workspace" in lib.pa_last_error_string().decode()
    # empty batch: nothing to do, OK without touching the GPU
    assert _kvcache_call(lib, B=0) == pa.PA_OK


def test_workspace_sizes(lib):
    # many independent (sequence, kv head) pairs: no split, no workspace
    assert lib.pa_fwd_kvcache_workspace_size(256, 1, 32, 32, 128, 4096, 0) == 0
    # a forced single split needs none either
    assert lib.pa_fwd_kvcache_workspace_size(8, 1, 32, 8, 128, 131072, 1) == 0
    # few long sequences: split partials (fp32 O + LSE) and split counts
    n = lib.pa_fwd_kvcache_workspace_size(8, 1, 32, 8, 128, 131072, 0)
    assert n >= 8 * 32 * 129 * 4 * 2
    # forced splits bound the partial buffers exactly
    n4 = lib.pa_fwd_kvcache_workspace_size(2, 1, 4, 2, 64, 1024, 4)
    assert n4 >= 4 * 2 * 4 * 65 * 4
    # the tensor-core prefill path takes no workspace
    assert lib.pa_fwd_kvcache_workspace_size(4, 170, 32, 32, 128, 1024, 0) == 0


def test_split_cap_respects_schedule_table(lib):
    # more sequences than the device schedule's prefix table: never split,
    # even when splits are requested
    assert lib.pa_fwd_kvcache_workspace_size(513, 1, 8, 8, 128, 4096, 4) == 0
    assert lib.pa_fwd_kvcache_workspace_size(512, 1, 8, 8, 128, 4096, 4) > 0
