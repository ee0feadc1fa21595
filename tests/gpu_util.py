"""Shared helpers for the GPU parity tests: oracle calls on torch inputs and
the tolerances the CUDA path must meet.

Tolerances (max abs error against the float64 oracle): output 2e-3 for fp16
and 1.6e-2 for bf16, LSE 1e-3; append and block-table indexing bit-exact.
"""

import numpy as np
import torch

import oracle

OUT_TOL = {"f16": 2e-3, "bf16": 1.6e-2}
LSE_TOL = 1e-3


def np64(t):
    return None if t is None else t.detach().cpu().double().numpy()


def bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


def oracle_kvcache(w, causal=None, rows=None):
    """Oracle forward for a kvcache workload dict (optionally only `rows`,
    a list of sequence indices, gathering just the pages those use)."""
    causal = w["causal"] if causal is None else causal
    table = w["block_table"]
    seqs = range(w["q"].shape[0]) if rows is None else rows
    outs, lses = [], []
    lnew = 0 if w.get("k_new") is None else w["k_new"].shape[1]
    for b in seqs:
        old = int(w["cache_seqlens"][b])
        lk = old + lnew
        if table is not None:
            npg = -(-old // w["k_cache"].shape[1])
            pages = table[b, :npg].long()
            kc = np64(w["k_cache"][pages])
            vc = np64(w["v_cache"][pages])
            tb = np.arange(npg)[None]
        else:
            kc = np64(w["k_cache"][b:b + 1, :old])
            vc = np64(w["v_cache"][b:b + 1, :old])
            tb = None
        kn = None if lnew == 0 else np64(w["k_new"][b:b + 1])
        vn = None if lnew == 0 else np64(w["v_new"][b:b + 1])
        o, l = oracle.fwd_kvcache(np64(w["q"][b:b + 1]), kc, vc, [old], tb, k_new=kn, v_new=vn,
                                  scale=w["scale"], causal=causal)
        outs.append(o[0])
        lses.append(l[0])
        del lk
    return np.stack(outs), np.stack(lses)


def assert_close(out, lse, ref_out, ref_lse, dtype, rows=None):
    o = np64(out) if rows is None else np64(out[rows])
    err = np.abs(o - ref_out).max() if o.size else 0.0
    assert err <= OUT_TOL[dtype], f"max |O - oracle| = {err:.3e} > {OUT_TOL[dtype]}"
    if lse is not None:
        l = np64(lse) if rows is None else np64(lse[rows])
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(l), fin), "LSE -inf pattern differs"
        if fin.any():
            lerr = np.abs(l[fin] - ref_lse[fin]).max()
            assert lerr <= LSE_TOL, f"max |LSE - oracle| = {lerr:.3e}"
    return err


def oracle_varlen(w, seqs=None):
    """Oracle for a varlen workload dict, one sequence at a time (only the
    pages each sequence uses are copied to the host).  Returns
    {b: (O [qlen, Hq, D], LSE [Hq, qlen])}."""
    cu = w["cu_seqlens_q"].cpu().tolist()
    lens = w["seqlens_k"].cpu().tolist()
    table = w["block_table"]
    res = {}
    for b in (range(len(lens)) if seqs is None else seqs):
        q0, q1 = cu[b], cu[b + 1]
        if q1 == q0:
            continue
        npg = -(-lens[b] // w["k_cache"].shape[1])
        pages = table[b, :npg].long()
        kc = np64(w["k_cache"][pages])
        vc = np64(w["v_cache"][pages])
        o, l = oracle.fwd_varlen(np64(w["q"][q0:q1]), kc, vc, [0, q1 - q0], [lens[b]],
                                 np.arange(max(npg, 1))[None], scale=w["scale"],
                                 causal=w["causal"])
        res[b] = (o, l)
    return res
