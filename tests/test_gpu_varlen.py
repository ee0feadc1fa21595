"""GPU parity of the unified varlen launch (pa_fwd_varlen_unified): one
launch over chunked-prefill and decode sequences of a paged cache."""

import numpy as np
import pytest
import torch

import paged_kv_cache_page_gb300 as pa
from paged_kv_cache_page_gb300 import workloads as wl

from gpu_util import LSE_TOL, OUT_TOL, np64, oracle_varlen

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(w, workspace=None):
    err = pa.new_err_word(DEV)
    out = torch.full_like(w["q"], float("nan"))
    lse = torch.full((w["q"].shape[1], w["q"].shape[0]), float("nan"), device=DEV)
    pa.pa_fwd_varlen_unified(w["q"], w["k_cache"], w["v_cache"], w["cu_seqlens_q"],
                             w["seqlens_k"], w["block_table"], w["max_seqlen_q"],
                             w["max_seqlen_k"], scale=w["scale"], causal=w["causal"], out=out,
                             lse=lse, err=err, workspace=workspace)
    torch.cuda.synchronize()
    assert err[0].item() == 0, err.tolist()
    return out, lse


def check(w, out, lse, dtype, seqs=None):
    ref = oracle_varlen(w, seqs)
    cu = w["cu_seqlens_q"].cpu().tolist()
    worst = 0.0
    for b, (ro, rl) in ref.items():
        o = np64(out[cu[b]:cu[b + 1]])
        l = np64(lse[:, cu[b]:cu[b + 1]])
        e = np.abs(o - ro).max()
        worst = max(worst, e)
        assert e <= OUT_TOL[dtype], (b, e)
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(l), fin)
        if fin.any():
            assert np.abs(l[fin] - rl[fin]).max() <= LSE_TOL, b
    return worst


@pytest.mark.parametrize("heads,d", [(12, 64), (32, 128), (64, 128)])
def test_unified_mixed_batch(heads, d):
    """Chunked prefills of 100 / 500 / 1000 query tokens over cached prefixes
    U[0, 2048] plus 64 decodes with contexts U[1024, 4096], causal, bf16."""
    w = wl.unified_mixed(num_heads=heads, head_dim=d, device=DEV, seed=1005 + heads)
    out, lse = run(w)
    # every sequence of the batch (the decodes' items are the last the
    # persistent grid deals, and each CTA's run of units ends in them)
    check(w, out, lse, "bf16")


@pytest.mark.parametrize("prefill_lens,num_decode,heads", [
    ((), 96, 32),                      # decode entries only
    ((300, 700, 1200, 64), 0, 16),     # prefill chunks only
    ((100,), 2, 4),                    # far fewer work units than CTAs
])
def test_unified_dealing_extremes(prefill_lens, num_decode, heads):
    """The engine deals a varlen batch's work units to CTAs in contiguous runs
    of equal estimated cost: batches of one kind only, and a batch with far
    fewer units than CTAs (most runs empty), match the oracle."""
    w = wl.unified_mixed(num_heads=heads, head_dim=128, prefill_lens=prefill_lens,
                         num_decode=num_decode, device=DEV, seed=1101 + num_decode + heads)
    out, lse = run(w)
    check(w, out, lse, "bf16")


def test_unified_gqa_and_padding_entries():
    w = wl.unified_mixed(num_heads=16, num_kv_heads=4, head_dim=128, prefill_lens=(7, 40, 300),
                         prefix_hi=700, num_decode=9, ctx_lo=1, ctx_hi=900, pad_to=16,
                         device=DEV, seed=77)
    out, lse = run(w)
    check(w, out, lse, "bf16")
    # padding sequences own no rows: every row of the batch was written
    assert torch.isfinite(out).all()


def test_unified_zero_length_keys_and_single_key():
    w = wl.unified_mixed(num_heads=4, head_dim=64, prefill_lens=(5,), prefix_hi=0,
                         num_decode=3, ctx_lo=1, ctx_hi=1, device=DEV, seed=78)
    w["seqlens_k"][1] = 0  # a decode sequence with no keys at all
    out, lse = run(w)
    cu = w["cu_seqlens_q"].cpu().tolist()
    assert torch.all(out[cu[1]] == 0) and torch.all(torch.isneginf(lse[:, cu[1]]))
    check(w, out, lse, "bf16", seqs=[0, 2, 3])


@pytest.mark.parametrize("fill", [0x01, 0x3F])
def test_unified_stale_workspace_bytes(fill):
    """Every launch rewrites the per-sequence split counts that the combine
    step reads, for every sequence (query-tile prefills and empty padding
    entries included): a workspace still holding other bytes -- here a
    constant byte, i.e. a split count of 0x01010101 or 0x3F3F3F3F and finite
    partials -- changes no output."""
    w = wl.unified_mixed(num_heads=16, num_kv_heads=4, head_dim=128, prefill_lens=(7, 40, 300),
                         prefix_hi=700, num_decode=9, ctx_lo=1, ctx_hi=900, pad_to=16,
                         device=DEV, seed=77)
    total_q, hq, d = w["q"].shape
    B = w["cu_seqlens_q"].numel() - 1
    nbytes = pa.load_library().pa_fwd_varlen_workspace_size(
        B, total_q, w["max_seqlen_q"], hq, w["k_cache"].shape[2], d, w["max_seqlen_k"])
    assert nbytes > 0  # the batch is split: the combine step runs
    ws = torch.full((nbytes,), fill, dtype=torch.uint8, device=DEV)
    out, lse = run(w, workspace=ws)
    check(w, out, lse, "bf16")


def test_unified_batch_beyond_512_entries():
    """A capacity of 600 batch entries (CUDA-graph style padding): 3 chunked
    prefills and 120 decodes followed by 477 empty entries, GQA 32/8 --
    beyond the 512 entries a launch used to be limited to."""
    w = wl.unified_mixed(num_heads=32, num_kv_heads=8, head_dim=128, prefill_lens=(100, 33, 257),
                         prefix_hi=900, num_decode=120, ctx_lo=16, ctx_hi=1500, pad_to=600,
                         device=DEV, seed=601)
    assert w["cu_seqlens_q"].numel() - 1 == 600
    out, lse = run(w)
    cu = w["cu_seqlens_q"].cpu().tolist()
    seqs = [0, 1, 2] + list(range(3, 123, 7)) + [122]
    check(w, out, lse, "bf16", seqs=seqs)
    assert torch.isfinite(out[:cu[-1]]).all()


def permute_sequences(w, order):
    """The same batch with its sequences in another order (rows of q,
    cu_seqlens_q, seqlens_k and block-table rows moved together)."""
    cu = w["cu_seqlens_q"].cpu().tolist()
    idx = torch.tensor(order, dtype=torch.long, device=w["q"].device)
    new_cu = [0]
    for b in order:
        new_cu.append(new_cu[-1] + cu[b + 1] - cu[b])
    w2 = dict(w)
    w2["q"] = torch.cat([w["q"][cu[b]:cu[b + 1]] for b in order])
    w2["cu_seqlens_q"] = torch.tensor(new_cu, dtype=torch.int32, device=w["q"].device)
    w2["seqlens_k"] = w["seqlens_k"][idx]
    w2["block_table"] = w["block_table"][idx]
    return w2


@pytest.mark.parametrize("d,dtype", [(64, "f16"), (128, "bf16"), (128, "f16")])
def test_unified_core_and_tensor_items_interleaved(d, dtype):
    """One-row decode entries, multi-row packed entries (chunks of 2-5
    tokens) and 128-row query tiles, in alternating order: each CTA's
    contiguous run of units switches item kind many times, with the
    pipeline state (stage and buffer parities) running on across them; head
    dim 64 uses the three-stage layout with its own stage-empty barriers."""
    w = wl.unified_mixed(num_heads=16, head_dim=d, prefill_lens=(300, 2, 3, 5, 2, 4, 170, 3),
                         prefix_hi=900, num_decode=40, ctx_lo=1, ctx_hi=2500, dtype=dtype,
                         device=DEV, seed=2024 + d)
    pre = list(range(8))
    dec = list(range(8, 48))
    order = []
    for i in range(40):
        order.append(dec[i])
        if i % 5 == 0 and pre:
            order.append(pre.pop(0))
    order += pre
    w = permute_sequences(w, order)
    out, lse = run(w)
    check(w, out, lse, dtype)


@pytest.mark.parametrize("d", [64, 128])
def test_unified_core_items_split(d):
    """A few long one-row decodes over 4 heads: far fewer (sequence, head)
    streams than CTAs, so the packed items are split over the keys and their
    partials (normalised O and LSE) are merged by the combine step."""
    w = wl.unified_mixed(num_heads=4, head_dim=d, prefill_lens=(3,), prefix_hi=100,
                         num_decode=5, ctx_lo=2000, ctx_hi=4096, device=DEV, seed=3030 + d)
    total_q, hq, _ = w["q"].shape
    B = w["cu_seqlens_q"].numel() - 1
    nbytes = pa.load_library().pa_fwd_varlen_workspace_size(
        B, total_q, w["max_seqlen_q"], hq, w["k_cache"].shape[2], d, w["max_seqlen_k"])
    assert nbytes > 0  # partials exist: the split path runs
    out, lse = run(w)
    check(w, out, lse, "bf16")
