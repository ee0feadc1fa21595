"""The seeded synthetic inputs against the recipes they stand for: shapes,
length ranges, block tables of distinct pages covering exactly the pages a
sequence needs, value distributions, padding entries, and determinism per
seed (CPU only, small sizes)."""

import math

import torch

from paged_kv_cache_page_gb300 import workloads as wl


def _rows_distinct_and_sized(table, pages, pool):
    used = []
    for b, n in enumerate(pages):
        row = table[b, :n].tolist()
        assert all(0 <= p < pool for p in row)
        assert all(p == pool for p in table[b, n:].tolist())  # padding sentinel, never read
        used += row
    assert len(used) == len(set(used))  # no physical page shared between sequences
    return used


def test_tiny_decode_recipe():
    w = wl.tiny_decode()
    assert w["q"].shape == (2, 1, 4, 64) and w["k_cache"].shape == (64, 16, 2, 64)
    assert w["cache_seqlens"].tolist() == [37, 100] and w["scale"] == 1.0 / 8.0
    # one permutation of the 64 pages split into two rows
    assert sorted(w["block_table"].flatten().tolist()) == list(range(64))


def test_paged_decode_recipe():
    w = wl.paged_decode(4, 100, num_q_heads=8, num_kv_heads=2, head_dim=64, lnew=1, seed=3)
    pages = [math.ceil(100 / 16)] * 4
    assert w["num_pages"] == sum(pages)  # pool = exactly the pages needed
    used = _rows_distinct_and_sized(w["block_table"], pages, w["num_pages"])
    assert sorted(used) == list(range(w["num_pages"]))  # a permutation of the pool
    assert w["cache_seqlens"].tolist() == [99] * 4  # ctx - lnew old tokens, lnew appended
    assert w["k_new"].shape == (4, 1, 2, 64) and w["q"].shape == (4, 1, 8, 64)
    x = w["k_cache"].float()
    assert abs(x.mean().item()) < 0.05 and abs(x.std().item() - 1) < 0.05  # N(0, 1)


def test_gqa_contiguous_recipe():
    w = wl.gqa_contiguous(capacity=8192)
    lens = w["cache_seqlens"].tolist()
    assert len(lens) == 8 and all(1024 <= n <= 8192 for n in lens)
    assert w["k_rows"].shape == (8, max(lens), 8, 128) and w["q"].shape == (8, 1, 32, 128)
    assert w["k_rows"].dtype == torch.bfloat16 and w["block_table"] is None


def test_prefill_append_recipe():
    w = wl.prefill_append(seed=1004)
    old = w["cache_seqlens"].tolist()
    assert len(old) == 4 and all(0 <= n <= 512 for n in old)
    pages = [math.ceil((n + 170) / 16) for n in old]
    _rows_distinct_and_sized(w["block_table"], pages, w["k_cache"].shape[0])
    assert w["k_cache"].shape[0] == 1000  # the reproduction's 1000-page pool
    x = w["q"].float()
    # U[0, 1) as in the reproduction, drawn in fp32 and rounded to fp16 (which
    # may round a draw just below 1 up to 1)
    assert x.min().item() >= 0 and x.max().item() <= 1 and abs(x.mean().item() - 0.5) < 0.01
    assert w["q"].shape == (4, 170, 32, 128) and w["k_new"].shape == (4, 170, 32, 128)


def test_unified_mixed_recipe_and_padding():
    w = wl.unified_mixed(num_heads=4, head_dim=64, prefill_lens=(100, 500, 1000), num_decode=6,
                         pad_to=12, seed=1005)
    cu = w["cu_seqlens_q"].tolist()
    kl = w["seqlens_k"].tolist()
    ql = [cu[i + 1] - cu[i] for i in range(len(kl))]
    assert ql == [100, 500, 1000] + [1] * 6 + [0] * 3  # padding entries repeat cu_seqlens_q
    assert all(l <= k <= l + 2048 for l, k in zip(ql[:3], kl[:3]))  # prefix ~ U[0, 2048]
    assert all(1024 <= k <= 4096 for k in kl[3:9]) and kl[9:] == [0, 0, 0]
    pages = [math.ceil(k / 16) for k in kl]
    _rows_distinct_and_sized(w["block_table"], pages, w["num_pages"])
    assert w["max_seqlen_q"] == 1000 and w["max_seqlen_k"] == max(kl) and w["causal"]


def test_draws_are_deterministic_per_seed():
    a = wl.paged_decode(2, 40, num_q_heads=2, num_kv_heads=2, head_dim=64, seed=7)
    b = wl.paged_decode(2, 40, num_q_heads=2, num_kv_heads=2, head_dim=64, seed=7)
    c = wl.paged_decode(2, 40, num_q_heads=2, num_kv_heads=2, head_dim=64, seed=8)
    for k in ("q", "k_cache", "v_cache", "block_table"):
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["q"], c["q"])
