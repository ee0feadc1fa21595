"""Pins of the CPU oracle against things other than itself (CPU only).

* golden worked examples derived by hand (``tests/golden/*.json``);
* torch's CPU ``scaled_dot_product_attention`` (an independent library
  routine) on contiguous inputs, including its own GQA expansion;
* a scalar pure-Python brute force that walks the block table page by page;
* closed forms (identical keys -> mean of V; a single key -> that value);
* invariants (page permutation, split + combine, causal prefix == stepwise
  decode, varlen == kvcache, inert padding sequences);
* planted mistakes: each plausible bug planted in the oracle makes one of the
  pins above fail.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _check_golden(name):
    g = _load(name)
    q = np.array(g["q"], dtype=np.float64)
    k = np.array(g["k"], dtype=np.float64)
    v = np.array(g["v"], dtype=np.float64)
    out, lse = oracle.attend_rows(q, k, v, g["scale"], g["causal"])
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(g["expected_lse"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", ["two_keys_softmax.json", "causal_bottom_right.json",
                                  "gqa_mapping.json"])
def test_golden_attention(name):
    _check_golden(name)


def _check_append_golden():
    g = _load("append_pages.json")
    pool = g["num_pages"]
    cache = np.zeros((pool, 16, 1, 1), dtype=np.uint16)
    for p in range(pool):
        for s in range(16):
            cache[p, s, 0, 0] = 100 * p + s
    k_new = np.array(g["k_new"], dtype=np.uint16).reshape(1, -1, 1, 1)
    kc, vc = oracle.append_kv(cache, cache, k_new, k_new, g["cache_seqlens"],
                              np.array(g["block_table"]))
    expect = cache.copy()
    for p, s, val in g["written"]:
        expect[p, s, 0, 0] = val
    assert np.array_equal(kc, expect)
    assert np.array_equal(vc, expect)


def test_golden_append():
    _check_append_golden()


def _paged_gather_closed_form():
    """Causal self-attention with equal scores over a permuted 2-page table.

    Pool of 3 pages, D = 1, value at (page p, slot s) = 100 p + s, table
    [2, 0], Lq = Lk = 20, q = 0.  Row i averages logical keys 0..i:
    i < 16 -> 200 + i/2; i >= 16 -> (sum_{t<16}(200+t) + sum_{u<=i-16} u)/(i+1).
    """
    cache = np.zeros((3, 16, 1, 1))
    for p in range(3):
        for s in range(16):
            cache[p, s, 0, 0] = 100 * p + s
    table = np.array([[2, 0]])
    q = np.zeros((1, 20, 1, 1))
    out, _ = oracle.fwd_kvcache(q, cache, cache, [20], table, scale=1.0, causal=True)
    for i in range(20):
        if i < 16:
            want = 200 + i / 2
        else:
            want = (3200 + 120 + (i - 16) * (i - 15) / 2) / (i + 1)
        assert abs(out[0, i, 0, 0] - want) < 1e-9, (i, out[0, i, 0, 0], want)


def test_paged_gather_closed_form():
    _paged_gather_closed_form()


def _rand_case(rng, lq, lk, hq, hkv, d):
    q = rng.standard_normal((lq, hq, d))
    k = rng.standard_normal((lk, hkv, d))
    v = rng.standard_normal((lk, hkv, d))
    return q, k, v


def _check_torch_sdpa(seed=0):
    rng = np.random.default_rng(seed)
    for (lq, lk, hq, hkv, d, causal) in [(1, 37, 4, 2, 64, False), (5, 40, 4, 4, 16, True),
                                         (7, 7, 6, 2, 8, True), (3, 50, 8, 1, 32, False),
                                         (4, 19, 2, 2, 8, True)]:
        q, k, v = _rand_case(rng, lq, lk, hq, hkv, d)
        scale = 1.0 / math.sqrt(d)
        out, _ = oracle.attend_rows(q, k, v, scale, causal)
        tq = torch.from_numpy(q).permute(1, 0, 2)[None]  # [1, Hq, Lq, D]
        tk = torch.from_numpy(k).permute(1, 0, 2)[None]
        tv = torch.from_numpy(v).permute(1, 0, 2)[None]
        mask = None
        if causal:
            i = torch.arange(lq)[:, None]
            t = torch.arange(lk)[None, :]
            mask = t <= i + (lk - lq)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=mask, scale=scale, enable_gqa=(hq != hkv))
        ref = ref[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_matches_torch_sdpa():
    _check_torch_sdpa()


def _brute_force_paged(q, k_cache, v_cache, cache_seqlens, table, scale, causal):
    """Scalar loops with math.exp: walk the table page by page."""
    bsz, lq, hq, d = q.shape
    hkv = k_cache.shape[2]
    out = np.zeros_like(q, dtype=np.float64)
    lse = np.zeros((bsz, hq, lq))
    for b in range(bsz):
        lk = int(cache_seqlens[b])
        keys, vals = [], []
        page_idx = 0
        while len(keys) < lk:
            phys = int(table[b][page_idx])
            for slot in range(16):
                if len(keys) == lk:
                    break
                keys.append(k_cache[phys, slot])
                vals.append(v_cache[phys, slot])
            page_idx += 1
        for h in range(hq):
            g = (h * hkv) // hq
            for i in range(lq):
                last = i + lk - lq if causal else lk - 1
                scores = []
                for t in range(0, last + 1):
                    acc = 0.0
                    for x in range(d):
                        acc += float(q[b, i, h, x]) * float(keys[t][g][x])
                    scores.append(acc * scale)
                mx = max(scores)
                den = sum(math.exp(s - mx) for s in scores)
                for x in range(d):
                    num = sum(math.exp(s - mx) * float(vals[t][g][x]) for t, s in enumerate(scores))
                    out[b, i, h, x] = num / den
                lse[b, h, i] = mx + math.log(den)
    return out, lse


def _check_brute_force(seed=1):
    rng = np.random.default_rng(seed)
    for trial in range(4):
        bsz = int(rng.integers(1, 4))
        lq = int(rng.integers(1, 6))
        hkv = int(rng.integers(1, 3))
        hq = hkv * int(rng.integers(1, 3))
        d = int(rng.choice([4, 8]))
        lens = [int(rng.integers(lq, 41)) for _ in range(bsz)]
        pages = [-(-l // 16) for l in lens]
        pool = sum(pages) + 2
        perm = rng.permutation(pool)
        table = np.full((bsz, max(pages)), -1)
        off = 0
        for b in range(bsz):
            table[b, :pages[b]] = perm[off:off + pages[b]]
            off += pages[b]
        kc = rng.standard_normal((pool, 16, hkv, d))
        vc = rng.standard_normal((pool, 16, hkv, d))
        q = rng.standard_normal((bsz, lq, hq, d))
        causal = bool(trial % 2)
        scale = 0.37
        out, lse = oracle.fwd_kvcache(q, kc, vc, lens, table, scale=scale, causal=causal)
        ref, ref_lse = _brute_force_paged(q, kc, vc, lens, table, scale, causal)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-11)


def test_brute_force_tiny():
    _check_brute_force()


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(2)
    lk, d = 33, 16
    key = rng.standard_normal(d)
    k = np.tile(key, (lk, 1, 1)).reshape(lk, 1, d)
    v = rng.standard_normal((lk, 1, d))
    q = rng.standard_normal((1, 1, d))
    out, lse = oracle.attend_rows(q, k, v, 0.5, False)
    np.testing.assert_allclose(out[0, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], 0.5 * q[0, 0] @ key + math.log(lk), atol=1e-12)


def test_single_key_returns_v():
    rng = np.random.default_rng(3)
    q, k, v = _rand_case(rng, 1, 1, 4, 2, 8)
    out, lse = oracle.attend_rows(q, k, v, 0.3, False)
    for h in range(4):
        assert np.array_equal(out[0, h], v[0, h // 2])
        assert abs(lse[h, 0] - 0.3 * q[0, h] @ k[0, h // 2]) < 1e-12


def test_empty_rows():
    q = np.ones((2, 1, 4))
    out, lse = oracle.attend_rows(q, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 1.0, False)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    # causal rows that see no key: Lq > Lk
    q3 = np.ones((3, 1, 4))
    k = np.ones((1, 1, 4))
    out, lse = oracle.attend_rows(q3, k, k, 1.0, True)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.array_equal(out[2, 0], k[0, 0])


@pytest.mark.parametrize("page", [16, 32, 256])
def test_page_permutation_matches_contiguous(page):
    """Any page size: the rows scattered over permuted pages of P slots (the
    cache's second dimension) give the contiguous result."""
    rng = np.random.default_rng(4)
    bsz, lk, hkv, hq, d = 3, 70 if page < 256 else 600, 2, 4, 8
    contig_k = rng.standard_normal((bsz, lk, hkv, d))
    contig_v = rng.standard_normal((bsz, lk, hkv, d))
    npg = -(-lk // page)
    pool = bsz * npg
    perm = rng.permutation(pool)
    table = perm.reshape(bsz, npg)
    kc = np.zeros((pool, page, hkv, d))
    vc = np.zeros((pool, page, hkv, d))
    for b in range(bsz):
        for t in range(lk):
            kc[table[b, t // page], t % page] = contig_k[b, t]
            vc[table[b, t // page], t % page] = contig_v[b, t]
    q = rng.standard_normal((bsz, 2, hq, d))
    lens = [lk, 50, 17] if page < 256 else [lk, 300, 257]
    o1, l1 = oracle.fwd_kvcache(q, kc, vc, lens, table, causal=True)
    o2, l2 = oracle.fwd_kvcache(q, contig_k, contig_v, lens, None, causal=True)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_split_then_combine_equals_unsplit(splits):
    rng = np.random.default_rng(5 + splits)
    q, k, v = _rand_case(rng, 3, 83, 4, 2, 16)
    o1, l1 = oracle.attend_rows(q, k, v, 0.25, True)
    o2, l2 = oracle.split_then_combine(q, k, v, 0.25, True, splits)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_combine_with_empty_splits():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((3, 2, 5))
    lse = np.array([[0.5, -np.inf], [-np.inf, -np.inf], [1.5, -np.inf]])
    out, l = oracle.combine_splits(o, lse)
    w0, w2 = math.exp(0.5), math.exp(1.5)
    np.testing.assert_allclose(out[0], (w0 * o[0, 0] + w2 * o[2, 0]) / (w0 + w2), atol=1e-12)
    assert abs(l[0] - math.log(w0 + w2)) < 1e-12
    assert np.all(out[1] == 0) and np.isneginf(l[1])
    # the partial output of an empty split is never read (it may hold anything)
    o_nan = o.copy()
    o_nan[1, 0] = np.nan
    out2, _ = oracle.combine_splits(o_nan, lse)
    assert np.array_equal(out2, out)


def test_causal_prefix_equals_stepwise_decode():
    rng = np.random.default_rng(7)
    old, n, hq, hkv, d = 21, 9, 4, 2, 8
    k_all = rng.standard_normal((1, old + n, hkv, d))
    v_all = rng.standard_normal((1, old + n, hkv, d))
    q = rng.standard_normal((1, n, hq, d))
    o_pre, l_pre = oracle.fwd_kvcache(q, k_all[:, :old], v_all[:, :old], [old], None,
                                      k_new=k_all[:, old:], v_new=v_all[:, old:], causal=True)
    for i in range(n):
        o_i, l_i = oracle.fwd_kvcache(q[:, i:i + 1], k_all, v_all, [old + i + 1], None,
                                      causal=False)
        np.testing.assert_allclose(o_pre[:, i], o_i[:, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_pre[:, :, i], l_i[:, :, 0], rtol=0, atol=1e-12)


def test_varlen_matches_kvcache_after_append():
    rng = np.random.default_rng(8)
    hq, hkv, d = 4, 4, 8
    old = [5, 40, 0]
    lq = [7, 1, 16]
    pages = [-(-(o + l) // 16) for o, l in zip(old, lq)]
    pool = sum(pages)
    perm = rng.permutation(pool)
    table = np.zeros((3, max(pages)), dtype=np.int64)
    off = 0
    for b in range(3):
        table[b, :pages[b]] = perm[off:off + pages[b]]
        off += pages[b]
    kc = rng.standard_normal((pool, 16, hkv, d))
    vc = rng.standard_normal((pool, 16, hkv, d))
    q_packed = rng.standard_normal((sum(lq), hq, d))
    kn = [rng.standard_normal((l, hkv, d)) for l in lq]
    vn = [rng.standard_normal((l, hkv, d)) for l in lq]
    cu = np.concatenate([[0], np.cumsum(lq)])
    kc2, vc2 = kc.copy(), vc.copy()
    for b in range(3):
        kc2, vc2 = oracle.append_kv(kc2, vc2, kn[b][None], vn[b][None], [old[b]],
                                    table[b:b + 1])
    o_var, l_var = oracle.fwd_varlen(q_packed, kc2, vc2, cu, [o + l for o, l in zip(old, lq)],
                                     table, causal=True)
    for b in range(3):
        o_b, l_b = oracle.fwd_kvcache(q_packed[None, cu[b]:cu[b + 1]], kc, vc, [old[b]],
                                      table[b:b + 1], k_new=kn[b][None], v_new=vn[b][None],
                                      causal=True)
        np.testing.assert_allclose(o_var[cu[b]:cu[b + 1]], o_b[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_var[:, cu[b]:cu[b + 1]], l_b[0], rtol=0, atol=1e-13)


def test_varlen_padding_sequences_are_inert():
    rng = np.random.default_rng(9)
    hq, d = 2, 8
    kc = rng.standard_normal((4, 16, hq, d))
    table = np.array([[0, 1], [2, 3], [0, 0], [0, 0]])
    q = rng.standard_normal((6, hq, d))
    o1, l1 = oracle.fwd_varlen(q, kc, kc, [0, 5, 6], [20, 30], table[:2], causal=True)
    o2, l2 = oracle.fwd_varlen(q, kc, kc, [0, 5, 6, 6, 6], [20, 30, 0, 0], table, causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---- planted mistakes: every one must break at least one pin --------------

def _pins():
    return [lambda: _check_golden("two_keys_softmax.json"),
            lambda: _check_golden("causal_bottom_right.json"),
            lambda: _check_golden("gqa_mapping.json"),
            _check_append_golden, _paged_gather_closed_form, _check_torch_sdpa,
            _check_brute_force]


def _some_pin_fails():
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            return True
    return False


def test_pins_pass_unmodified():
    assert not _some_pin_fails()


MUTATIONS = {
    "gqa_modulo_mapping": ("kv_head_of", lambda h, hq, hkv: h % hkv),
    "causal_top_left": ("visible_keys",
                        lambda i, lq, lk, causal: min(lk, i + 1) if causal else lk),
    "causal_off_by_one": ("visible_keys",
                          lambda i, lq, lk, causal: max(0, min(lk, i + lk - lq)) if causal else lk),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(monkeypatch, name):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(oa, attr, fn)
    assert _some_pin_fails(), name


def test_planted_gather_mistake_is_caught(monkeypatch):
    def bad_gather(cache, table_row, length, page_size=16):
        t = np.arange(length)
        return cache[np.asarray(table_row)[t % len(table_row)], t % page_size]
    monkeypatch.setattr(oa, "gather_pages", bad_gather)
    assert _some_pin_fails()


def test_planted_append_mistake_is_caught(monkeypatch):
    real = oa.append_kv

    def bad_append(k_cache, v_cache, k_new, v_new, cache_seqlens, block_table=None, page_size=16):
        return real(k_cache, v_cache, k_new, v_new, [int(s) + 1 for s in cache_seqlens],
                    block_table, page_size)
    monkeypatch.setattr(oa, "append_kv", bad_append)
    monkeypatch.setattr(oracle, "append_kv", bad_append)
    assert _some_pin_fails()


def test_planted_scale_mistake_is_caught(monkeypatch):
    real = oa.attend_rows

    def bad(q, k, v, scale, causal):
        return real(q, k, v, scale * 1.01, causal)
    monkeypatch.setattr(oa, "attend_rows", bad)
    monkeypatch.setattr(oracle, "attend_rows", bad)
    assert _some_pin_fails()
