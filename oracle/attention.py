"""Exact paged KV-cache attention in numpy float64 (oracle; test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA library.

Definition followed (restated from the pages, see the package docstring for
the page list):

* Paged cache layout ``[num_pages, P, Hkv, D]`` with P tokens per page (the
  cache's second dimension: 16 in the configurations, 256 in the comparison
  of [p4]); ``block_table[b, j]`` is the physical page holding logical page j
  of sequence b -- [p1] "Add support for small page sizes", reproduction
  snippet (``key_cache = [num_blocks, block_size, num_heads, head_dim]``,
  ``block_tables = [bs, cdiv(seq_len, block_size)]``); [p4] "Introduce
  flash-attn", the block size 16 vs 256 comparison.
* Non-paged cache ``[B, max_len, Hkv, D]`` whose valid length per sequence is
  ``cache_seqlens[b]`` -- [p3] "Inappropriate Number of Splits ...", opening
  report (cache preallocated to 131072 tokens, real length from
  ``cache_seqlens``).
* ``k=``/``v=`` append: the new tokens are written at positions
  ``cache_seqlens[b] .. cache_seqlens[b] + Lnew - 1`` through the block table;
  nothing is allocated -- [p1], reply explaining that the function uses
  ``block_table`` to find the addresses to read and write.
* Attention: ``softmax(scale * q k^T) v`` per query head, with query head h
  reading kv head ``h // (Hq / Hkv)`` (MHA when Hq == Hkv, GQA otherwise) --
  [p4] "Introduce flash-attn", opening description (MHA and MQA/GQA).
* Causal masking aligned to the bottom-right corner: query row i of Lq sees
  keys ``t <= i + Lk - Lq``.  This is the only alignment under which a
  causal prefill over a cached prefix reproduces token-by-token decoding,
  which is what the [p1] reproduction (``causal=True`` with a non-empty cache)
  relies on.
* Split-KV: per-split partial outputs and log-sum-exps merged by a combine
  step -- [p2] "Unify the kernel ...", comment on ``flash_fwd_splitkv_kernel``
  being dispatched when ``num_splits`` is 0 with a page table; [p3] the
  ``num_splits`` discussion.  The pages do not spell out the combine; the
  oracle uses the exact log-sum-exp merge, which is the unique way to recover
  the unsplit softmax from per-split (O, LSE) pairs.

Readings where the pages are silent: the default scale is 1/sqrt(D); LSE is
the natural-log log-sum-exp of the scaled scores; a row with no visible key
gives O = 0 and LSE = -inf; ``cache_seqlens`` is an input only (the append
does not update it).
"""

import math

import numpy as np

PAGE_SIZE = 16


def kv_head_of(h, num_q_heads, num_kv_heads):
    """KV head read by query head h: consecutive query heads share a kv head."""
    group = num_q_heads // num_kv_heads
    return h // group


def visible_keys(i, lq, lk, causal):
    """Number of keys (a prefix [0, n)) visible to query row i of lq rows.

    Non-causal rows see all lk keys.  Causal rows see ``t <= i + lk - lq``
    (bottom-right alignment), clipped to [0, lk].
    """
    if not causal:
        return lk
    return max(0, min(lk, i + lk - lq + 1))


def gather_pages(cache, table_row, length, page_size=PAGE_SIZE):
    """Logical rows [0, length) of one sequence in a paged cache.

    Row t lives in physical page ``table_row[t // page_size]`` at slot
    ``t % page_size``.  Entries of ``table_row`` past ``ceil(length/P)`` are
    never read.
    """
    t = np.arange(length)
    pages = np.asarray(table_row)[t // page_size]
    return cache[pages, t % page_size]


def logical_kv(k_cache, v_cache, b, old_len, k_new=None, v_new=None, block_table=None):
    """Keys/values of sequence b as float64 ``[Lk, Hkv, D]``.

    Positions ``< old_len`` come from the cache (through ``block_table[b]`` if
    paged, else row ``[b, t]`` of a contiguous cache); positions ``>= old_len``
    come from ``k_new[b]`` / ``v_new[b]``.
    """
    if block_table is None:
        k_old = k_cache[b, :old_len]
        v_old = v_cache[b, :old_len]
    else:
        k_old = gather_pages(k_cache, block_table[b], old_len, k_cache.shape[1])
        v_old = gather_pages(v_cache, block_table[b], old_len, v_cache.shape[1])
    k_old = np.asarray(k_old, dtype=np.float64)
    v_old = np.asarray(v_old, dtype=np.float64)
    if k_new is None:
        return k_old, v_old
    kk = np.concatenate([k_old, np.asarray(k_new[b], dtype=np.float64)], axis=0)
    vv = np.concatenate([v_old, np.asarray(v_new[b], dtype=np.float64)], axis=0)
    return kk, vv


def attend_rows(q, k, v, scale, causal):
    """Exact attention of one sequence.

    q ``[Lq, Hq, D]``, k/v ``[Lk, Hkv, D]`` -> (O ``[Lq, Hq, D]``, LSE ``[Hq, Lq]``)
    in float64.  For each query head h and row i: s_t = scale * <q_i, k_t>
    over the visible keys, m = max s, l = sum exp(s - m),
    O = sum exp(s - m) v_t / l, LSE = m + ln l.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lq, hq, d = q.shape
    lk, hkv = k.shape[0], k.shape[1]
    out = np.zeros((lq, hq, d), dtype=np.float64)
    lse = np.full((hq, lq), -np.inf, dtype=np.float64)
    for h in range(hq):
        g = kv_head_of(h, hq, hkv)
        scores = scale * (q[:, h, :] @ k[:, g, :].T)  # [Lq, Lk]
        for i in range(lq):
            n = visible_keys(i, lq, lk, causal)
            if n == 0:
                continue
            s = scores[i, :n]
            m = s.max()
            w = np.exp(s - m)
            l = w.sum()
            out[i, h] = (w @ v[:n, g, :]) / l
            lse[h, i] = m + math.log(l)
    return out, lse


def append_kv(k_cache, v_cache, k_new, v_new, cache_seqlens, block_table=None,
              page_size=None):
    """Bit copy of the new tokens into the cache; returns updated copies.

    Works on any dtype (pass integer bit views for a bit-exact check).  New
    token i of sequence b lands at position ``cache_seqlens[b] + i``: page
    ``block_table[b, pos // P]`` slot ``pos % P`` (paged) or row ``[b, pos]``
    (contiguous).  Sequences are applied in order b = 0, 1, ...
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    if page_size is None:
        page_size = kc.shape[1]
    bsz, lnew = k_new.shape[0], k_new.shape[1]
    for b in range(bsz):
        for i in range(lnew):
            pos = int(cache_seqlens[b]) + i
            if block_table is None:
                kc[b, pos] = k_new[b, i]
                vc[b, pos] = v_new[b, i]
            else:
                page = int(block_table[b][pos // page_size])
                kc[page, pos % page_size] = k_new[b, i]
                vc[page, pos % page_size] = v_new[b, i]
    return kc, vc


def fwd_kvcache(q, k_cache, v_cache, cache_seqlens, block_table=None, k_new=None,
                v_new=None, scale=None, causal=False):
    """``flash_attn_with_kvcache``-style forward (optionally with append).

    q ``[B, Lq, Hq, D]``; caches paged ``[num_pages, 16, Hkv, D]`` (with
    ``block_table [B, max_pages]``) or contiguous ``[B, max_len, Hkv, D]``
    (``block_table=None``); optional ``k_new``/``v_new`` ``[B, Lnew, Hkv, D]``.
    Sequence b attends over Lk = cache_seqlens[b] + Lnew keys.
    Returns O ``[B, Lq, Hq, D]`` and LSE ``[B, Hq, Lq]`` in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, lq, hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((bsz, lq, hq, d), dtype=np.float64)
    lse = np.full((bsz, hq, lq), -np.inf, dtype=np.float64)
    for b in range(bsz):
        kk, vv = logical_kv(k_cache, v_cache, b, int(cache_seqlens[b]), k_new, v_new,
                            block_table)
        out[b], lse[b] = attend_rows(q[b], kk, vv, scale, causal)
    return out, lse


def fwd_varlen(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table, scale=None,
               causal=True):
    """Unified varlen forward over a paged cache (one mixed batch).

    q ``[total_q, Hq, D]`` packed by ``cu_seqlens_q [B+1]`` (non-decreasing;
    repeated entries are empty padding sequences that produce nothing).
    Sequence b's keys are the first ``seqlens_k[b]`` cache rows (the new chunk
    is already in the cache).  Returns O ``[total_q, Hq, D]`` and LSE
    ``[Hq, total_q]`` in float64; rows of padding never exist.
    """
    q = np.asarray(q, dtype=np.float64)
    total_q, hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((total_q, hq, d), dtype=np.float64)
    lse = np.full((hq, total_q), -np.inf, dtype=np.float64)
    for b in range(len(cu_seqlens_q) - 1):
        q0, q1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        if q1 == q0:
            continue
        lk = int(seqlens_k[b])
        kk = np.asarray(gather_pages(k_cache, block_table[b], lk, k_cache.shape[1]),
                        dtype=np.float64)
        vv = np.asarray(gather_pages(v_cache, block_table[b], lk, v_cache.shape[1]),
                        dtype=np.float64)
        o_b, lse_b = attend_rows(q[q0:q1], kk, vv, scale, causal)
        out[q0:q1] = o_b
        lse[:, q0:q1] = lse_b
    return out, lse


def combine_splits(o_parts, lse_parts):
    """Merge per-split normalised outputs by their log-sum-exps.

    o_parts ``[S, ..., D]``, lse_parts ``[S, ...]``:
    LSE = ln sum_s exp(LSE_s);  O = sum_s exp(LSE_s - LSE) O_s.
    Splits with LSE_s = -inf contribute nothing; if all are -inf the result
    is O = 0, LSE = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe), 0.0)
    total = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, total, 1.0)), -np.inf)
    coef = np.where(finite, w / np.where(finite, total, 1.0), 0.0)
    # an empty split's partial output is undefined and is never read
    live = np.isfinite(lse_parts)[..., None]
    out = np.where(live, coef[..., None] * np.where(live, o_parts, 0.0), 0.0).sum(axis=0)
    return out, lse


def split_then_combine(q, k, v, scale, causal, num_splits, page_size=PAGE_SIZE):
    """Same result as :func:`attend_rows`, computed as split-KV + combine.

    Split s covers keys ``[s*C, min((s+1)*C, Lk))`` with
    ``C = ceil(ceil(Lk/P)/S) * P``; each split attends over its visible keys
    and the partials are merged with :func:`combine_splits`.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lq, hq, d = q.shape
    lk, hkv = k.shape[0], k.shape[1]
    pages = -(-lk // page_size)
    chunk = max(1, -(-pages // num_splits)) * page_size
    o_parts = np.zeros((num_splits, lq, hq, d))
    lse_parts = np.full((num_splits, hq, lq), -np.inf)
    for s in range(num_splits):
        k0, k1 = s * chunk, min((s + 1) * chunk, lk)
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            for i in range(lq):
                n = min(visible_keys(i, lq, lk, causal), k1)
                if n <= k0:
                    continue
                sc = scale * (k[k0:n, g, :] @ q[i, h, :])
                m = sc.max()
                w = np.exp(sc - m)
                l = w.sum()
                o_parts[s, i, h] = (w @ v[k0:n, g, :]) / l
                lse_parts[s, h, i] = m + math.log(l)
    # o_parts is [S, Lq, Hq, D] but lse_parts is [S, Hq, Lq]: align them.
    o, lse_hl = combine_splits(o_parts.transpose(0, 2, 1, 3), lse_parts)
    return o.transpose(1, 0, 2), lse_hl
