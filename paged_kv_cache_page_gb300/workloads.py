"""Seeded synthetic inputs for paged KV-cache attention.

This module holds no attention arithmetic: it only draws tensors (values,
lengths, block tables) so that the CUDA path and the CPU oracle see the same
bits.  Shapes, value distributions and length mixes follow the workloads the
pages benchmark (vLLM ``benchmark_paged_attention.py`` decode sweep, the
flash-attention small-page reproduction, the ``determine_num_splits`` report
and the unified-kernel A100 table); the scripts themselves are not available,
so these seeded draws stand in for them.

Every generator takes a ``seed`` and a ``device``; with the same seed and
device the draw is identical.  Values are generated directly on ``device``
(large pools would take minutes to draw on the host).
"""

import math

import torch

PAGE_SIZE = 16

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _values(shape, dtype, dist, g, device):
    if dist == "normal":
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)
    if dist == "uniform":
        return torch.rand(shape, generator=g, device=device, dtype=torch.float32).to(dtype)
    raise ValueError(dist)


def _distinct_tables(pages_per_seq, pool, g, device):
    """Block tables of distinct random physical pages, one row per sequence.

    Row b holds ``pages_per_seq[b]`` distinct pages drawn from a random
    permutation of the pool; the row is padded to the widest row with the
    value ``pool`` (an out-of-range sentinel that is never read).
    """
    width = max(1, max(pages_per_seq))
    perm = torch.randperm(pool, generator=g, device="cpu").to(torch.int32)
    table = torch.full((len(pages_per_seq), width), pool, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[off:off + n]
        off += n
    if off > pool:
        raise ValueError("pool too small for the requested pages")
    return table.to(device)


def paged_decode(batch, ctx, num_q_heads=32, num_kv_heads=32, head_dim=128, dtype="f16",
                 lnew=0, seed=1002, device="cpu", lens=None, dist="normal", pool=None,
                 page_size=PAGE_SIZE):
    """Paged decode: Lq = 1 (or ``lnew`` new tokens with in-kernel append).

    Every sequence holds ``ctx`` keys after the call: ``cache_seqlens = ctx - lnew``
    old tokens plus ``lnew`` appended ones (or the given per-sequence ``lens``).
    Pool = exactly the pages the batch needs; the block table is a random
    permutation of the pool reshaped per sequence, each row exactly
    ``ceil(Lk/16)`` wide when all lengths are equal.
    """
    dt = DTYPES[dtype]
    g = _gen(seed, device)
    if lens is None:
        lens = [ctx] * batch
    pages = [-(-int(l) // page_size) for l in lens]
    num_pages = sum(pages) if pool is None else pool
    table = _distinct_tables(pages, num_pages, torch.Generator().manual_seed(seed), device)
    lq = max(1, lnew)
    k_cache = _values((num_pages, page_size, num_kv_heads, head_dim), dt, dist, g, device)
    v_cache = _values((num_pages, page_size, num_kv_heads, head_dim), dt, dist, g, device)
    q = _values((batch, lq, num_q_heads, head_dim), dt, dist, g, device)
    if lnew > 0:
        k_new = _values((batch, lnew, num_kv_heads, head_dim), dt, dist, g, device)
        v_new = _values((batch, lnew, num_kv_heads, head_dim), dt, dist, g, device)
    else:
        k_new = v_new = None
    cache_seqlens = torch.tensor([int(l) - lnew for l in lens], dtype=torch.int32, device=device)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
                cache_seqlens=cache_seqlens, block_table=table, num_pages=num_pages,
                scale=1.0 / math.sqrt(head_dim), causal=False, dtype=dtype,
                num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim)


def tiny_decode(seed=1001, device="cpu"):
    """Two sequences of 37 and 100 cached tokens, 4 q / 2 kv heads, D = 64.

    64-page pool; the block table is one seeded permutation of the 64 pages
    split into two rows of 32 (only the first 3 and 7 entries are used).
    """
    g = _gen(seed, device)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(seed)).to(torch.int32)
    table = perm.reshape(2, 32).to(device)
    k_cache = _values((64, PAGE_SIZE, 2, 64), torch.float16, "normal", g, device)
    v_cache = _values((64, PAGE_SIZE, 2, 64), torch.float16, "normal", g, device)
    q = _values((2, 1, 4, 64), torch.float16, "normal", g, device)
    cache_seqlens = torch.tensor([37, 100], dtype=torch.int32, device=device)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, k_new=None, v_new=None,
                cache_seqlens=cache_seqlens, block_table=table, num_pages=64,
                scale=1.0 / 8.0, causal=False, dtype="f16",
                num_q_heads=4, num_kv_heads=2, head_dim=64)


def gqa_contiguous(batch=8, capacity=131072, num_q_heads=32, num_kv_heads=8, head_dim=128,
                   dtype="bf16", len_lo=1024, len_hi=8192, seed=1003, device="cpu"):
    """Non-paged decode on a preallocated contiguous cache.

    ``cache_seqlens[b] ~ U[len_lo, len_hi]`` (integers).  Only the first
    ``max(cache_seqlens)`` rows of each sequence are drawn (``k_rows``,
    ``v_rows``, shape ``[B, max_len, Hkv, D]``); the caller places them in a
    ``[B, capacity, Hkv, D]`` cache.
    """
    dt = DTYPES[dtype]
    lens = torch.randint(len_lo, len_hi + 1, (batch,), generator=torch.Generator().manual_seed(seed))
    g = _gen(seed, device)
    max_len = int(lens.max())
    k_rows = _values((batch, max_len, num_kv_heads, head_dim), dt, "normal", g, device)
    v_rows = _values((batch, max_len, num_kv_heads, head_dim), dt, "normal", g, device)
    q = _values((batch, 1, num_q_heads, head_dim), dt, "normal", g, device)
    return dict(q=q, k_rows=k_rows, v_rows=v_rows, capacity=capacity,
                cache_seqlens=lens.to(torch.int32).to(device), block_table=None,
                scale=1.0 / math.sqrt(head_dim), causal=False, dtype=dtype,
                num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim)


def prefill_append(batch=4, lnew=170, num_heads=32, head_dim=128, old_lo=0, old_hi=512,
                   pool=1000, dtype="f16", seed=1004, device="cpu", dist="uniform",
                   num_kv_heads=None, page_size=PAGE_SIZE):
    """Causal prefill with the new tokens' k/v appended in the same call.

    ``old_b ~ U[old_lo, old_hi]`` cached tokens per sequence; ``lnew`` new
    query tokens whose k/v are appended; block table of distinct random pages
    covering exactly ``ceil((old_b + lnew)/16)`` pages per sequence from a
    pool of ``pool`` pages.  Values U[0, 1) as in the small-page reproduction.
    """
    dt = DTYPES[dtype]
    hkv = num_heads if num_kv_heads is None else num_kv_heads
    cpu_g = torch.Generator().manual_seed(seed)
    old = torch.randint(old_lo, old_hi + 1, (batch,), generator=cpu_g)
    pages = [-(-(int(o) + lnew) // page_size) for o in old]
    pool = max(pool if page_size == PAGE_SIZE else 0, sum(pages))
    table = _distinct_tables(pages, pool, cpu_g, device)
    g = _gen(seed, device)
    k_cache = _values((pool, page_size, hkv, head_dim), dt, dist, g, device)
    v_cache = _values((pool, page_size, hkv, head_dim), dt, dist, g, device)
    q = _values((batch, lnew, num_heads, head_dim), dt, dist, g, device)
    k_new = _values((batch, lnew, hkv, head_dim), dt, dist, g, device)
    v_new = _values((batch, lnew, hkv, head_dim), dt, dist, g, device)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
                cache_seqlens=old.to(torch.int32).to(device), block_table=table,
                num_pages=pool, scale=1.0 / math.sqrt(head_dim), causal=True, dtype=dtype,
                num_q_heads=num_heads, num_kv_heads=hkv, head_dim=head_dim)


def unified_mixed(num_heads=32, head_dim=128, prefill_lens=(100, 500, 1000), prefix_hi=2048,
                  num_decode=64, ctx_lo=1024, ctx_hi=4096, dtype="bf16", seed=1005,
                  device="cpu", num_kv_heads=None, pad_to=0, page_size=PAGE_SIZE):
    """One mixed batch: chunked-prefill sequences plus decode sequences.

    Prefill sequence j has ``prefill_lens[j]`` query tokens over a cached
    prefix ``~ U[0, prefix_hi]`` (Lk = prefix + Lq; the chunk's own k/v are
    already in the cache).  Decode sequences have Lq = 1 and
    ``Lk ~ U[ctx_lo, ctx_hi]``.  Causal.  ``pad_to`` > B appends empty padding
    sequences (repeated ``cu_seqlens_q`` entries, zero ``seqlens_k``), the
    CUDA-graph padding of the unified-kernel page.
    """
    dt = DTYPES[dtype]
    hkv = num_heads if num_kv_heads is None else num_kv_heads
    cpu_g = torch.Generator().manual_seed(seed)
    prefix = torch.randint(0, prefix_hi + 1, (len(prefill_lens),), generator=cpu_g)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (num_decode,), generator=cpu_g)
    q_lens = list(prefill_lens) + [1] * num_decode
    k_lens = [int(p) + int(l) for p, l in zip(prefix, prefill_lens)] + [int(c) for c in ctx]
    n_real = len(q_lens)
    if pad_to > n_real:
        q_lens += [0] * (pad_to - n_real)
        k_lens += [0] * (pad_to - n_real)
    pages = [-(-k // page_size) for k in k_lens]
    pool = sum(pages)
    table = _distinct_tables(pages, pool, cpu_g, device)
    cu = [0]
    for l in q_lens:
        cu.append(cu[-1] + l)
    g = _gen(seed, device)
    k_cache = _values((pool, page_size, hkv, head_dim), dt, "normal", g, device)
    v_cache = _values((pool, page_size, hkv, head_dim), dt, "normal", g, device)
    q = _values((cu[-1], num_heads, head_dim), dt, "normal", g, device)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache,
                cu_seqlens_q=torch.tensor(cu, dtype=torch.int32, device=device),
                seqlens_k=torch.tensor(k_lens, dtype=torch.int32, device=device),
                block_table=table, num_pages=pool, max_seqlen_q=max(q_lens),
                max_seqlen_k=max(k_lens), scale=1.0 / math.sqrt(head_dim), causal=True,
                dtype=dtype, num_q_heads=num_heads, num_kv_heads=hkv, head_dim=head_dim)
