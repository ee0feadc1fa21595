"""Rotary position embedding of the new tokens (oracle; test infrastructure).

The pages name the feature only: [p1] "Add support for small page sizes"
mentions a fix to fused RoPE embeddings in the kvcache forward, without
defining it.  The definition followed here is the published one (Su et al.,
"RoFormer: Enhanced Transformer with Rotary Position Embedding", 2021, the
rotation of each 2-D pair of features by the angle pos * theta_i), with the
two common pairings of the features and tables supplied by the caller:

* rotary_dim = 2 * cos.shape[1] <= D features are rotated; the rest pass
  through unchanged.
* Split halves (interleaved=False): feature p pairs with p + rotary_dim / 2.
  Interleaved (interleaved=True): feature 2p pairs with 2p + 1.
* (x1, x2) -> (x1 cos - x2 sin, x1 sin + x2 cos), with cos = cos[pos, p] and
  sin = sin[pos, p] for pair p of a token at position pos.

Readings where the pages are silent (stated once more in the design notes):
new token i of sequence b sits at position cache_seqlens[b] + i, the slot
the append writes it to; query row i of Lq sits at cache_seqlens[b] + Lnew -
Lq + i (the new tokens are the last Lq positions, the bottom-right alignment
of the causal mask); the rotated values are rounded once to the cache dtype,
as they are stored (k) or fed to the attention (q) in that dtype.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA library.
"""

import numpy as np


def round_to(x, dtype):
    """Round float64 values to the nearest fp16 ('f16') or bf16 ('bf16') value
    (ties to even), returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        # 8 significant bits: scale the mantissa to an integer grid of 2^8
        # steps per binade and round half to even (np.round), then scale back
        m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
        return np.ldexp(np.round(m * 256.0) / 256.0, e)
    raise ValueError(dtype)


def rotary(x, cos, sin, positions, interleaved=False):
    """Rotate the first 2 * cos.shape[1] features of every row of x.

    x ``[L, H, D]`` (or ``[L, D]``) float64; cos, sin ``[S, r/2]``;
    positions ``[L]`` integers in [0, S).  Returns float64, unrounded.
    """
    x = np.asarray(x, dtype=np.float64)
    squeeze = x.ndim == 2
    if squeeze:
        x = x[:, None, :]
    cos = np.asarray(cos, dtype=np.float64)
    sin = np.asarray(sin, dtype=np.float64)
    half = cos.shape[1]
    out = x.copy()
    for row, pos in enumerate(positions):
        c = cos[int(pos)]
        s = sin[int(pos)]
        for p in range(half):
            if interleaved:
                i1, i2 = 2 * p, 2 * p + 1
            else:
                i1, i2 = p, p + half
            x1 = x[row, :, i1]
            x2 = x[row, :, i2]
            out[row, :, i1] = x1 * c[p] - x2 * s[p]
            out[row, :, i2] = x1 * s[p] + x2 * c[p]
    return out[:, 0, :] if squeeze else out


def rotate_new_tokens(q, k_new, cos, sin, cache_seqlens, interleaved, dtype):
    """Rotated q ``[B, Lq, Hq, D]`` and k_new ``[B, Lnew, Hkv, D]`` of a
    kvcache call, rounded to ``dtype``, at the positions stated above."""
    q = np.asarray(q, dtype=np.float64)
    k_new = np.asarray(k_new, dtype=np.float64)
    bsz, lq = q.shape[0], q.shape[1]
    lnew = k_new.shape[1]
    q_rot = np.empty_like(q)
    k_rot = np.empty_like(k_new)
    for b in range(bsz):
        base = int(cache_seqlens[b])
        q_rot[b] = round_to(rotary(q[b], cos, sin, [base + lnew - lq + i for i in range(lq)],
                                   interleaved), dtype)
        k_rot[b] = round_to(rotary(k_new[b], cos, sin, [base + i for i in range(lnew)],
                                   interleaved), dtype)
    return q_rot, k_rot
