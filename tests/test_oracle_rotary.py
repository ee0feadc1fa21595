"""Pins of the rotary-embedding oracle against what the mathematics fixes
(CPU only).  RoFormer's rotation of feature pairs by pos * theta_i is an
orthogonal map whose composition depends only on relative position:
  <R_m q, R_n k> = <R_{m-n} q, k>,
and pairing features as interleaved (2p, 2p+1) or as split halves
(p, p + r/2) differ by a fixed permutation of the features.  A dropped
term, a wrong sign of sin, a swapped pair or a wrong position fails one of
these."""

import math

import numpy as np
import pytest

import oracle


def tables(n_pos, rotary_dim, base=10000.0):
    """cos/sin tables of angle pos * base^(-2p / rotary_dim), float64."""
    p = np.arange(rotary_dim // 2)
    theta = base ** (-2.0 * p / rotary_dim)
    ang = np.arange(n_pos)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


@pytest.mark.parametrize("interleaved", [False, True])
def test_pair_norms_preserved(interleaved):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 64))
    cos, sin = tables(50, 48)
    pos = [0, 7, 13, 31, 49]
    y = oracle.rotary(x, cos, sin, pos, interleaved)
    for p in range(24):
        i1, i2 = (2 * p, 2 * p + 1) if interleaved else (p, p + 24)
        assert np.allclose(x[..., i1] ** 2 + x[..., i2] ** 2, y[..., i1] ** 2 + y[..., i2] ** 2)
    # features past rotary_dim pass through
    assert np.array_equal(x[..., 48:], y[..., 48:])


@pytest.mark.parametrize("interleaved", [False, True])
def test_relative_position(interleaved):
    rng = np.random.default_rng(2)
    d = 32
    q = rng.standard_normal((1, d))
    k = rng.standard_normal((1, d))
    cos, sin = tables(64, d)
    for m, n in [(5, 2), (40, 40), (63, 0), (17, 11)]:
        lhs = float(oracle.rotary(q, cos, sin, [m], interleaved)[0]
                    @ oracle.rotary(k, cos, sin, [n], interleaved)[0])
        rhs = float(oracle.rotary(q, cos, sin, [m - n], interleaved)[0] @ k[0])
        assert math.isclose(lhs, rhs, rel_tol=1e-12, abs_tol=1e-12), (m, n)


def test_interleaved_is_a_permutation_of_split_halves():
    rng = np.random.default_rng(3)
    d, r = 64, 64
    x = rng.standard_normal((4, 2, d))
    cos, sin = tables(10, r)
    perm = np.concatenate([np.arange(0, r, 2), np.arange(1, r, 2)])  # interleaved -> halves
    a = oracle.rotary(x, cos, sin, [1, 3, 5, 9], interleaved=True)
    b = oracle.rotary(x[..., perm], cos, sin, [1, 3, 5, 9], interleaved=False)
    assert np.allclose(a[..., perm], b)


def test_identity_at_zero_angle_and_quarter_turn():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 16))
    cos = np.array([[1.0] * 8, [0.0] * 8])
    sin = np.array([[0.0] * 8, [1.0] * 8])
    assert np.array_equal(oracle.rotary(x, cos, sin, [0, 0]), x)
    # a quarter turn maps (x1, x2) -> (-x2, x1)
    y = oracle.rotary(x, cos, sin, [1, 1])
    assert np.array_equal(y[:, :8], -x[:, 8:]) and np.array_equal(y[:, 8:], x[:, :8])


def test_round_to_matches_the_formats():
    import torch
    rng = np.random.default_rng(5)
    x = rng.standard_normal(10000) * 3
    # fp16: numpy's correctly rounded conversion; bf16: against torch's
    # float32 -> bfloat16 conversion on values exact in float32
    x32 = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.round_to(x32, "f16"), x32.astype(np.float16).astype(np.float64))
    ref = torch.from_numpy(x32).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_to(x32, "bf16"), ref)


def test_new_token_positions_follow_the_append():
    """Token i of sequence b is rotated at cache_seqlens[b] + i (k) and the
    last Lq positions (q): with Lq = Lnew the two agree row by row."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 3, 2, 32))
    k = rng.standard_normal((2, 3, 1, 32))
    cos, sin = tables(40, 32)
    lens = [5, 30]
    qr, kr = oracle.rotate_new_tokens(q, k, cos, sin, lens, False, "f16")
    for b in range(2):
        for i in range(3):
            pos = lens[b] + i
            assert np.array_equal(kr[b, i], oracle.round_to(
                oracle.rotary(k[b, i:i + 1], cos, sin, [pos])[0], "f16"))
            assert np.array_equal(qr[b, i], oracle.round_to(
                oracle.rotary(q[b, i:i + 1], cos, sin, [pos])[0], "f16"))


def test_planted_mistakes_are_caught(monkeypatch):
    """A rotation the wrong way (sin negated) still satisfies the relative-
    position identity; the quarter turn fixes the direction and the pairing."""
    real = oracle.rotary

    def wrong_sign(x, cos, sin, positions, interleaved=False):
        return real(x, cos, -np.asarray(sin), positions, interleaved)

    def wrong_pairing(x, cos, sin, positions, interleaved=False):
        return real(x, cos, sin, positions, not interleaved)

    for wrong in (wrong_sign, wrong_pairing):
        monkeypatch.setattr(oracle, "rotary", wrong)
        with pytest.raises(AssertionError):
            test_identity_at_zero_angle_and_quarter_turn()
    monkeypatch.setattr(oracle, "rotary", real)
