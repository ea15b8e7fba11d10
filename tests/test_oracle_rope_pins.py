"""Pins for the oracle's decoupled RoPE ("Tearing open DeepSeek MLA source"
page, §1: a 64-d RoPE key carries position apart from the latent; §3 and §4:
the RoPE table is generated and applied in fp32).

The pages print no rotation formula, so these pins check what any correct
rotary embedding must satisfy, plus textbook values that fix the reading
(consecutive pairs, angle p * 10000^(-2i/64)):

* position 0 is the identity; every pair keeps its norm;
* the score of two rotated vectors depends only on their position
  difference, and rotations compose;
* pair 0 at position 1 turns a unit vector by exactly 1 rad, i.e. lands on
  (cos 1, sin 1) = (0.5403023058681398, 0.8414709848078965), and the last
  pair turns by 1 rad at position 10000^(62/64);
* planted mistakes (a flipped sign, the rotate-half pair layout, an
  off-by-one frequency index) each fail at least one pin.
"""
import numpy as np
import pytest

import oracle

COS1, SIN1 = 0.5403023058681398, 0.8414709848078965  # textbook values of cos(1), sin(1)


def _pins(apply):
    """Run every pin against a rotation function; return the names that fail."""
    rng = np.random.default_rng(7)
    failed = []
    x = rng.standard_normal((5, 64))
    if not np.array_equal(apply(x, 0), x):
        failed.append("identity")
    p = rng.integers(0, 65536, size=5)
    r = apply(x, p)
    n0 = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    n1 = r[:, 0::2] ** 2 + r[:, 1::2] ** 2
    if not np.allclose(n0, n1, rtol=1e-12, atol=0):
        failed.append("pair norms")
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in [(7, 3), (40000, 123), (65535, 65000)]:
        lhs = np.dot(apply(q, m), apply(k, n))
        rhs = np.dot(apply(q, m - n), k)
        if abs(lhs - rhs) > 1e-9 * (np.linalg.norm(q) * np.linalg.norm(k)):
            failed.append(f"relative position {m},{n}")
            break
    if not np.allclose(apply(apply(x, 1000), 2345), apply(x, 3345), rtol=0, atol=1e-9):
        failed.append("composition")
    e0 = np.zeros(64)
    e0[0] = 1.0
    if not np.allclose(apply(e0, 1)[:2], [COS1, SIN1], rtol=0, atol=1e-15) or np.any(apply(e0, 1)[2:] != 0):
        failed.append("pair 0 at position 1")
    e_last = np.zeros(64)
    e_last[62] = 1.0
    got = apply(e_last, 10000.0 ** (62.0 / 64.0))
    if not np.allclose(got[62:], [COS1, SIN1], rtol=0, atol=1e-12):
        failed.append("last pair at position 10000^(62/64)")
    return failed


def test_rope_oracle_passes_every_pin():
    assert _pins(oracle.rope_apply) == []


def test_rope_table_matches_the_rotation_of_unit_vectors():
    tab = oracle.rope_table(300)
    rng = np.random.default_rng(1)
    for p in rng.integers(0, 300, size=6):
        for i in (0, 5, 31):
            e = np.zeros(64)
            e[2 * i] = 1.0
            r = oracle.rope_apply(e, int(p))
            assert np.allclose(r[2 * i:2 * i + 2], tab[p, i], rtol=0, atol=1e-15)


def test_rope_broadcasts_positions_over_heads():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 128, 64))
    pos = np.array([5, 900, 60000])
    r = oracle.rope_apply(x, pos[:, None])
    for t in range(3):
        for h in (0, 77, 127):
            assert np.allclose(r[t, h], oracle.rope_apply(x[t, h], pos[t]), rtol=0, atol=1e-13)


def _flipped_sign(x, positions):
    x = np.asarray(x, dtype=np.float64)
    a = oracle.rope_angles(positions)
    c, s = np.cos(a), np.sin(a)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c + x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


def _rotate_half(x, positions):
    x = np.asarray(x, dtype=np.float64)
    a = oracle.rope_angles(positions)
    c, s = np.cos(a), np.sin(a)
    out = np.empty_like(x)
    out[..., :32] = x[..., :32] * c - x[..., 32:] * s
    out[..., 32:] = x[..., :32] * s + x[..., 32:] * c
    return out


def _freq_off_by_one(x, positions):
    x = np.asarray(x, dtype=np.float64)
    p = np.asarray(positions, dtype=np.float64)[..., None]
    a = p * 10000.0 ** (-2.0 * (np.arange(32) + 1) / 64)
    c, s = np.cos(a), np.sin(a)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


@pytest.mark.parametrize("wrong", [_flipped_sign, _rotate_half, _freq_off_by_one])
def test_planted_rope_mistakes_are_caught(wrong):
    assert _pins(wrong), f"{wrong.__name__} passed every pin"
