"""Pins for the oracle's FP8 (E4M3) latent cache.

The E4M3 format is fixed by the OCP 8-bit floating point specification
(1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals m·2^-9,
S.1111.111 NaN, largest finite 448); the pages ([P3] bjbfmj.com/news/60700,
[P1] opening section and §5) only say that a quantised cache carries scale
factors beside its codes.  The pins check the oracle against what does not
depend on it:

* the value of every one of the 256 codes, against PyTorch's float8_e4m3fn
  conversion (a library routine) and against hand-worked values;
* encoding against PyTorch's round-to-nearest-even conversion on random
  values across the normal and subnormal ranges, and on every exact
  midpoint between neighbouring codes (ties go to the even code);
* the scale rule, against a brute-force search for the smallest k;
* the quantisation error bound and the cache round trip.

Planted mistakes (bias 8, truncation, ties away from zero, a scale one step
too small or too large) each fail a pin.
"""
import math

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
f8 = oracle.fp8_cache


def _torch_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(x):
    return torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ------------------------------------------------------------------ value table
def _decode_pins(values):
    failed = []
    t = _torch_values()
    if not (np.array_equal(np.isnan(values), np.isnan(t)) and np.array_equal(values[~np.isnan(t)], t[~np.isnan(t)])):
        failed.append("library table")
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
            0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    if any(values[c] != v for c, v in hand.items()):
        failed.append("hand-worked codes")
    if not (np.isnan(values[0x7F]) and np.isnan(values[0xFF])):
        failed.append("NaN codes")
    return failed


def test_value_table_passes_every_pin():
    assert _decode_pins(f8.E4M3_VALUES) == []


def test_planted_bias_mistake_is_caught():
    wrong = f8.E4M3_VALUES.copy()
    normal = np.array([((c >> 3) & 0xF) != 0 for c in range(256)])
    wrong[normal] = wrong[normal] / 2.0        # exponent bias 8 instead of 7
    assert _decode_pins(wrong)


# ------------------------------------------------------------------ encoding
def _midpoints():
    v = f8.E4M3_VALUES[:0x7F]
    mid = (v[:-1] + v[1:]) / 2.0               # exact in float64
    return np.concatenate([mid, -mid])


def _encode_pins(encode):
    failed = []
    rng = np.random.default_rng(3)
    x = rng.uniform(-448.0, 448.0, 20000)
    x = np.concatenate([x, x * 2.0 ** -8, x * 2.0 ** -14, [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, -2.0 ** -10]])
    if not np.array_equal(encode(x), _torch_encode(x)):
        failed.append("random values vs library")
    mid = _midpoints()
    got = encode(mid)
    if not np.array_equal(got, _torch_encode(mid)) or np.any(got & 1):
        failed.append("midpoints go to the even code")
    codes = np.array([c for c in range(256) if not np.isnan(f8.E4M3_VALUES[c])])
    if not np.array_equal(encode(f8.E4M3_VALUES[codes]), codes):
        failed.append("round trip of every finite code")
    return failed


def test_encoding_passes_every_pin():
    assert _encode_pins(f8.e4m3_encode) == []


def _truncate(x):
    x = np.asarray(x, dtype=np.float64)
    v = f8.E4M3_VALUES[:0x7F]
    idx = np.searchsorted(v, np.abs(x), side="right") - 1
    return idx.astype(np.uint8) | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))


def _ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    v = f8.E4M3_VALUES[:0x7F]
    ax = np.abs(x)
    hi = np.minimum(np.searchsorted(v, ax, side="left"), len(v) - 1)
    lo = np.maximum(hi - 1, 0)
    pick = (v[hi] - ax) <= (ax - v[lo])
    return np.where(pick, hi, lo).astype(np.uint8) | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))


@pytest.mark.parametrize("wrong", [_truncate, _ties_away])
def test_planted_encoding_mistakes_are_caught(wrong):
    assert _encode_pins(wrong), f"{wrong.__name__} passed every pin"


def test_encoding_rejects_out_of_range():
    with pytest.raises(ValueError):
        f8.e4m3_encode([449.0])
    with pytest.raises(ValueError):
        f8.e4m3_encode([math.inf])


# ------------------------------------------------------------------ scale rule
def _brute_k(amax):
    if amax == 0:
        return 0
    k = -200
    while amax > 448.0 * 2.0 ** k:
        k += 1
    return k


def _scale_pins(rule):
    failed = []
    rng = np.random.default_rng(4)
    amaxes = list(rng.uniform(0, 10, 200)) + list(np.exp(rng.uniform(-60, 60, 200)))
    amaxes += [448.0, 449.0, 224.0, 224.5, 0.875, 0.876, 2.0 ** -20, 3.0e38, 0.0]
    for a in amaxes:
        if rule(a) != _brute_k(a):
            failed.append(f"brute force at {a!r}")
            break
    for a in amaxes:
        if a > 0 and not (224.0 < a * 2.0 ** -rule(a) <= 448.0):
            failed.append(f"range at {a!r}")
            break
    return failed


def test_scale_rule_passes_every_pin():
    assert _scale_pins(f8.scale_exponent) == []


@pytest.mark.parametrize("delta", [-1, 1])
def test_planted_scale_mistakes_are_caught(delta):
    assert _scale_pins(lambda a: f8.scale_exponent(a) + delta if a else 0)


# ------------------------------------------------------------------ rows and cache
def test_quantisation_error_bound():
    rng = np.random.default_rng(5)
    c = rng.standard_normal((50, 512)).astype(np.float32).astype(np.float64)
    c[3] = 0.0
    c[4] *= 1e-30
    c[5] *= 1e30
    codes, scales = f8.quantize_rows(c)
    deq = f8.dequantize_rows(codes, scales)
    # half an ulp of E4M3 (3 mantissa bits) relative, or half the subnormal step absolute
    bound = np.maximum(np.abs(c) * 2.0 ** -4, scales[:, None] * 2.0 ** -10)
    assert np.all(np.abs(deq - c) <= bound)
    assert np.all(codes[3] == 0) and scales[3] == 1.0
    for i in range(50):
        k = int(round(math.log2(scales[i])))
        assert scales[i] == 2.0 ** k
        if np.any(c[i] != 0):
            assert 224.0 < np.max(np.abs(c[i])) / scales[i] <= 448.0
    # the row maximum itself is always representable to 3 bits: at most one rounding
    assert np.all(np.abs(np.max(np.abs(deq), 1) - np.max(np.abs(c), 1)) <= np.max(np.abs(c), 1) * 2.0 ** -4)


def test_cache_round_trip_and_gather():
    rng = np.random.default_rng(6)
    n, pages = 150, 4
    c = rng.standard_normal((n, 512)).astype(np.float32)
    k = rng.standard_normal((n, 64)).astype(np.float32)
    c = (c.view(np.uint32) & 0xFFFF0000).view(np.float32)     # bf16-exact inputs
    k = (k.view(np.uint32) & 0xFFFF0000).view(np.float32)
    bt = np.array([[2, 0, 3]], dtype=np.int32)
    pos = np.arange(n)
    slots = oracle.slot_mapping(bt, np.zeros(n, np.int32), pos)
    rows, scales = f8.empty_cache(pages)
    rows, scales = f8.append(rows, scales, c, k, slots)
    lat, rope = f8.gather(rows, scales, bt, 0, n)
    codes, sc = f8.quantize_rows(c)
    assert np.array_equal(lat, f8.dequantize_rows(codes, sc))
    assert np.array_equal(rope, k.astype(np.float64))
    # page 1 is untouched
    assert np.all(rows[1] == 0) and np.all(scales[1] == 0)
    # bf16 bytes are little-endian bit patterns
    assert np.array_equal(f8.bytes_bf16(f8.bf16_bytes(k)), k.astype(np.float64))
    assert f8.bf16_bytes(np.array([1.0], np.float32)).tolist() == [0x80, 0x3F]


def test_fp8_decode_stays_near_the_bf16_decode():
    """The quantised cache moves attention outputs by about the E4M3 step,
    not more: a sanity bound on the whole FP8 path of the oracle."""
    rng = np.random.default_rng(7)
    n = 300
    c = rng.standard_normal((n, 512)).astype(np.float32)
    k = rng.standard_normal((n, 64)).astype(np.float32)
    bt = np.array([[0, 1, 2, 3, 4]], dtype=np.int32)
    slots = oracle.slot_mapping(bt, np.zeros(n, np.int32), np.arange(n))
    rows, scales = f8.append(*f8.empty_cache(5), c, k, slots)
    ref_cache = oracle.append(np.zeros((5, 64, 576)), c, k, slots)
    q_abs = rng.standard_normal((1, 128, 512)) * 0.5
    q_r = rng.standard_normal((1, 128, 64))
    s = 1.0 / math.sqrt(192)
    o8, l8 = f8.decode(q_abs, q_r, rows, scales, bt, [n], [1], s)
    o, l = oracle.decode(q_abs, q_r, ref_cache, bt, [n], [1], s)
    rel = np.abs(o8 - o).sum() / np.abs(o).sum()
    assert rel < 0.06, rel
    assert np.max(np.abs(l8 - l)) < 0.05
