"""Pins for the oracle's NVFP4 latent cache (E2M1 elements, E4M3 block scales
per 16 elements, an fp32 tensor scale).

The element format and the 16-element blocks follow NVIDIA's published NVFP4
definition; the pages ([P1] opening section and §5) only name an NVFP4
gather with 16-byte loads.  Pins that do not depend on the oracle's code:

* the 16 E2M1 values, worked by hand from the bit layout;
* encoding against a brute-force nearest-value search (ties to the even
  code, saturation at 6) over random values and every midpoint;
* E4M3 saturation of block scales against PyTorch's float8_e4m3fn
  conversion of the clipped value;
* exact round trips for blocks built from representable values, and the
  block maximum always landing on magnitude 6 (or 4 at a rounding edge);
* a quantisation error bound, nibble order, and the cache round trip.

Planted mistakes (truncation, ties away from zero, 32-element blocks, a
block scale that ignores the tensor scale, swapped nibbles) each fail a pin.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
n4 = oracle.nvfp4_cache
f8 = oracle.fp8_cache

HAND = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _brute_e2m1(x):
    out = []
    for v in np.asarray(x, dtype=np.float64):
        a = min(abs(v), 6.0)
        d = [abs(a - m) for m in HAND]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        code = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        out.append(code | (8 if np.signbit(v) else 0))
    return np.array(out, dtype=np.uint8)


def test_e2m1_values_by_hand():
    assert list(n4.E2M1_VALUES[:8]) == HAND
    assert list(n4.E2M1_VALUES[8:]) == [-v for v in HAND]
    assert np.signbit(n4.E2M1_VALUES[8])


def _encode_pins(encode):
    failed = []
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.uniform(-8, 8, 5000), rng.uniform(-1, 1, 2000), [0.0, -0.0, 6.0, -6.0, 100.0, -7.0]])
    if not np.array_equal(encode(x), _brute_e2m1(x)):
        failed.append("random values vs brute force")
    v = np.array(HAND)
    mid = np.concatenate([(v[:-1] + v[1:]) / 2, -(v[:-1] + v[1:]) / 2])
    if not np.array_equal(encode(mid), _brute_e2m1(mid)):
        failed.append("midpoints")
    return failed


def test_encoding_passes_every_pin():
    assert _encode_pins(n4.e2m1_encode) == []


def _truncate(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    idx = np.searchsorted(np.array(HAND), a, side="right") - 1
    return idx.astype(np.uint8) | np.where(np.signbit(x), np.uint8(8), np.uint8(0))


def _ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    h = np.array(HAND)
    hi = np.minimum(np.searchsorted(h, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    pick = (h[hi] - a) <= (a - h[lo])
    return np.where(pick, hi, lo).astype(np.uint8) | np.where(np.signbit(x), np.uint8(8), np.uint8(0))


@pytest.mark.parametrize("wrong", [_truncate, _ties_away])
def test_planted_encoding_mistakes_are_caught(wrong):
    assert _encode_pins(wrong)


def test_block_scale_saturates_like_the_library():
    x = np.array([0.001, 1.0, 447.0, 448.0, 460.0, 1e6])
    clipped = np.minimum(x, 448.0)
    want = torch.tensor(clipped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(n4.e4m3_encode_sat(x), want)


def _block_pins(quantize, dequantize, pack=n4.pack_codes):
    failed = []
    st = 2.0 ** -8
    rng = np.random.default_rng(12)
    # representable blocks: e2m1 values times a representable block scale whose 6x is the block max
    codes = rng.integers(0, 16, size=(3, 512)).astype(np.uint8)
    codes[:, ::16] = 7                           # every block holds +6, so amax = 6 * s_b * s_t
    sb_codes = rng.choice([0x30, 0x38, 0x44, 0x50, 0x5C], size=(3, 32)).astype(np.uint8)
    sb = f8.e4m3_decode(sb_codes)
    x = (n4.E2M1_VALUES[codes].reshape(3, 32, 16) * sb[:, :, None] * st).reshape(3, 512)
    c2, s2 = quantize(x, st)
    if not (np.array_equal(c2, codes) and np.array_equal(s2, sb_codes)):
        failed.append("representable round trip")
    if not np.array_equal(dequantize(c2, s2, st), x):
        failed.append("exact dequantisation")
    # random rows: the block max lands on magnitude 6 (4 only when the scale rounded up a lot)
    c = _bf16(rng.standard_normal((20, 512)))
    cc, ss = quantize(c, st)
    blocks = c.reshape(20, 32, 16)
    arg = np.argmax(np.abs(blocks), axis=2)
    top = np.take_along_axis(cc.reshape(20, 32, 16), arg[:, :, None], 2)[:, :, 0] & 7
    if not np.all(top >= 6):
        failed.append("block maximum maps to 6")
    d = dequantize(cc, ss, st)
    sbv = f8.e4m3_decode(ss)[:, :, None] * st
    amax = np.max(np.abs(blocks), axis=2)[:, :, None]
    bound = 0.25 * np.abs(blocks) + 0.25 * sbv + amax * 2.0 ** -4 + np.abs(blocks) * 2.0 ** -8
    if not np.all(np.abs(d.reshape(20, 32, 16) - blocks) <= bound):
        failed.append("error bound")
    # nibble order: element 2i in the low nibble
    p = pack(np.array([[1, 2] + [0] * 510], dtype=np.uint8))
    if p[0, 0] != 0x21:
        failed.append("nibble order")
    return failed


def test_quantisation_passes_every_pin():
    assert _block_pins(n4.quantize_rows, n4.dequantize_rows) == []


def _blocks32(c, st):
    c = np.asarray(c, dtype=np.float32)
    n = c.shape[0]
    big = c.reshape(n, 16, 32)
    amax = np.repeat(np.max(np.abs(big), axis=2), 2, axis=1).reshape(n, 32)
    t = (amax / np.float32(6 * np.float32(st))).astype(np.float64)
    sb_code = n4.e4m3_encode_sat(t)
    sb = f8.e4m3_decode(sb_code).astype(np.float32)
    q = c.reshape(n, 32, 16) / (sb * np.float32(st))[:, :, None]
    return n4.e2m1_encode(np.nan_to_num(q).astype(np.float64)).reshape(n, 512), sb_code


def _no_tensor_scale_in_codes(c, st):
    c = np.asarray(c, dtype=np.float32)
    n = c.shape[0]
    blocks = c.reshape(n, 32, 16)
    amax = np.max(np.abs(blocks), axis=2)
    sb_code = n4.e4m3_encode_sat((amax / np.float32(6 * np.float32(st))).astype(np.float64))
    sb = f8.e4m3_decode(sb_code).astype(np.float32)
    q = blocks / sb[:, :, None]
    return n4.e2m1_encode(np.nan_to_num(q).astype(np.float64)).reshape(n, 512), sb_code


def _swapped_pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 1::2] | (codes[:, 0::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("case", ["blocks32", "no_tensor_scale", "swapped_pack"])
def test_planted_block_mistakes_are_caught(case):
    if case == "blocks32":
        failed = _block_pins(_blocks32, n4.dequantize_rows)
    elif case == "no_tensor_scale":
        failed = _block_pins(_no_tensor_scale_in_codes, n4.dequantize_rows)
    else:
        failed = _block_pins(n4.quantize_rows, n4.dequantize_rows, pack=_swapped_pack)
    assert failed


def test_cache_round_trip_and_gather():
    rng = np.random.default_rng(13)
    n, st = 130, 2.0 ** -8
    c = _bf16(rng.standard_normal((n, 512)))
    k = _bf16(rng.standard_normal((n, 64)))
    bt = np.array([[3, 1, 0]], dtype=np.int32)
    slots = oracle.slot_mapping(bt, np.zeros(n, np.int32), np.arange(n))
    rows = n4.append(n4.empty_cache(4), c, k, slots, st)
    assert rows.shape == (4, 64, 416)
    lat, rope = n4.gather(rows, bt, 0, n, st)
    codes, sb = n4.quantize_rows(c, st)
    assert np.array_equal(lat, n4.dequantize_rows(codes, sb, st))
    assert np.array_equal(rope, k.astype(np.float64))
    assert np.all(rows[2] == 0)
    assert np.array_equal(n4.unpack_codes(n4.pack_codes(codes)), codes)
    # an all-zero block has a zero scale and zero codes
    z = np.zeros((1, 512), np.float32)
    cz, sz = n4.quantize_rows(z, st)
    assert np.all(cz == 0) and np.all(sz == 0)
