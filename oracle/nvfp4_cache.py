"""NVFP4 latent cache (E2M1 codes, E4M3 block scales) — TEST INFRASTRUCTURE ONLY.

Like the rest of ``oracle/`` this module may be imported only by the tests,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``; it shares no
code with the CUDA path and imports nothing from the product.

Sources:

* [P1] "撕开 DeepSeek MLA 源码…" (sheratonhq.com/news/189140), opening
  section and §5: the latent cache is gathered in NVFP4 with 16-byte vector
  loads; a page-table base that is not 16-byte aligned, or a byte offset
  (element offset / 2) that is not a multiple of 8, faults the load.
* [P3] bjbfmj.com/news/60700: quantisation scale factors are stored beside
  the cached elements.
* The NVFP4 format as NVIDIA publishes it: 4-bit E2M1 elements (sign, two
  exponent bits with bias 1, one mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2,
  3, 4, 6), one E4M3 scale per block of 16 elements, and one fp32 scale per
  tensor; an element's value is e2m1 * block_scale * tensor_scale.

Readings (the pages give no layout):
* the tensor scale s_t is a caller-supplied fp32 constant (an append-only
  cache cannot rescale what it already holds);
* block scale: the E4M3 rounding (nearest, ties to even, saturating at 448)
  of fp32(amax_block / fp32(6 * s_t)); codes: the E2M1 rounding (nearest,
  ties to even, saturating at 6) of fp32(x / fp32(s_b * s_t)), all zero when
  s_b is zero; every division and product is one correctly rounded fp32
  operation, in that order, so the quantised codes are fixed bit for bit;
* dequantised value: bf16(fp32(fp32(e2m1 * s_b) * s_t)), rounded to nearest
  even at each step (the first product is exact);
* the 64 RoPE values stay bf16.

Row layout (416 bytes per token, a multiple of 16): bytes 0..255 the 512
codes, two per byte, element 2i in the low nibble; bytes 256..287 the 32
block scales; bytes 288..415 the RoPE values (bf16, little-endian).
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from . import fp8_cache, mla_oracle

BLOCK = 16
LATENT = 512
CODE_BYTES = LATENT // 2          # 256
SCALE_OFF = CODE_BYTES            # 256
ROPE_OFF = SCALE_OFF + LATENT // BLOCK   # 288
ROW_BYTES = ROPE_OFF + 128        # 416
E2M1_MAX = 6.0


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * m * 0.5
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E2M1_VALUES = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_NONNEG = E2M1_VALUES[:8]         # 0, 0.5, 1, 1.5, 2, 3, 4, 6


def e2m1_encode(x) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code, magnitudes above 6 saturate
    to 6); the sign bit is the sign of x.  Returns uint8 codes 0..15."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("E2M1 encoding needs finite values")
    ax = np.minimum(np.abs(x), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_NONNEG, ax, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = ax - _NONNEG[lo]
    d_hi = _NONNEG[hi] - ax
    pick_hi = (_NONNEG[hi] == ax) | (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x8), np.uint8(0))


def e4m3_encode_sat(x) -> np.ndarray:
    """E4M3 rounding that saturates at 448 (values above 448 give 448's code)."""
    x = np.asarray(x, dtype=np.float64)
    return fp8_cache.e4m3_encode(np.clip(x, -fp8_cache.E4M3_MAX, fp8_cache.E4M3_MAX))


def quantize_rows(c_kv: np.ndarray, tensor_scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Rows [n, 512] of bf16-exact values -> (codes uint8 [n, 512] one code per
    element, block-scale codes uint8 [n, 32])."""
    c = np.asarray(c_kv, dtype=np.float32)
    n = c.shape[0]
    st = np.float32(tensor_scale)
    blocks = c.reshape(n, LATENT // BLOCK, BLOCK)
    amax = np.max(np.abs(blocks), axis=2)                          # exact (bf16 values)
    t = amax / np.float32(np.float32(6.0) * st)                    # one fp32 division
    sb_code = e4m3_encode_sat(t.astype(np.float64))
    sb = fp8_cache.e4m3_decode(sb_code).astype(np.float32)
    denom = (sb * st).astype(np.float32)                           # one fp32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blocks / denom[:, :, None]).astype(np.float32)        # one fp32 division
    q = np.where(denom[:, :, None] == 0, np.float32(0), q)
    codes = e2m1_encode(q.astype(np.float64)).reshape(n, LATENT)
    return codes, sb_code


def dequantize_rows(codes: np.ndarray, sb_code: np.ndarray, tensor_scale: float) -> np.ndarray:
    """bf16(fp32(fp32(e2m1 * s_b) * s_t)) as float64 [n, 512]."""
    n = codes.shape[0]
    v = E2M1_VALUES[np.asarray(codes, dtype=np.int64)].astype(np.float32).reshape(n, LATENT // BLOCK, BLOCK)
    sb = fp8_cache.e4m3_decode(sb_code).astype(np.float32)
    prod = (v * sb[:, :, None]).astype(np.float32)                 # exact
    val = (prod * np.float32(tensor_scale)).astype(np.float32)      # one rounding
    return _bf16_rne(val).reshape(n, LATENT).astype(np.float64)


def _bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16, nearest even (as float32)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[n, 512] codes -> [n, 256] bytes, element 2i in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def empty_cache(num_pages: int, page: int = mla_oracle.PAGE) -> np.ndarray:
    return np.zeros((num_pages, page, ROW_BYTES), dtype=np.uint8)


def append(rows: np.ndarray, c_kv_new: np.ndarray, k_r_new: np.ndarray, slots: np.ndarray,
           tensor_scale: float) -> np.ndarray:
    """Quantise each new token and store its 416-byte row at its slot (a copy)."""
    rows = np.array(rows, copy=True)
    flat = rows.reshape(-1, ROW_BYTES)
    codes, sb = quantize_rows(c_kv_new, tensor_scale)
    slots = np.asarray(slots, dtype=np.int64)
    flat[slots, :CODE_BYTES] = pack_codes(codes)
    flat[slots, SCALE_OFF:ROPE_OFF] = sb
    flat[slots, ROPE_OFF:] = fp8_cache.bf16_bytes(k_r_new)
    return rows


def dequantize_cache(rows: np.ndarray, tensor_scale: float) -> np.ndarray:
    """float64 [pages, 64, 576]: dequantised latent, then the bf16 RoPE key."""
    flat = rows.reshape(-1, ROW_BYTES)
    lat = dequantize_rows(unpack_codes(flat[:, :CODE_BYTES]), flat[:, SCALE_OFF:ROPE_OFF], tensor_scale)
    rope = fp8_cache.bytes_bf16(flat[:, ROPE_OFF:])
    return np.concatenate([lat, rope], axis=1).reshape(rows.shape[0], rows.shape[1], LATENT + 64)


def gather(rows: np.ndarray, block_table: np.ndarray, b: int, n: int, tensor_scale: float):
    """The first n tokens of sequence b, dequantised: (c_KV [n, 512], k_R [n, 64])."""
    return mla_oracle.gather(dequantize_cache(rows, tensor_scale), block_table, b, n)
