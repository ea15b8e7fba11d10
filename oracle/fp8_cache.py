"""FP8 (E4M3) latent cache — TEST INFRASTRUCTURE ONLY.

Like the rest of ``oracle/`` this module may be imported only by the tests,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``; it shares no
code with the CUDA path and imports nothing from the product.

Sources:

* [P3] bjbfmj.com/news/60700 — its KV-byte formula counts only the latent and
  RoPE elements and says in so many words that quantisation scale factors,
  alignment and page tables come on top: a quantised cache stores a scale
  beside the codes.
* [P1] "撕开 DeepSeek MLA 源码…" (sheratonhq.com/news/189140), opening
  section and §5 — a quantised gather of the latent cache with 16-byte
  vector loads, whose base and offsets must be 16-byte aligned.
* OCP 8-bit Floating Point Specification (OFP8), the E4M3 format: one sign
  bit, four exponent bits with bias 7, three mantissa bits; exponent field 0
  holds the subnormals m·2^-9; S.1111.111 is NaN; there are no infinities;
  the largest finite magnitude is 448.

Reading (the pages give no FP8 layout): each
token's 512 latent values share one power-of-two scale 2^k, k the smallest
integer with max|c| <= 448·2^k (k = 0 for an all-zero row); the codes are
c·2^-k rounded to the nearest E4M3 value, ties to the even code.  Because the
scale is a power of two, c·2^-k is exact, so the rounding decision is the
same in any binary precision.  The 64 RoPE dims stay bf16.

Cache layout: ``rows`` uint8 [num_pages, 64, 640] (bytes 0..511 the codes,
bytes 512..639 the 64 bf16 RoPE values, little-endian) and ``scales``
float [num_pages, 64] (2^k per token).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

from . import mla_oracle

E4M3_MAX = 448.0
ROW_BYTES = 640          # 512 codes + 64 bf16 RoPE values
LATENT = 512


def e4m3_value(code: int) -> float:
    """Real value of one E4M3 code (OFP8 definition); NaN for S.1111.111."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_VALUES = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
_NONNEG = E4M3_VALUES[:0x7F]          # codes 0x00..0x7E: 0 .. 448, strictly increasing


def e4m3_encode(x) -> np.ndarray:
    """Round each finite |x| <= 448 to the nearest E4M3 code, ties to the even
    code; the sign bit is the sign of x (so -0.0 and negative values that
    round to zero give 0x80).  Returns uint8 codes."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)) or np.any(np.abs(x) > E4M3_MAX):
        raise ValueError("E4M3 encoding needs finite values with |x| <= 448")
    ax = np.abs(x)
    hi = np.searchsorted(_NONNEG, ax, side="left")          # first code with value >= |x|
    hi = np.minimum(hi, len(_NONNEG) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = ax - _NONNEG[lo]
    d_hi = _NONNEG[hi] - ax
    exact = _NONNEG[hi] == ax
    pick_hi = exact | (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_VALUES[np.asarray(codes, dtype=np.int64)]


def scale_exponent(amax: float) -> int:
    """Smallest integer k with amax <= 448·2^k (0 for amax == 0).

    With amax = f·2^e, f in [0.5, 1) (frexp) and 448 = 0.875·2^9:
    k = e - 9 when f <= 0.875, else e - 8.
    """
    amax = float(amax)
    if amax == 0.0:
        return 0
    f, e = math.frexp(amax)
    return e - 9 if f <= 0.875 else e - 8


def quantize_rows(c_kv: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-token quantisation of the latent rows: (codes uint8 [n, 512], scales [n] = 2^k)."""
    c = np.asarray(c_kv, dtype=np.float64)
    n = c.shape[0]
    codes = np.zeros((n, c.shape[1]), dtype=np.uint8)
    scales = np.ones(n, dtype=np.float64)
    for i in range(n):
        k = scale_exponent(np.max(np.abs(c[i])) if c.shape[1] else 0.0)
        codes[i] = e4m3_encode(np.ldexp(c[i], -k))
        scales[i] = math.ldexp(1.0, k)
    return codes, scales


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def bf16_bytes(x: np.ndarray) -> np.ndarray:
    """Little-endian bytes of bf16-exact float32 values ([..., d] -> uint8 [..., 2d])."""
    u = (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype("<u2")
    return u.view(np.uint8).reshape(*u.shape[:-1], 2 * u.shape[-1])


def bytes_bf16(b: np.ndarray) -> np.ndarray:
    """Inverse of bf16_bytes: uint8 [..., 2d] -> float64 [..., d]."""
    u = np.ascontiguousarray(b, dtype=np.uint8).view("<u2").astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def empty_cache(num_pages: int, page: int = mla_oracle.PAGE) -> Tuple[np.ndarray, np.ndarray]:
    return np.zeros((num_pages, page, ROW_BYTES), dtype=np.uint8), np.zeros((num_pages, page), dtype=np.float64)


def append(rows: np.ndarray, scales: np.ndarray, c_kv_new: np.ndarray, k_r_new: np.ndarray,
           slots: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Quantise each new token and store [codes | k_R bf16] and its scale at its slot
    (the FP8 counterpart of step A1).  Returns copies."""
    rows = np.array(rows, copy=True)
    scales = np.array(scales, dtype=np.float64, copy=True)
    flat = rows.reshape(-1, rows.shape[-1])
    fs = scales.reshape(-1)
    codes, sc = quantize_rows(c_kv_new)
    slots = np.asarray(slots, dtype=np.int64)
    flat[slots, :LATENT] = codes
    flat[slots, LATENT:] = bf16_bytes(k_r_new)
    fs[slots] = sc
    return rows, scales


def dequantize_cache(rows: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 [num_pages, 64, 576]: code·2^k latent, then the bf16 RoPE key."""
    lat = dequantize_rows(rows[..., :LATENT], scales)
    rope = bytes_bf16(rows[..., LATENT:])
    return np.concatenate([lat, rope], axis=-1)


def gather(rows: np.ndarray, scales: np.ndarray, block_table: np.ndarray, b: int, n: int):
    """The first n tokens of sequence b, dequantised: (c_KV [n, 512], k_R [n, 64]) float64."""
    return mla_oracle.gather(dequantize_cache(rows, scales), block_table, b, n)


def decode(q_abs: np.ndarray, q_r: np.ndarray, rows: np.ndarray, scales: np.ndarray,
           block_table: np.ndarray, seq_lens: Sequence[int], q_lens: Sequence[int], scale: float,
           rows_wanted: Optional[Iterable[int]] = None):
    """Absorbed paged attention (steps A3 + A4) over the dequantised FP8 cache."""
    cache = dequantize_cache(rows, scales)
    return mla_oracle.decode(q_abs, q_r, cache, block_table, seq_lens, q_lens, scale, rows=rows_wanted)
