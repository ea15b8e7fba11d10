"""CPU oracle for absorbed paged MLA decode — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and
its Python binding) never imports, calls or links it, and this module imports
nothing from the product.

Everything is plain NumPy in float64: inputs are the bf16-exact float32 arrays
of the seeded generator, up-cast exactly; no intermediate is rounded.

Sources (cited by page title and section):

* [P1] "撕开 DeepSeek MLA 源码：C++ 与 TensorRT-LLM 算子设计优化全景与 TaoToken 实践"
  (sheratonhq.com/news/189140).  §1 gives the cached token (512-d latent c_KV
  plus a 64-d decoupled RoPE key k_R, 576 elements); §3 gives the dimension
  constants and page_size 64; §4 gives the numerical-equivalence script whose
  "path A" (decompress K = c_KV·W_UK, then score) and "path B" (absorb
  q_abs = q_c·W_UK, score against c_KV) and score scale (d_hc + d_r)^-1/2
  define the score.
* [P2] "DeepSeek的推理为什么比别人便宜一个数量级？——MLA、MoE、MTP技术拆解"
  (leslieaibin.github.io).  Its MLA section (compressing the KV cache to
  1/5) defines the up-projections K = c·W_UK and V = c·W_UV; its closing
  one-picture summary of the inference flow has each decode step append the
  new token's latent to the cache; its MTP section gives the two-token decode.
* [P3] bjbfmj.com/news/60700 — the KV-byte formula
  L × (d_c + d_r) × b × tokens × sequences and its calculator's checks.

Readings where the pages are silent: softmax is the exact softmax over the visible tokens (the pages print none;
online softmax and split-KV are implementations of it); a query at sequence
position p sees positions [0, p]; V is the latent itself in the absorbed path
(o_lat = P·c_KV, then out = o_lat·W_UV), which equals softmax·(c_KV·W_UV) by
associativity.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

PAGE = 64


# --------------------------------------------------------------------------
# [P3] KV-byte formula
# --------------------------------------------------------------------------
def kv_bytes(layers: int, dc: int, dr: int, element_bytes: int, tokens: int,
             sequences: int = 1) -> int:
    """Unsharded latent-cache bytes, [P3]: L × (d_c + d_r) × b × tokens × seqs.

    Non-positive layers/d_c/element_bytes/tokens/sequences or a negative d_r is
    an invalid dimension ([P3] calculator's guard).
    """
    for x in (layers, dc, element_bytes, tokens, sequences):
        if int(x) <= 0:
            raise ValueError("invalid dimension")
    if int(dr) < 0:
        raise ValueError("invalid dimension")
    return int(layers) * (int(dc) + int(dr)) * int(element_bytes) * int(tokens) * int(sequences)


def gib(nbytes: int) -> Fraction:
    """Bytes in binary GiB as an exact fraction ([P3]: 1 GiB = 1024**3 B)."""
    return Fraction(int(nbytes), 1024 ** 3)


# --------------------------------------------------------------------------
# Paged cache: placement (step A1) and gather
# --------------------------------------------------------------------------
def slot_mapping(block_table: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray,
                 page_size: int = PAGE) -> np.ndarray:
    """Physical slot of token (b, pos): block_table[b][pos // page] * page + pos % page.

    Pages of ``page_size`` tokens ([P1] §3 plugin config, page_size 64).
    """
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    out = np.empty(seq_ids.shape[0], dtype=np.int64)
    for i in range(seq_ids.shape[0]):
        b, p = int(seq_ids[i]), int(positions[i])
        out[i] = int(block_table[b, p // page_size]) * page_size + p % page_size
    return out


def append(kv_cache: np.ndarray, c_kv_new: np.ndarray, k_r_new: np.ndarray,
           slots: np.ndarray) -> np.ndarray:
    """Store each new token's [c_KV | k_R] row at its slot ([P2] one-picture summary of
    the inference flow: after each step the new latent joins the cache).  Returns a copy.

    ``kv_cache`` is [num_pages, page, 576]; slots index its flattened rows.
    """
    out = np.array(kv_cache, copy=True)
    flat = out.reshape(-1, out.shape[-1])
    dc = c_kv_new.shape[1]
    slots = np.asarray(slots, dtype=np.int64)
    flat[slots, :dc] = c_kv_new
    flat[slots, dc:] = k_r_new
    return out


def gather(kv_cache: np.ndarray, block_table: np.ndarray, b: int, n: int,
           dc: int = 512) -> Tuple[np.ndarray, np.ndarray]:
    """The first ``n`` cached tokens of sequence b, in position order.

    Returns (c_KV [n, dc], k_R [n, dr]) exactly as stored (integer indexing only).
    """
    page = kv_cache.shape[1]
    npages = (int(n) + page - 1) // page
    pages = np.asarray(block_table[b, :npages], dtype=np.int64)
    rows = kv_cache[pages].reshape(npages * page, kv_cache.shape[2])[:n]
    return rows[:, :dc], rows[:, dc:]


# --------------------------------------------------------------------------
# Steps A2, A3, A5
# --------------------------------------------------------------------------
def absorb_q(q_c: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """[P1] §4 path B: q_abs[t, h, c] = Σ_d q_c[t, h, d] · W_UK[h, d, c].

    One query row at a time (per head, a vector times W_UK[h]), so a row's
    value does not depend on which other rows are computed with it."""
    q = np.asarray(q_c, dtype=np.float64)
    w = np.asarray(w_uk, dtype=np.float64)
    out = np.empty((q.shape[0], q.shape[1], w.shape[2]), dtype=np.float64)
    for t in range(q.shape[0]):
        out[t] = np.matmul(q[t][:, None, :], w)[:, 0, :]
    return out


def up_v(o_lat: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """out[t, h, d] = Σ_c o_lat[t, h, c] · W_UV[h, c, d] ([P2] V = c·W_UV, absorbed
    into the output by associativity).  One query row at a time, like absorb_q."""
    o = np.asarray(o_lat, dtype=np.float64)
    w = np.asarray(w_uv, dtype=np.float64)
    out = np.empty((o.shape[0], o.shape[1], w.shape[2]), dtype=np.float64)
    for t in range(o.shape[0]):
        out[t] = np.matmul(o[t][:, None, :], w)[:, 0, :]
    return out


def scores(q_abs_row: np.ndarray, q_r_row: np.ndarray, c_kv: np.ndarray,
           k_r: np.ndarray, scale: float) -> np.ndarray:
    """[P1] §4 path B score: s[h, j] = (q_abs[h]·c_KV[j] + q_R[h]·k_R[j]) · scale."""
    qa = np.asarray(q_abs_row, dtype=np.float64)
    qr = np.asarray(q_r_row, dtype=np.float64)
    c = np.asarray(c_kv, dtype=np.float64)
    k = np.asarray(k_r, dtype=np.float64)
    return (qa @ c.T + qr @ k.T) * scale


def softmax_lse(s: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Exact softmax over the last axis and its natural log-sum-exp."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def default_scale(d_hc: int = 128, d_r: int = 64) -> float:
    """[P1] §4: scale = 1 / sqrt(d_hc + d_r)."""
    return 1.0 / math.sqrt(d_hc + d_r)


def visible_tokens(seq_len: int, q_len: int, i: int) -> int:
    """Tokens seen by query i of a sequence whose cache holds ``seq_len`` tokens
    after appending its ``q_len`` query tokens: the query sits at position
    seq_len - q_len + i and sees positions [0, that position]."""
    return int(seq_len) - int(q_len) + int(i) + 1


def attention_row(q_abs_row, q_r_row, c_kv, k_r, scale):
    """One query token, all heads: (o_lat [H, dc], lse [H]) over the given tokens."""
    s = scores(q_abs_row, q_r_row, c_kv, k_r, scale)
    p, lse = softmax_lse(s)
    return p @ np.asarray(c_kv, dtype=np.float64), lse


def row_index(seq_lens: Sequence[int], q_lens: Sequence[int]) -> List[Tuple[int, int, int]]:
    """(row t, sequence b, query index i) for every query token, in row order."""
    out, t = [], 0
    for b, q in enumerate(q_lens):
        for i in range(int(q)):
            out.append((t, b, i))
            t += 1
    return out


def decode(q_abs: np.ndarray, q_r: np.ndarray, kv_cache: np.ndarray, block_table: np.ndarray,
           seq_lens: Sequence[int], q_lens: Sequence[int], scale: float,
           rows: Optional[Iterable[int]] = None, dc: int = 512):
    """Step A3 (+A4): absorbed paged attention.

    Returns (o_lat [T, H, dc], lse [T, H]) as float64; rows not requested stay NaN.
    """
    T, Hn = q_abs.shape[0], q_abs.shape[1]
    o = np.full((T, Hn, dc), np.nan)
    lse = np.full((T, Hn), np.nan)
    want = None if rows is None else set(int(r) for r in rows)
    for t, b, i in row_index(seq_lens, q_lens):
        if want is not None and t not in want:
            continue
        n = visible_tokens(seq_lens[b], q_lens[b], i)
        c, k = gather(kv_cache, block_table, b, n, dc)
        o[t], lse[t] = attention_row(q_abs[t], q_r[t], c, k, scale)
    return o, lse


def mla_step(q_c, q_r, w_uk, w_uv, kv_cache, block_table, seq_lens, q_lens, scale,
             rows=None, dc: int = 512):
    """A2 → A3/A4 → A5 without rounding any intermediate.

    Returns dict with q_abs, o_lat, lse, out (float64; unrequested rows NaN).
    """
    if rows is None:
        qa = absorb_q(q_c, w_uk)
    else:
        qa = np.full((q_c.shape[0], q_c.shape[1], w_uk.shape[2]), np.nan)
        idx = sorted(int(r) for r in rows)
        qa[idx] = absorb_q(q_c[idx], w_uk)
    o, lse = decode(qa, q_r, kv_cache, block_table, seq_lens, q_lens, scale, rows, dc)
    if rows is None:
        out = up_v(o, w_uv)
    else:
        # only the requested rows are up-projected; the others stay NaN
        out = np.full((o.shape[0], o.shape[1], w_uv.shape[2]), np.nan)
        out[idx] = up_v(o[idx], w_uv)
    return dict(q_abs=qa, o_lat=o, lse=lse, out=out)


# --------------------------------------------------------------------------
# Split-KV partials and their merge (step A4)
# --------------------------------------------------------------------------
def attention_partial(q_abs_row, q_r_row, c_kv, k_r, scale):
    """Normalised output and lse over one slice of the visible tokens."""
    return attention_row(q_abs_row, q_r_row, c_kv, k_r, scale)


def combine(partials: Sequence[Tuple[np.ndarray, np.ndarray]]):
    """Merge per-slice (o_s [H, dc], lse_s [H]) into the full-sequence result:
    lse = ln Σ_s e^{lse_s};  o = Σ_s e^{lse_s - lse} o_s."""
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in partials])   # [S, H]
    m = np.max(lses, axis=0)
    w = np.exp(lses - m)
    z = np.sum(w, axis=0)
    lse = m + np.log(z)
    o = sum((w[s] / z)[:, None] * np.asarray(partials[s][0], dtype=np.float64)
            for s in range(len(partials)))
    return o, lse


# --------------------------------------------------------------------------
# [P1] §4 path A: decompress, the cross-check of absorption
# --------------------------------------------------------------------------
def naive_attention_row(q_c_row, q_r_row, c_kv, k_r, w_uk, w_uv, scale):
    """Decompress then attend, per head h:
    K_h = c_KV·W_UK[h]^T  ([n, d_hc]),  V_h = c_KV·W_UV[h]  ([n, d_hc]),
    s = (q_c[h]·K_h^T + q_R[h]·k_R^T)·scale,  out_h = softmax(s)·V_h.

    Returns (out [H, d_hc], lse [H]).
    """
    c = np.asarray(c_kv, dtype=np.float64)
    k = np.asarray(k_r, dtype=np.float64)
    Hn = q_c_row.shape[0]
    out = np.empty((Hn, w_uv.shape[2]))
    lse = np.empty(Hn)
    for h in range(Hn):
        K_h = c @ np.asarray(w_uk[h], dtype=np.float64).T
        V_h = c @ np.asarray(w_uv[h], dtype=np.float64)
        s = (K_h @ np.asarray(q_c_row[h], dtype=np.float64)
             + k @ np.asarray(q_r_row[h], dtype=np.float64)) * scale
        p, l = softmax_lse(s[None, :])
        out[h] = p[0] @ V_h
        lse[h] = l[0]
    return out, lse


def expand_kv(c_kv: np.ndarray, w_uk: np.ndarray, w_uv: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """[P1] §4 path A expansion, every head at once:
    K_c[t, h, d] = Σ_c c_KV[t, c]·W_UK[h, d, c],  V_c[t, h, e] = Σ_c c_KV[t, c]·W_UV[h, c, e]."""
    c = np.asarray(c_kv, dtype=np.float64)
    k = np.einsum("tc,hdc->thd", c, np.asarray(w_uk, dtype=np.float64))
    v = np.einsum("tc,hce->the", c, np.asarray(w_uv, dtype=np.float64))
    return k, v


def naive_scores(q_c_row, q_r_row, c_kv, k_r, w_uk, scale):
    """[P1] §4 path A scores [H, n]."""
    c = np.asarray(c_kv, dtype=np.float64)
    k = np.asarray(k_r, dtype=np.float64)
    s = np.empty((q_c_row.shape[0], c.shape[0]))
    for h in range(q_c_row.shape[0]):
        K_h = c @ np.asarray(w_uk[h], dtype=np.float64).T
        s[h] = (K_h @ np.asarray(q_c_row[h], dtype=np.float64)
                + k @ np.asarray(q_r_row[h], dtype=np.float64)) * scale
    return s


def absorbed_scores(q_c_row, q_r_row, c_kv, k_r, w_uk, scale):
    """[P1] §4 path B scores [H, n]."""
    qa = absorb_q(np.asarray(q_c_row)[None], w_uk)[0]
    return scores(qa, q_r_row, c_kv, k_r, scale)


# --------------------------------------------------------------------------
# Decoupled RoPE in fp32 ([P1] §1, §3, §4)
# --------------------------------------------------------------------------
# [P1] §1: the 64-d shared RoPE vector carries the position, apart from the
# 512-d latent.  [P1] §3's plugin settings fix the RoPE compute dtype to fp32,
# and [P1] §4 traces a failed equivalence check to RoPE computed in fp16
# (phase error), fixed by generating the precomputed RoPE table in fp32 and
# multiply-adding in fp32.  The pages print no rotation formula; the reading
# used here is the standard rotary embedding:
# consecutive pairs (x[2i], x[2i+1]), i < d/2, rotated by the angle
# p * base^(-2i/d) with base 10000.
ROPE_BASE = 10000.0


def rope_angles(positions, dim: int = 64, base: float = ROPE_BASE) -> np.ndarray:
    """Angle of pair i at position p: p * base^(-2i/dim), float64 [..., dim/2]."""
    p = np.asarray(positions, dtype=np.float64)[..., None]
    inv = base ** (-2.0 * np.arange(dim // 2, dtype=np.float64) / dim)
    return p * inv


def rope_table(max_pos: int, dim: int = 64, base: float = ROPE_BASE) -> np.ndarray:
    """cos/sin of every position's angles, float64 [max_pos, dim/2, 2]."""
    a = rope_angles(np.arange(max_pos), dim, base)
    return np.stack([np.cos(a), np.sin(a)], axis=-1)


def rope_apply(x: np.ndarray, positions, dim: int = 64, base: float = ROPE_BASE) -> np.ndarray:
    """Rotate each pair (x[2i], x[2i+1]) of the last axis by its angle at the
    broadcast position; float64.  x: [..., dim]; positions broadcast against
    x's leading axes."""
    x = np.asarray(x, dtype=np.float64)
    a = rope_angles(positions, dim, base)
    c, s = np.cos(a), np.sin(a)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out
