"""Seeded synthetic inputs for absorbed paged MLA decode.

This module only draws random numbers, rounds them to bf16 and lays out the
page pool; it holds none of the attention arithmetic.  Both the CUDA path and
the CPU oracle consume exactly the arrays produced here.

Shapes follow the MLA dimensions of the DeepSeek MLA teardown page
(sheratonhq.com/news/189140, §1 and the ``mla_config.h`` constants of §3):
128 heads, content head dim 128, latent 512, decoupled RoPE key 64, pages of
64 tokens.

Draw order (one ``numpy.random.Generator(PCG64(seed))`` per case):
context lengths (only when drawn), q_c, q_R, c_KV, k_R, W_UK, W_UV, the page
permutation, then the optional stand-alone q_abs used to test the decode step
in isolation.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

H = 128          # query heads
D_HC = 128       # content head dim
D_C = 512        # latent dim
D_R = 64         # decoupled RoPE key dim
D_QK = D_C + D_R  # 576 elements per cached token
PAGE = 64        # tokens per page


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even); returns float32.

    In uint32 arithmetic: for finite inputs u + 0x8000 cannot wrap.
    """
    x = np.array(x, dtype=np.float32, copy=True, order="C")
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u &= np.uint32(0xFFFF0000)
    return x


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return bf16_round(v)


@dataclass
class Case:
    """One synthetic decode problem.

    Every floating array is float32 holding bf16-exact values.
    Sequence b owns the rows [tok_off[b], tok_off[b] + seq_lens[b]) of
    ``c_kv``/``k_r``, in position order.  The last
    ``q_lens[b]`` of them are the tokens appended in this step.
    """
    name: str
    seq_lens: np.ndarray          # int32 [B], tokens in the cache after this step's append
    q_lens: np.ndarray            # int32 [B], query tokens per sequence (>= 0)
    q_c: np.ndarray               # [T, H, D_HC]
    q_r: np.ndarray               # [T, H, D_R]
    c_kv: np.ndarray              # [sum(seq_lens), D_C]
    k_r: np.ndarray               # [sum(seq_lens), D_R]
    w_uk: Optional[np.ndarray]    # [H, D_HC, D_C]
    w_uv: Optional[np.ndarray]    # [H, D_C, D_HC]
    block_table: np.ndarray       # int32 [B, max_pages], -1 past each sequence's pages
    num_pages: int
    q_abs: Optional[np.ndarray] = None   # [T, H, D_C], stand-alone decode input
    seed: int = 0
    meta: Dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.q_lens.sum())

    @property
    def tok_off(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens.astype(np.int64))]).astype(np.int64)

    @property
    def q_start(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens.astype(np.int64))]).astype(np.int64)

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def new_token_index(self) -> np.ndarray:
        """Rows of c_kv/k_r appended in this step, in query order (length T)."""
        out = []
        off = self.tok_off
        for b in range(self.B):
            n, q = int(self.seq_lens[b]), int(self.q_lens[b])
            out.extend(range(int(off[b]) + n - q, int(off[b]) + n))
        return np.asarray(out, dtype=np.int64)

    def query_positions(self) -> np.ndarray:
        """Position of each query row's token in its sequence (int32 [T])."""
        out = [np.arange(int(n) - int(q), int(n), dtype=np.int32) for n, q in zip(self.seq_lens, self.q_lens)]
        return np.concatenate(out) if out else np.zeros(0, np.int32)

    def positions(self) -> tuple:
        """(seq_ids, positions) of every cached token, in c_kv row order."""
        seq = np.repeat(np.arange(self.B, dtype=np.int32), self.seq_lens)
        pos = np.concatenate([np.arange(n, dtype=np.int32) for n in self.seq_lens]) if self.B else np.zeros(0, np.int32)
        return seq, pos


def pages_for(n_tokens: int) -> int:
    return (int(n_tokens) + PAGE - 1) // PAGE


def make_case(seq_lens: Sequence[int], q_lens: Sequence[int], seed: int = 0,
              page_order: str = "random", with_weights: bool = True,
              with_q_abs: bool = False, name: str = "custom",
              draw_lens: Optional[tuple] = None, extra_pages: int = 0) -> Case:
    """Build a case.

    ``draw_lens=(B, lo, hi)`` draws B context lengths uniformly from the closed
    range [lo, hi] first (then ``seq_lens`` is ignored and q_lens must be a
    single broadcast value).  ``extra_pages`` adds unused pages to the pool.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if draw_lens is not None:
        B, lo, hi = draw_lens
        seq_lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
        q_lens = np.full(B, int(q_lens[0]), dtype=np.int32)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    if seq_lens.shape != q_lens.shape:
        raise ValueError("seq_lens and q_lens differ in length")
    if np.any(seq_lens < 1) or np.any(q_lens < 0) or np.any(q_lens > seq_lens):
        raise ValueError("need seq_len >= 1 and 0 <= q_len <= seq_len")
    B = seq_lens.shape[0]
    T = int(q_lens.sum())
    total = int(seq_lens.astype(np.int64).sum())

    q_c = _normal_bf16(rng, (T, H, D_HC))
    q_r = _normal_bf16(rng, (T, H, D_R))
    c_kv = _normal_bf16(rng, (total, D_C))
    k_r = _normal_bf16(rng, (total, D_R))
    w_uk = w_uv = None
    if with_weights:
        std = float(np.sqrt(1.0 / 512.0))
        w_uk = _normal_bf16(rng, (H, D_HC, D_C), std)
        w_uv = _normal_bf16(rng, (H, D_C, D_HC), std)

    npages = [pages_for(n) for n in seq_lens]
    num_pages = int(sum(npages)) + int(extra_pages)
    # the permutation is always drawn so later draws do not depend on the order
    perm = rng.permutation(num_pages).astype(np.int32)
    if page_order == "identity":
        perm = np.arange(num_pages, dtype=np.int32)
    elif page_order != "random":
        raise ValueError(page_order)
    max_pages = max(npages) if B else 1
    block_table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        block_table[b, :npages[b]] = perm[k:k + npages[b]]
        k += npages[b]

    q_abs = _normal_bf16(rng, (T, H, D_C), 0.5) if with_q_abs else None
    return Case(name=name, seq_lens=seq_lens, q_lens=q_lens, q_c=q_c, q_r=q_r,
                c_kv=c_kv, k_r=k_r, w_uk=w_uk, w_uv=w_uv, block_table=block_table,
                num_pages=num_pages, q_abs=q_abs, seed=seed)


# The five workloads the method is measured on.  Sequence lengths count the
# tokens in the cache after this step's append (cached context + query tokens
# for the MTP and chunked-prefill shapes).
WORKLOADS = {
    0: dict(name="decode_b1_ctx1024", seq_lens=[1024], q_lens=[1], page_order="identity"),
    1: dict(name="decode_b16_ctx1k_4k_ragged", draw_lens=(16, 1024, 4096), q_lens=[1]),
    2: dict(name="mtp2_decode_b64_ctx8k", seq_lens=[8192 + 2] * 64, q_lens=[2] * 64),
    3: dict(name="decode_b16_ctx64k", seq_lens=[65536] * 16, q_lens=[1] * 16),
    4: dict(name="chunked_prefill_b4_chunk512_after16k", seq_lens=[16384 + 512] * 4, q_lens=[512] * 4),
}


def workload(idx: int, seed: int = 0, with_q_abs: bool = False, with_weights: bool = True,
             batch: Optional[int] = None) -> Case:
    """Workload ``idx``; ``batch`` keeps only its first sequences (a smaller
    case of the same shape, e.g. for profiler captures)."""
    w = dict(WORKLOADS[idx])
    name = w.pop("name")
    if batch is not None:
        name = f"{name}_first{batch}"
        if "draw_lens" in w:
            B, lo, hi = w["draw_lens"]
            w["draw_lens"] = (min(B, batch), lo, hi)
        else:
            w["seq_lens"] = w["seq_lens"][:batch]
            w["q_lens"] = w["q_lens"][:batch]
    page_order = w.pop("page_order", "random")
    if "draw_lens" in w:
        return make_case(seq_lens=[], q_lens=w["q_lens"], seed=seed, page_order=page_order,
                         with_weights=with_weights, with_q_abs=with_q_abs, name=name,
                         draw_lens=w["draw_lens"])
    return make_case(w["seq_lens"], w["q_lens"], seed=seed, page_order=page_order,
                     with_weights=with_weights, with_q_abs=with_q_abs, name=name)

