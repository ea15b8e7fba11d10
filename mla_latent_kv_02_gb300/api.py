"""Python binding of the C ABI (include/mla.h), same names, torch tensors in.

Only argument marshalling happens here: shapes, dtypes and devices are
checked, raw pointers and the current CUDA stream are passed to libmla, and a
non-zero status raises :class:`MlaError`.  Every step of the path runs in the
library's CUDA kernels.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from ._lib import lib, mla_plan_info

H, D_HC, D_C, D_R, PAGE = 128, 128, 512, 64, 64
D_QK = D_C + D_R

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_MISALIGNED", 3: "MLA_ERR_UNSUPPORTED",
          4: "MLA_ERR_CUDA", 5: "MLA_ERR_DEVICE", 6: "MLA_ERR_TIMEOUT", 7: "MLA_ERR_NO_SPACE"}
DEVERR_PAGE_OOB, DEVERR_SLOT_OOB, DEVERR_TIMEOUT, DEVERR_PLAN, DEVERR_POS_OOB, DEVERR_FP8_RANGE = 1, 2, 4, 8, 16, 32
DEVERR_BATCH = 64


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != 0:
        raise MlaError(status, lib().mla_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None, cuda: bool = True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


# ------------------------------------------------------------------ host-only calls
def mla_version() -> int:
    return int(lib().mla_version())


def mla_config_default():
    return lib().mla_config_default()


def mla_kv_bytes(layers: int, dc: int, dr: int, elem_bytes: int, tokens: int, seqs: int = 1) -> int:
    out = C.c_uint64()
    _check(lib().mla_kv_bytes(layers, dc, dr, elem_bytes, tokens, seqs, C.byref(out)))
    return int(out.value)


class MlaPool:
    """Host page pool (mla_pool_*)."""

    def __init__(self, num_pages: int):
        self._h = C.c_void_p()
        _check(lib().mla_pool_create(int(num_pages), C.byref(self._h)))

    def alloc(self, n: int) -> np.ndarray:
        ids = np.zeros(max(n, 1), dtype=np.int32)
        _check(lib().mla_pool_alloc(self._h, int(n), ids.ctypes.data_as(C.POINTER(C.c_int32))))
        return ids[:n]

    def free(self, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().mla_pool_free(self._h, ids.ctypes.data_as(C.POINTER(C.c_int32)), int(ids.size)))

    def available(self) -> int:
        out = C.c_int32()
        _check(lib().mla_pool_available(self._h, C.byref(out)))
        return int(out.value)

    def close(self) -> None:
        if self._h:
            lib().mla_pool_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mla_slot_mapping(block_table: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray) -> np.ndarray:
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sid = np.ascontiguousarray(seq_ids, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    n = int(sid.size)
    out = np.zeros(max(n, 1), dtype=np.int64)
    P32 = C.POINTER(C.c_int32)
    _check(lib().mla_slot_mapping(bt.ctypes.data_as(P32), int(bt.shape[0]), int(bt.shape[1]),
                                  sid.ctypes.data_as(P32), pos.ctypes.data_as(P32), n,
                                  out.ctypes.data_as(C.POINTER(C.c_int64))))
    return out[:n]


# ------------------------------------------------------------------ device steps
def mla_cache_init(kv_cache: torch.Tensor, stream=None) -> None:
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _check(lib().mla_cache_init(_ptr(kv_cache), kv_cache.shape[0], _stream(stream)))


def mla_kv_append(c_kv_new, k_r_new, slots, kv_cache, dev_err, stream=None) -> None:
    n = c_kv_new.shape[0]
    _need(c_kv_new, "c_kv_new", torch.bfloat16, (n, D_C))
    _need(k_r_new, "k_r_new", torch.bfloat16, (n, D_R))
    _need(slots, "slots", torch.int64, (n,))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_kv_append(_ptr(c_kv_new), _ptr(k_r_new), _ptr(slots), int(n), _ptr(kv_cache),
                               kv_cache.shape[0], _ptr(dev_err), _stream(stream)))


FP8_ROW_BYTES = 640


def mla_kv_append_fp8(c_kv_new, k_r_new, slots, rows, scales, dev_err, stream=None) -> None:
    """Quantise new tokens into the FP8 cache: rows uint8 [pages, 64, 640], scales fp32 [pages, 64]."""
    n = c_kv_new.shape[0]
    _need(c_kv_new, "c_kv_new", torch.bfloat16, (n, D_C))
    _need(k_r_new, "k_r_new", torch.bfloat16, (n, D_R))
    _need(slots, "slots", torch.int64, (n,))
    _need(rows, "rows", torch.uint8, (rows.shape[0], PAGE, FP8_ROW_BYTES))
    _need(scales, "scales", torch.float32, (rows.shape[0], PAGE))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_kv_append_fp8(_ptr(c_kv_new), _ptr(k_r_new), _ptr(slots), int(n), _ptr(rows), _ptr(scales),
                                   rows.shape[0], _ptr(dev_err), _stream(stream)))


def mla_gather_paged_fp8(rows, scales, block_table, b: int, n_tokens: int, out, dev_err, stream=None) -> None:
    _need(rows, "rows", torch.uint8, (rows.shape[0], PAGE, FP8_ROW_BYTES))
    _need(scales, "scales", torch.float32, (rows.shape[0], PAGE))
    _need(block_table, "block_table", torch.int32)
    _need(out, "out", torch.bfloat16, (n_tokens, D_QK))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_gather_paged_fp8(_ptr(rows), _ptr(scales), rows.shape[0], _ptr(block_table),
                                      block_table.shape[1], int(b), int(n_tokens), _ptr(out), _ptr(dev_err),
                                      _stream(stream)))


NVFP4_ROW_BYTES = 416


def mla_kv_append_nvfp4(c_kv_new, k_r_new, slots, rows, tensor_scale: float, dev_err, stream=None) -> None:
    """Quantise new tokens into the NVFP4 cache: rows uint8 [pages, 64, 416]."""
    n = c_kv_new.shape[0]
    _need(c_kv_new, "c_kv_new", torch.bfloat16, (n, D_C))
    _need(k_r_new, "k_r_new", torch.bfloat16, (n, D_R))
    _need(slots, "slots", torch.int64, (n,))
    _need(rows, "rows", torch.uint8, (rows.shape[0], PAGE, NVFP4_ROW_BYTES))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_kv_append_nvfp4(_ptr(c_kv_new), _ptr(k_r_new), _ptr(slots), int(n), float(tensor_scale),
                                     _ptr(rows), rows.shape[0], _ptr(dev_err), _stream(stream)))


def mla_gather_paged_nvfp4(rows, tensor_scale: float, block_table, b: int, n_tokens: int, out, dev_err,
                           stream=None) -> None:
    _need(rows, "rows", torch.uint8)
    if rows.dim() != 3 or tuple(rows.shape[1:]) != (PAGE, NVFP4_ROW_BYTES):
        raise ValueError(f"rows has shape {tuple(rows.shape)}, expected (pages, {PAGE}, {NVFP4_ROW_BYTES})")
    _need(block_table, "block_table", torch.int32)
    _need(out, "out", torch.bfloat16, (n_tokens, D_QK))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_gather_paged_nvfp4(_ptr(rows), float(tensor_scale), rows.shape[0], _ptr(block_table),
                                        block_table.shape[1], int(b), int(n_tokens), _ptr(out), _ptr(dev_err),
                                        _stream(stream)))


def mla_gather_paged_nvfp4_batch(rows, tensor_scale: float, block_table, seq_ids, out_offsets, out, dev_err,
                                 stream=None) -> None:
    """Gather the sequences seq_ids (device int32 [nb]) into out bf16 [total, 576]:
    sequence seq_ids[i] fills rows out_offsets[i] .. out_offsets[i+1] (device
    int64 [nb + 1], out_offsets[0] = 0, out_offsets[nb] = total)."""
    _need(rows, "rows", torch.uint8)
    if rows.dim() != 3 or tuple(rows.shape[1:]) != (PAGE, NVFP4_ROW_BYTES):
        raise ValueError(f"rows has shape {tuple(rows.shape)}, expected (pages, {PAGE}, {NVFP4_ROW_BYTES})")
    _need(block_table, "block_table", torch.int32)
    _need(seq_ids, "seq_ids", torch.int32)
    nb = seq_ids.shape[0]
    _need(out_offsets, "out_offsets", torch.int64, (nb + 1,))
    _need(out, "out", torch.bfloat16)
    if out.dim() != 2 or out.shape[1] != D_QK:
        raise ValueError(f"out has shape {tuple(out.shape)}, expected (total, {D_QK})")
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_gather_paged_nvfp4_batch(_ptr(rows), float(tensor_scale), rows.shape[0], _ptr(block_table),
                                              block_table.shape[0], block_table.shape[1], _ptr(seq_ids),
                                              _ptr(out_offsets), nb, out.shape[0], _ptr(out), _ptr(dev_err),
                                              _stream(stream)))


def mla_prefill_threshold() -> int:
    return int(lib().mla_prefill_threshold())


def mla_branch_for(q_len: int) -> int:
    """0 = absorbed (steps A2-A5), 1 = decompress branch."""
    return int(lib().mla_branch_for(int(q_len)))


def mla_expand_kv(rows, w_uk, w_uv, k_c, v_c, dev_err, stream=None) -> None:
    n = rows.shape[0]
    _need(rows, "rows", torch.bfloat16, (n, D_QK))
    _need(w_uk, "w_uk", torch.bfloat16, (H, D_HC, D_C))
    _need(w_uv, "w_uv", torch.bfloat16, (H, D_C, D_HC))
    _need(k_c, "k_c", torch.bfloat16, (H, n, D_HC))
    _need(v_c, "v_c", torch.bfloat16, (H, n, D_HC))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_expand_kv(_ptr(rows), int(n), _ptr(w_uk), _ptr(w_uv), _ptr(k_c), _ptr(v_c), _ptr(dev_err),
                               _stream(stream)))


def mla_prefill_attention(q_c, q_r, rows, k_c, v_c, out, dev_err, scale: float = 1.0 / (192 ** 0.5),
                          stream=None) -> None:
    M, N = q_c.shape[0], rows.shape[0]
    _need(q_c, "q_c", torch.bfloat16, (M, H, D_HC))
    _need(q_r, "q_r", torch.bfloat16, (M, H, D_R))
    _need(rows, "rows", torch.bfloat16, (N, D_QK))
    _need(k_c, "k_c", torch.bfloat16, (H, N, D_HC))
    _need(v_c, "v_c", torch.bfloat16, (H, N, D_HC))
    _need(out, "out", torch.bfloat16, (M, H, D_HC))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_prefill_attention(_ptr(q_c), _ptr(q_r), int(M), _ptr(rows), _ptr(k_c), _ptr(v_c), int(N),
                                       float(scale), _ptr(out), _ptr(dev_err), _stream(stream)))


def mla_prefill_workspace_size(N: int) -> int:
    out = C.c_size_t()
    _check(lib().mla_prefill_workspace_size(int(N), C.byref(out)))
    return int(out.value)


def mla_prefill_decompress(q_c, q_r, kv_cache, block_table, b: int, n_tokens: int, w_uk, w_uv, workspace, out,
                           dev_err, scale: float = 1.0 / (192 ** 0.5), stream=None) -> None:
    """The decompress branch for sequence b (n_tokens cached, the chunk's M = q_c.shape[0] rows last)."""
    M = q_c.shape[0]
    _need(q_c, "q_c", torch.bfloat16, (M, H, D_HC))
    _need(q_r, "q_r", torch.bfloat16, (M, H, D_R))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(w_uk, "w_uk", torch.bfloat16, (H, D_HC, D_C))
    _need(w_uv, "w_uv", torch.bfloat16, (H, D_C, D_HC))
    _need(workspace, "workspace", torch.uint8)
    _need(out, "out", torch.bfloat16, (M, H, D_HC))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_prefill_decompress(_ptr(q_c), _ptr(q_r), int(M), _ptr(kv_cache), kv_cache.shape[0],
                                        _ptr(block_table), block_table.shape[1], int(b), int(n_tokens), _ptr(w_uk),
                                        _ptr(w_uv), float(scale), _ptr(workspace), workspace.numel(), _ptr(out),
                                        _ptr(dev_err), _stream(stream)))


def mla_prefill_batch_workspace_size(n_tokens: Sequence[int]) -> int:
    n = np.ascontiguousarray(n_tokens, dtype=np.int32)
    out = C.c_size_t()
    _check(lib().mla_prefill_batch_workspace_size(n.ctypes.data_as(C.POINTER(C.c_int32)), int(n.size),
                                                  C.byref(out)))
    return int(out.value)


def mla_prefill_decompress_batch(q_c, q_r, kv_cache, block_table, seq_ids, q_starts, q_lens, n_tokens, w_uk, w_uv,
                                 workspace, out, dev_err, scale: float = 1.0 / (192 ** 0.5), stream=None) -> None:
    """The decompress branch for several sequences at once: sequence seq_ids[i]
    (n_tokens[i] cached) with its chunk's q_lens[i] query rows at rows
    q_starts[i].. of q_c, q_r and out."""
    rows = q_c.shape[0]
    _need(q_c, "q_c", torch.bfloat16, (rows, H, D_HC))
    _need(q_r, "q_r", torch.bfloat16, (rows, H, D_R))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(w_uk, "w_uk", torch.bfloat16, (H, D_HC, D_C))
    _need(w_uv, "w_uv", torch.bfloat16, (H, D_C, D_HC))
    _need(workspace, "workspace", torch.uint8)
    _need(out, "out", torch.bfloat16, (rows, H, D_HC))
    _need(dev_err, "dev_err", torch.int32, (1,))
    arrs = [np.ascontiguousarray(x, dtype=np.int32) for x in (seq_ids, q_starts, q_lens, n_tokens)]
    nb = int(arrs[0].size)
    if any(a.size != nb for a in arrs):
        raise ValueError("seq_ids, q_starts, q_lens and n_tokens must have the same length")
    if any(int(s0) + int(m) > rows for s0, m in zip(arrs[1], arrs[2])):
        raise ValueError("a chunk's rows run past q_c")
    P32 = C.POINTER(C.c_int32)
    _check(lib().mla_prefill_decompress_batch(
        _ptr(q_c), _ptr(q_r), *[a.ctypes.data_as(P32) for a in arrs], nb, _ptr(kv_cache), kv_cache.shape[0],
        _ptr(block_table), block_table.shape[0], block_table.shape[1], _ptr(w_uk), _ptr(w_uv), float(scale),
        _ptr(workspace), workspace.numel(), _ptr(out), _ptr(dev_err), _stream(stream)))


def mla_rope_table(max_pos: int, table, base: float = 10000.0, stream=None) -> None:
    _need(table, "table", torch.float32, (max_pos, D_R // 2, 2))
    _check(lib().mla_rope_table(int(max_pos), float(base), _ptr(table), _stream(stream)))


def mla_kv_append_rope(c_kv_new, k_pe_new, positions, table, slots, kv_cache, dev_err, stream=None) -> None:
    n = c_kv_new.shape[0]
    _need(c_kv_new, "c_kv_new", torch.bfloat16, (n, D_C))
    _need(k_pe_new, "k_pe_new", torch.bfloat16, (n, D_R))
    _need(positions, "positions", torch.int32, (n,))
    _need(table, "table", torch.float32)
    _need(slots, "slots", torch.int64, (n,))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(dev_err, "dev_err", torch.int32, (1,))
    if table.dim() != 3 or tuple(table.shape[1:]) != (D_R // 2, 2):
        raise ValueError(f"table has shape {tuple(table.shape)}, expected (max_pos, {D_R // 2}, 2)")
    _check(lib().mla_kv_append_rope(_ptr(c_kv_new), _ptr(k_pe_new), _ptr(positions), _ptr(table), table.shape[0],
                                    _ptr(slots), int(n), _ptr(kv_cache), kv_cache.shape[0], _ptr(dev_err),
                                    _stream(stream)))


def mla_rope_q(q_pe, positions, table, q_r, dev_err, stream=None) -> None:
    T = q_pe.shape[0]
    _need(q_pe, "q_pe", torch.bfloat16, (T, H, D_R))
    _need(positions, "positions", torch.int32, (T,))
    _need(table, "table", torch.float32)
    _need(q_r, "q_r", torch.bfloat16, (T, H, D_R))
    _need(dev_err, "dev_err", torch.int32, (1,))
    if table.dim() != 3 or tuple(table.shape[1:]) != (D_R // 2, 2):
        raise ValueError(f"table has shape {tuple(table.shape)}, expected (max_pos, {D_R // 2}, 2)")
    _check(lib().mla_rope_q(_ptr(q_pe), _ptr(positions), _ptr(table), table.shape[0], _ptr(q_r), int(T),
                            _ptr(dev_err), _stream(stream)))


def mla_gather_paged(kv_cache, block_table, b: int, n_tokens: int, out, dev_err, stream=None) -> None:
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(out, "out", torch.bfloat16, (n_tokens, D_QK))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_gather_paged(_ptr(kv_cache), kv_cache.shape[0], _ptr(block_table), block_table.shape[1],
                                  int(b), int(n_tokens), _ptr(out), _ptr(dev_err), _stream(stream)))


def mla_absorb_q(q_c, w_uk, q_abs, dev_err, stream=None) -> None:
    T = q_c.shape[0]
    _need(q_c, "q_c", torch.bfloat16, (T, H, D_HC))
    _need(w_uk, "w_uk", torch.bfloat16, (H, D_HC, D_C))
    _need(q_abs, "q_abs", torch.bfloat16, (T, H, D_C))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_absorb_q(_ptr(q_c), _ptr(w_uk), _ptr(q_abs), int(T), _ptr(dev_err), _stream(stream)))


def mla_up_v(o_lat, w_uv, out, dev_err, stream=None) -> None:
    T = o_lat.shape[0]
    _need(o_lat, "o_lat", torch.bfloat16, (T, H, D_C))
    _need(w_uv, "w_uv", torch.bfloat16, (H, D_C, D_HC))
    _need(out, "out", torch.bfloat16, (T, H, D_HC))
    _need(dev_err, "dev_err", torch.int32, (1,))
    _check(lib().mla_up_v(_ptr(o_lat), _ptr(w_uv), _ptr(out), int(T), _ptr(dev_err), _stream(stream)))


def mla_decode_max_clusters() -> int:
    out = C.c_int32()
    _check(lib().mla_decode_max_clusters(C.byref(out)))
    return int(out.value)


def mla_decode_plan_bytes(T: int, num_clusters: int) -> int:
    out = C.c_size_t()
    _check(lib().mla_decode_plan_bytes(int(T), int(num_clusters), C.byref(out)))
    return int(out.value)


def mla_decode_workspace_size(num_clusters: int) -> int:
    out = C.c_size_t()
    _check(lib().mla_decode_workspace_size(int(num_clusters), C.byref(out)))
    return int(out.value)


def mla_decode_plan_host(seq_lens: Sequence[int], q_lens: Sequence[int], num_clusters: int):
    """Host planner only (no GPU): returns (plan int32 array, info)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    T = int(ql.sum()) if ql.size else 0
    nbytes = mla_decode_plan_bytes(T, num_clusters)
    buf = np.zeros(nbytes // 4, dtype=np.int32)
    info = mla_plan_info()
    P32 = C.POINTER(C.c_int32)
    _check(lib().mla_decode_plan_host(sl.ctypes.data_as(P32), ql.ctypes.data_as(P32), int(sl.size),
                                      int(num_clusters), buf.ctypes.data_as(C.c_void_p), nbytes, C.byref(info)))
    return buf, info


@dataclass
class DecodePlan:
    """A plan on the device plus its host summary (mla_decode_plan)."""
    plan: torch.Tensor          # int32 device buffer
    info: mla_plan_info
    workspace: torch.Tensor     # uint8 device buffer
    host: Optional[torch.Tensor] = None   # pinned int32 staging of the plan (reused by `into=`)

    @property
    def num_clusters(self) -> int:
        return int(self.info.num_clusters)


def mla_decode_plan(seq_lens: Sequence[int], q_lens: Sequence[int], device=None, num_clusters: Optional[int] = None,
                    stream=None, into: Optional[DecodePlan] = None) -> DecodePlan:
    """Plan on the host into a pinned buffer and upload it with an
    asynchronous copy on `stream` (a copy from pageable memory would make
    the host wait for the stream).  `into` reuses a previous plan's buffers
    when they are large enough; the caller must not reuse a plan whose
    previous upload or decode may still be running."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    T = int(ql.sum()) if ql.size else 0
    if num_clusters is None:
        num_clusters = into.num_clusters if into is not None else mla_decode_max_clusters()
    nbytes = mla_decode_plan_bytes(T, num_clusters)
    words = (nbytes + 15) // 16 * 4
    device = device or torch.device("cuda", torch.cuda.current_device())
    ws_bytes = max(mla_decode_workspace_size(num_clusters), 16)
    if (into is not None and into.host is not None and into.plan.numel() >= words
            and into.workspace.numel() >= ws_bytes and into.plan.device == torch.device(device)):
        plan, ws, host = into.plan, into.workspace, into.host
    else:
        plan = torch.empty(words, dtype=torch.int32, device=device)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        host = torch.zeros(words, dtype=torch.int32).pin_memory()
    info = mla_plan_info()
    P32 = C.POINTER(C.c_int32)
    _check(lib().mla_decode_plan_host(sl.ctypes.data_as(P32), ql.ctypes.data_as(P32), int(sl.size),
                                      int(num_clusters), C.c_void_p(host.data_ptr()), nbytes, C.byref(info)))
    if stream is None:
        plan[:words].copy_(host[:words], non_blocking=True)
    else:
        with torch.cuda.stream(stream):
            plan[:words].copy_(host[:words], non_blocking=True)
    return DecodePlan(plan=plan, info=info, workspace=ws, host=host)


def plan_rows(plan: DecodePlan) -> dict:
    """The query rows a plan treats specially, read from its host copy (the
    plan layout of csrc/internal.h): rows cut into several pieces (merged by
    the combine) and rows whose segment starts or ends a cluster's range.
    For choosing parity samples; no device work."""
    w = plan.host.numpy() if plan.host is not None else None
    if w is None:
        raise ValueError("the plan has no host copy")
    nc, ns, nsplit = int(w[3]), int(w[4]), int(w[6])
    seg_off = 16
    seg_base = (seg_off + nc + 1 + 7) // 8 * 8
    split_base = seg_base + 8 * ns
    split = sorted(int(w[split_base + 4 * i]) for i in range(nsplit))
    boundary = set()
    for c in range(nc):
        a, b = int(w[seg_off + c]), int(w[seg_off + c + 1])
        if b > a:
            boundary.add(int(w[seg_base + 8 * a]))
            boundary.add(int(w[seg_base + 8 * (b - 1)]))
    return {"split": split, "boundary": sorted(boundary)}


def mla_decode_paged(q_abs, q_r, kv_cache, block_table, plan: DecodePlan, o_lat, dev_err, lse=None,
                     scale: float = 1.0 / (192 ** 0.5), stream=None) -> None:
    T = q_abs.shape[0]
    _need(q_abs, "q_abs", torch.bfloat16, (T, H, D_C))
    _need(q_r, "q_r", torch.bfloat16, (T, H, D_R))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    if kv_cache.dim() != 3 or tuple(kv_cache.shape[1:]) != (PAGE, D_QK):
        raise ValueError("kv_cache must be [num_pages, 64, 576]")
    _need(block_table, "block_table", torch.int32)
    _need(o_lat, "o_lat", torch.bfloat16, (T, H, D_C))
    _need(dev_err, "dev_err", torch.int32, (1,))
    if lse is not None:
        _need(lse, "lse", torch.float32, (T, H))
    if int(plan.info.T) != T:
        raise ValueError(f"plan has {plan.info.T} rows, q_abs has {T}")
    _check(lib().mla_decode_paged(_ptr(q_abs), _ptr(q_r), _ptr(kv_cache), kv_cache.shape[0], _ptr(block_table),
                                  block_table.shape[1], _ptr(plan.plan), C.byref(plan.info), float(scale),
                                  _ptr(plan.workspace), plan.workspace.numel(), _ptr(o_lat), _ptr(lse),
                                  _ptr(dev_err), _stream(stream)))


def mla_decode_paged_fp8(q_abs, q_r, rows, scales, block_table, plan: DecodePlan, o_lat, dev_err, lse=None,
                         scale: float = 1.0 / (192 ** 0.5), stream=None) -> None:
    """Steps A3 + A4 over the FP8 cache (rows uint8 [pages, 64, 640], scales fp32 [pages, 64])."""
    T = q_abs.shape[0]
    _need(q_abs, "q_abs", torch.bfloat16, (T, H, D_C))
    _need(q_r, "q_r", torch.bfloat16, (T, H, D_R))
    _need(rows, "rows", torch.uint8, (rows.shape[0], PAGE, FP8_ROW_BYTES))
    _need(scales, "scales", torch.float32, (rows.shape[0], PAGE))
    _need(block_table, "block_table", torch.int32)
    _need(o_lat, "o_lat", torch.bfloat16, (T, H, D_C))
    _need(dev_err, "dev_err", torch.int32, (1,))
    if lse is not None:
        _need(lse, "lse", torch.float32, (T, H))
    if int(plan.info.T) != T:
        raise ValueError(f"plan has {plan.info.T} rows, q_abs has {T}")
    _check(lib().mla_decode_paged_fp8(_ptr(q_abs), _ptr(q_r), _ptr(rows), _ptr(scales), rows.shape[0],
                                      _ptr(block_table), block_table.shape[1], _ptr(plan.plan), C.byref(plan.info),
                                      float(scale), _ptr(plan.workspace), plan.workspace.numel(), _ptr(o_lat),
                                      _ptr(lse), _ptr(dev_err), _stream(stream)))


def mla_check(dev_err, stream=None) -> int:
    """Synchronise and return the device error word; raises on a non-zero word."""
    word = C.c_int32()
    _check(lib().mla_check(_stream(stream), _ptr(dev_err), C.byref(word)))
    return int(word.value)


def mla_debug_set_decode_wait_limit(cycles: int) -> None:
    """Test hook: every wait of the decode loop gives up after `cycles` SM
    cycles (0 restores the default of 2^31); process-wide."""
    _check(lib().mla_debug_set_decode_wait_limit(int(cycles)))


def mla_decode_paged_noalloc(q_abs, q_r, kv_cache, block_table, seq_lens, q_lens, o_lat, dev_err, lse=None,
                             scale: float = 1.0 / (192 ** 0.5), stream=None) -> None:
    """mla_decode_paged without caller-provided plan or workspace: for callers
    that cannot allocate device memory (the library keeps both in a device
    array of its own).  Calls that may overlap on the GPU must be serialised."""
    T = q_abs.shape[0]
    _need(q_abs, "q_abs", torch.bfloat16, (T, H, D_C))
    _need(q_r, "q_r", torch.bfloat16, (T, H, D_R))
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need(block_table, "block_table", torch.int32)
    _need(o_lat, "o_lat", torch.bfloat16, (T, H, D_C))
    _need(dev_err, "dev_err", torch.int32, (1,))
    if lse is not None:
        _need(lse, "lse", torch.float32, (T, H))
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    if int(ql.sum()) != T:
        raise ValueError(f"q_lens sum to {int(ql.sum())} rows, q_abs has {T}")
    P32 = C.POINTER(C.c_int32)
    _check(lib().mla_decode_paged_noalloc(_ptr(q_abs), _ptr(q_r), _ptr(kv_cache), kv_cache.shape[0],
                                          _ptr(block_table), block_table.shape[1], sl.ctypes.data_as(P32),
                                          ql.ctypes.data_as(P32), int(sl.size), float(scale), _ptr(o_lat),
                                          _ptr(lse), _ptr(dev_err), _stream(stream)))
