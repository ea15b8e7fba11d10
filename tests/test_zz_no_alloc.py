"""The allocation-free decode entry point, mla_decode_paged_noalloc.

It serves callers that cannot allocate device memory (a plugin handed only
its input and output tensors, an engine whose pool already owns all free
device memory), so it keeps the split plan and workspace in a device array
of the library instead of caller buffers.  These tests call it through the C
ABI and compare it with the regular entry point, mla_decode_paged, within
the tolerance the parity tests use, on two calls in a row that reuse the
shared array.  This file is collected last on purpose.
"""
import ctypes as C
import math

import numpy as np
import pytest

from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import DeviceCase, assert_close, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from mla_latent_kv_02_gb300 import _lib
    return _lib.lib()


def _call_noalloc(lib, dc, case):
    T = case.T
    o = torch.full((T, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, 128), float("nan"), dtype=torch.float32, device="cuda")
    sl = np.ascontiguousarray(case.seq_lens, dtype=np.int32)
    ql = np.ascontiguousarray(case.q_lens, dtype=np.int32)
    P32 = C.POINTER(C.c_int32)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.mla_decode_paged_noalloc(
        C.c_void_p(dc.q_abs.data_ptr()), C.c_void_p(dc.q_r.data_ptr()), C.c_void_p(dc.kv_cache.data_ptr()),
        dc.kv_cache.shape[0], C.c_void_p(dc.block_table.data_ptr()), dc.block_table.shape[1],
        sl.ctypes.data_as(P32), ql.ctypes.data_as(P32), int(sl.size), C.c_float(SCALE),
        C.c_void_p(o.data_ptr()), C.c_void_p(lse.data_ptr()), C.c_void_p(dc.dev_err.data_ptr()), stream)
    assert st == 0, lib.mla_last_error().decode()
    word = C.c_int32()
    assert lib.mla_check(stream, C.c_void_p(dc.dev_err.data_ptr()), C.byref(word)) == 0, word.value
    return o, lse


def test_noalloc_matches_regular_entry_point_on_two_calls(lib):
    # Two different batches back to back: the second call reuses (and must
    # fully overwrite) the shared plan and workspace of the first.
    cases = [wl.make_case([300, 1500, 64, 4000], [1, 2, 1, 1], seed=31, with_weights=False, with_q_abs=True),
             wl.make_case([5000, 70, 9000], [2, 1, 1], seed=32, with_weights=False, with_q_abs=True)]
    for case in cases:
        dc = DeviceCase(case, with_weights=False)
        o_ref, lse_ref, plan = dc.decode()
        assert plan.info.num_split_rows > 0          # the split-KV workspace is exercised
        o, lse = _call_noalloc(lib, dc, case)
        assert_close(to_np(o), to_np(o_ref), "o_lat no-alloc vs regular")
        assert_close(lse.cpu().numpy(), lse_ref.cpu().numpy(), "lse no-alloc vs regular",
                     max_frac=1e-3, mean_rel=1e-4)


def test_noalloc_uses_fewer_clusters_when_the_split_pieces_exceed_its_scratch(lib):
    # Sixteen sequences of 64K tokens (the long-context workload): with every
    # cluster, each row is cut into pieces that need more workspace than the
    # array holds, so the call plans with fewer clusters, still splitting rows
    # (the workspace in use), and must match the regular entry point.
    from mla_latent_kv_02_gb300 import _lib
    case = wl.workload(3, with_q_abs=True, with_weights=False)
    dc = DeviceCase(case, with_weights=False)
    o_ref, lse_ref, plan = dc.decode()
    o, lse = _call_noalloc(lib, dc, case)
    info = _lib.mla_plan_info()
    assert lib.mla_debug_noalloc_last_plan(C.byref(info)) == 0, lib.mla_last_error().decode()
    assert 0 < info.num_partials and info.num_clusters < plan.info.num_clusters
    assert info.num_partials * (128 * 512 * 4 + 128 * 4) <= 16 * 1024 * 1024
    assert_close(to_np(o), to_np(o_ref), "o_lat no-alloc (fewer clusters) vs regular")
    assert_close(lse.cpu().numpy(), lse_ref.cpu().numpy(), "lse no-alloc (fewer clusters) vs regular",
                 max_frac=1e-3, mean_rel=1e-4)


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    # A plan for this many query rows exceeds the fixed plan area: the call must
    # fail on the host with a clear message and enqueue nothing.
    B = 20000
    sl = np.full(B, 2, dtype=np.int32)
    ql = np.ones(B, dtype=np.int32)
    P32 = C.POINTER(C.c_int32)
    dummy = C.c_void_p(0x1000)
    st = lib.mla_decode_paged_noalloc(dummy, dummy, dummy, 1, dummy, 1, sl.ctypes.data_as(P32),
                                      ql.ctypes.data_as(P32), B, C.c_float(SCALE), dummy, None, dummy, None)
    assert st == 1
    assert "no-alloc scratch" in lib.mla_last_error().decode()
