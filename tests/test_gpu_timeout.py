"""The decode kernel's failure path on the GPU, exercised without a fault.

Every wait inside the decode loop is bounded.  The test hook
mla_debug_set_decode_wait_limit shortens that bound to a few dozen SM cycles,
far below the latency of the first page load, so the first wait that is not
satisfied at once gives up: the kernel sets MLA_DEVERR_TIMEOUT in the call's
error word, raises its abort flag, drains its own loads, MMAs and the score
copies already in flight between the CTAs of a pair, frees its tensor memory
and returns.  Nothing hangs and no access faults.  The next call on the same
buffers, with the default bound restored, must be correct against the oracle:
that proves the context stayed usable and the tensor memory was released.
"""
import math

import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import DeviceCase, assert_close, oracle_cache, oracle_cache_fp8, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192)
SHORT_LIMIT = 64  # SM cycles


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from mla_latent_kv_02_gb300 import api as a
    a.mla_version()
    return a


def _reference(case, fp8):
    if fp8:
        rows, scales = oracle_cache_fp8(case)
        return oracle.fp8_cache.decode(case.q_abs, case.q_r, rows, scales, case.block_table, case.seq_lens,
                                       case.q_lens, SCALE)
    return oracle.decode(case.q_abs, case.q_r, oracle_cache(case), case.block_table, case.seq_lens, case.q_lens,
                         SCALE)


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_wait_expiry_is_reported_and_the_next_call_is_correct(api, fp8):
    # ragged lengths, a two-token row and split rows: several clusters, each
    # with score exchanges in flight when the bound runs out
    case = wl.make_case([700, 300, 130], [2, 1, 1], seed=41, with_weights=False, with_q_abs=True)
    dc = DeviceCase(case, with_weights=False, fp8=fp8)
    plan = api.mla_decode_plan(case.seq_lens, case.q_lens, num_clusters=3)
    T = case.T
    o = torch.zeros((T, wl.H, wl.D_C), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((T, wl.H), dtype=torch.float32, device="cuda")
    try:
        api.mla_debug_set_decode_wait_limit(SHORT_LIMIT)
        if fp8:
            api.mla_decode_paged_fp8(dc.q_abs, dc.q_r, dc.rows, dc.scales, dc.block_table, plan, o, dc.dev_err,
                                     lse=lse)
        else:
            api.mla_decode_paged(dc.q_abs, dc.q_r, dc.kv_cache, dc.block_table, plan, o, dc.dev_err, lse=lse)
    finally:
        api.mla_debug_set_decode_wait_limit(0)
    with pytest.raises(api.MlaError):
        api.mla_check(dc.dev_err)
    assert int(dc.dev_err.item()) & api.DEVERR_TIMEOUT
    # the same buffers with the default bound
    dc.dev_err.zero_()
    o2, lse2, _ = dc.decode(num_clusters=3)
    ref_o, ref_lse = _reference(case, fp8)
    assert_close(to_np(o2), ref_o, "o_lat after a timed-out call")
    assert_close(lse2.cpu().numpy(), ref_lse, "lse after a timed-out call", max_frac=2e-3, mean_rel=5e-4)


def test_wait_limit_hook_rejects_a_bound_above_the_default(api):
    with pytest.raises(api.MlaError):
        api.mla_debug_set_decode_wait_limit(1 << 40)
    api.mla_debug_set_decode_wait_limit(0)
