"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element on the same seeded inputs.

Integer/byte work (append, gather) must be bit-exact.  Floating outputs must
satisfy max|err| <= 2e-2 * max|ref| and sum|err|/sum|ref| <= 5e-3.
"""
import math

import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import DeviceCase, assert_close, oracle_cache, to_bf16, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192)


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from mla_latent_kv_02_gb300 import api as a
    a.mla_version()
    return a


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


# ------------------------------------------------------------------ A1 / gather (bit-exact)
def test_kv_append_and_gather_bit_exact(api):
    case = wl.make_case([1, 63, 64, 65, 130, 700], [1, 1, 1, 2, 3, 1], seed=1, with_weights=False)
    dc = DeviceCase(case, with_weights=False)
    ref = oracle_cache(case)
    got = dc.kv_cache.float().cpu().numpy()
    assert np.array_equal(got, ref)
    # gather each sequence back, compare bits with the generated rows
    off = case.tok_off
    for b in range(case.B):
        n = int(case.seq_lens[b])
        out = torch.empty((n, wl.D_QK), dtype=torch.bfloat16, device="cuda")
        api.mla_gather_paged(dc.kv_cache, dc.block_table, b, n, out, dc.dev_err)
        want = np.concatenate([case.c_kv[off[b]:off[b] + n], case.k_r[off[b]:off[b] + n]], 1)
        assert np.array_equal(out.float().cpu().numpy(), want)
    assert api.mla_check(dc.dev_err) == 0


def test_kv_append_slot_out_of_range_sets_error_word(api):
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = torch.zeros((2, 64, 576), dtype=torch.bfloat16, device="cuda")
    c = torch.ones((3, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((3, 64), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([0, 128, 5], dtype=torch.int64, device="cuda")   # 128 is past 2 pages
    api.mla_kv_append(c, k, slots, cache, dev_err)
    with pytest.raises(api.MlaError):
        api.mla_check(dev_err)
    assert int(dev_err.item()) == api.DEVERR_SLOT_OOB
    got = cache.float().cpu().numpy().reshape(-1, 576)
    assert np.all(got[0] == 1) and np.all(got[5] == 1) and np.all(got[1] == 0)


# ------------------------------------------------------------------ A2 / A5
@pytest.mark.parametrize("T", [1, 16, 130])
def test_absorb_q(api, T):
    case = wl.make_case([T], [T], seed=2 + T)
    q_c, w_uk = to_bf16(case.q_c, "cuda"), to_bf16(case.w_uk, "cuda")
    # rows past T (a guard band after the output) must stay untouched by the tile stores
    buf = torch.full((T + 3, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    buf[T:] = 7.0
    out = buf[:T]
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_absorb_q(q_c, w_uk, out, dev_err)
    assert api.mla_check(dev_err) == 0
    assert_close(to_np(out), oracle.absorb_q(case.q_c, case.w_uk), f"q_abs T={T}")
    assert bool((buf[T:] == 7.0).all()), "a store wrote past the last row"


@pytest.mark.parametrize("T", [1, 16, 130])
def test_up_v(api, T):
    rng = np.random.Generator(np.random.PCG64(T))
    o_lat = wl.bf16_round(rng.standard_normal((T, 128, 512), dtype=np.float32) * 0.1)
    case = wl.make_case([1], [1], seed=3)
    buf = torch.full((T + 3, 128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    buf[T:] = 7.0
    out = buf[:T]
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_up_v(to_bf16(o_lat, "cuda"), to_bf16(case.w_uv, "cuda"), out, dev_err)
    assert api.mla_check(dev_err) == 0
    assert_close(to_np(out), oracle.up_v(o_lat, case.w_uv), f"out T={T}")
    assert bool((buf[T:] == 7.0).all()), "a store wrote past the last row"


# ------------------------------------------------------------------ A3 / A4
def _check_decode(api, case, num_clusters=None, tag=""):
    dc = DeviceCase(case, with_weights=False)
    o, lse, plan = dc.decode(num_clusters=num_clusters)
    ref_o, ref_lse = oracle.decode(case.q_abs, case.q_r, oracle_cache(case), case.block_table,
                                   case.seq_lens, case.q_lens, SCALE)
    assert_close(to_np(o), ref_o, f"o_lat {tag}")
    assert_close(lse.cpu().numpy(), ref_lse, f"lse {tag}", max_frac=2e-3, mean_rel=5e-4)
    return plan


@pytest.mark.parametrize("num_clusters", [1, 2, 5, None])
def test_decode_ragged_lengths(api, num_clusters):
    """Lengths 1, 63, 64, 65, 130, 700: single-token, partial and full pages,
    several tiles and ragged tails; one cluster (no splits) up to all clusters
    (split rows merged by the combine kernel)."""
    case = wl.make_case([1, 63, 64, 65, 130, 700], [1, 1, 1, 2, 3, 1], seed=7, with_weights=False,
                        with_q_abs=True)
    plan = _check_decode(api, case, num_clusters, f"clusters={num_clusters}")
    if num_clusters == 1:
        assert plan.info.num_partials == 0


def test_decode_split_rows_are_combined(api):
    case = wl.make_case([2000, 3000], [1, 1], seed=8, with_weights=False, with_q_abs=True)
    plan = _check_decode(api, case, 16, "split")
    assert plan.info.num_split_rows == 2 and plan.info.num_partials >= 4


def test_decode_mtp_two_tokens_causal(api):
    case = wl.make_case([300, 513, 64 * 5 + 2], [2, 2, 2], seed=9, with_weights=False, with_q_abs=True)
    _check_decode(api, case, None, "mtp")


def test_decode_chunked_prefill_causal(api):
    case = wl.make_case([250], [130], seed=10, with_weights=False, with_q_abs=True)
    _check_decode(api, case, None, "prefill")


def test_decode_prefill_from_empty_cache(api):
    case = wl.make_case([70], [70], seed=11, with_weights=False, with_q_abs=True)
    _check_decode(api, case, 3, "prefill-from-empty")


def test_decode_zero_query_sequences_are_skipped(api):
    case = wl.make_case([100, 200, 300], [1, 0, 2], seed=12, with_weights=False, with_q_abs=True)
    _check_decode(api, case, None, "q_len 0")


def test_decode_page_permutation_invariance(api):
    a = wl.make_case([150, 260], [1, 2], seed=13, page_order="identity", with_weights=False, with_q_abs=True)
    b = wl.make_case([150, 260], [1, 2], seed=13, page_order="random", with_weights=False, with_q_abs=True)
    oa, la, _ = DeviceCase(a, with_weights=False).decode()
    ob, lb, _ = DeviceCase(b, with_weights=False).decode()
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_decode_empty_batch_is_noop(api):
    plan = api.mla_decode_plan([], [], num_clusters=4)
    assert plan.info.T == 0
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    z = torch.zeros((0, 128, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_decode_paged(z, torch.zeros((0, 128, 64), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((1, 64, 576), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((1, 1), dtype=torch.int32, device="cuda"), plan, z, dev_err)
    assert api.mla_check(dev_err) == 0


def test_decode_bad_page_id_sets_error_word(api):
    case = wl.make_case([130], [1], seed=14, with_weights=False, with_q_abs=True)
    dc = DeviceCase(case, with_weights=False)
    bt = dc.block_table.clone()
    bt[0, 1] = case.num_pages + 5
    plan = api.mla_decode_plan(case.seq_lens, case.q_lens, num_clusters=2)
    o = torch.empty((1, 128, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_decode_paged(dc.q_abs, dc.q_r, dc.kv_cache, bt, plan, o, dc.dev_err)
    with pytest.raises(api.MlaError):
        api.mla_check(dc.dev_err)
    assert int(dc.dev_err.item()) & api.DEVERR_PAGE_OOB


# ------------------------------------------------------------------ A1..A5 together
def test_full_step_small(api):
    case = wl.make_case([90, 200, 64], [1, 2, 1], seed=15)
    dc = DeviceCase(case)
    T = case.T
    q_abs = torch.empty((T, 128, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_absorb_q(dc.q_c, dc.w_uk, q_abs, dc.dev_err)
    o, lse, _ = dc.decode(q_abs=q_abs)
    out = torch.empty((T, 128, 128), dtype=torch.bfloat16, device="cuda")
    api.mla_up_v(o, dc.w_uv, out, dc.dev_err)
    assert api.mla_check(dc.dev_err) == 0
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, oracle_cache(case), case.block_table,
                          case.seq_lens, case.q_lens, SCALE)
    assert_close(to_np(q_abs), ref["q_abs"], "q_abs")
    assert_close(to_np(o), ref["o_lat"], "o_lat")
    assert_close(to_np(out), ref["out"], "out")


# ------------------------------------------------------------------ the five workloads at full size
def _check_rows(case, plan):
    """Rows checked against the oracle at full size: every row of workloads
    0-3; for the 2048-row chunked prefill, every split row, every row whose
    segment starts or ends a cluster's range, and the first and last row of
    each block of 128 rows."""
    if case.T <= 128:
        return list(range(case.T))
    r = api_mod().plan_rows(plan)
    pick = set(r["split"]) | set(r["boundary"])
    for b0 in range(0, case.T, 128):
        pick |= {b0, min(case.T, b0 + 128) - 1}
    return sorted(pick)


def api_mod():
    from mla_latent_kv_02_gb300 import api as a
    return a


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_workload_full_size_rows(api, cfg):
    """Full-size workload in the bench's launch configuration; the oracle
    computes every row (workloads 0-3) or every split, boundary and block-end
    row (workload 4)."""
    case = wl.workload(cfg)
    dc = DeviceCase(case)
    T = case.T
    q_abs = torch.empty((T, 128, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_absorb_q(dc.q_c, dc.w_uk, q_abs, dc.dev_err)
    o, lse, plan = dc.decode(q_abs=q_abs)
    out = torch.empty((T, 128, 128), dtype=torch.bfloat16, device="cuda")
    api.mla_up_v(o, dc.w_uv, out, dc.dev_err)
    assert api.mla_check(dc.dev_err) == 0
    rows = _check_rows(case, plan)
    split = api.plan_rows(plan)["split"]
    assert set(split) <= set(rows)
    if cfg in (2, 3, 4):
        assert split, "the full-size workloads split rows across clusters"
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, oracle_cache(case), case.block_table,
                          case.seq_lens, case.q_lens, SCALE, rows=rows)
    assert_close(to_np(o)[rows], ref["o_lat"][rows], f"cfg{cfg} o_lat")
    assert_close(to_np(out)[rows], ref["out"][rows], f"cfg{cfg} out")
    assert_close(lse.cpu().numpy()[rows], ref["lse"][rows], f"cfg{cfg} lse", max_frac=2e-3, mean_rel=5e-4)
    if split:
        # the rows merged by the combine, on their own
        assert_close(to_np(o)[split], ref["o_lat"][split], f"cfg{cfg} o_lat split rows")
    # property over every row: finite outputs
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
