"""GPU parity of the FP8 (E4M3) latent cache against the oracle.

Integer and byte work, so the bar is bit-exactness:
* the quantising append: every code byte, every RoPE byte and every scale
  equal the oracle's (the scale is a power of two, so the rounding decision
  is the same in any precision);
* the dequantising gather: every bf16 bit pattern equals the oracle's
  code * 2^k (exactly representable), including -0 and, through a cache
  written by hand, all 254 finite codes at scales on both sides of the
  one- and two-multiply paths.
"""
import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

import math

from _helpers import DeviceCase, assert_close, oracle_cache_fp8, to_bf16, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
f8 = oracle.fp8_cache


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from mla_latent_kv_02_gb300 import api as a
    a.mla_version()
    return a


def _bits(t):
    return t.view(torch.int16).cpu().numpy().astype(np.uint16)


def _bf16_bits_of(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _special_rows(rng):
    """Latent rows that reach every branch of the quantiser."""
    rows = [wl.bf16_round(rng.standard_normal(512, dtype=np.float32)) for _ in range(5)]
    rows.append(np.zeros(512, np.float32))                                        # all zero: k = 0
    r = wl.bf16_round(rng.standard_normal(512, dtype=np.float32) * np.float32(1e-30))
    rows.append(r)                                                                # small k
    rows.append(wl.bf16_round(rng.standard_normal(512, dtype=np.float32) * np.float32(1e30)))  # large k
    r = np.zeros(512, np.float32)
    r[0] = 448.0                                   # amax exactly 448: k = 0
    mids = np.array([1.0625, 1.1875, -1.0625, 0.005859375, 2.0 ** -10, -2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -12],
                    np.float32)
    r[1:1 + len(mids)] = mids                      # exact ties, subnormal codes, values rounding to +-0
    r[20] = -0.0
    rows.append(r)
    r = np.zeros(512, np.float32)
    r[5] = 450.0                                   # just over 448 (449 is not a bf16 value): k = 1
    r[6] = -224.0
    rows.append(r)
    r = wl.bf16_round(rng.standard_normal(512, dtype=np.float32) * np.float32(1e-40))   # bf16 subnormals
    rows.append(r)
    out = np.stack(rows)
    assert np.array_equal(wl.bf16_round(out), out, equal_nan=False), "special rows must be bf16 values"
    return out


@pytest.mark.parametrize("n_random", [0, 50, 1000])
def test_kv_append_fp8_bit_exact(api, n_random):
    rng = np.random.default_rng(40 + n_random)
    special = _special_rows(rng)
    c = np.concatenate([special, wl.bf16_round(rng.standard_normal((n_random, 512), dtype=np.float32))])
    n = c.shape[0]
    k = wl.bf16_round(rng.standard_normal((n, 64), dtype=np.float32))
    pages = (n + 63) // 64 + 2
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    rows = torch.zeros((pages, 64, 640), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((pages, 64), dtype=torch.float32, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_fp8(to_bf16(c, "cuda"), to_bf16(k, "cuda"), torch.from_numpy(slots).cuda(), rows, scales,
                          dev_err)
    assert api.mla_check(dev_err) == 0
    want_rows, want_scales = f8.append(*f8.empty_cache(pages), c, k, slots)
    got_rows = rows.cpu().numpy()
    bad = np.nonzero(np.any(got_rows.reshape(-1, 640) != want_rows.reshape(-1, 640), axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first slot {bad[:5]}"
    assert np.array_equal(scales.cpu().numpy().astype(np.float64), want_scales)


def test_gather_fp8_bit_exact_after_append(api):
    rng = np.random.default_rng(44)
    special = _special_rows(rng)[:-1]              # bf16-subnormal rows fall below bf16 after scaling
    c = np.concatenate([special, wl.bf16_round(rng.standard_normal((300, 512), dtype=np.float32))])
    n = c.shape[0]
    k = wl.bf16_round(rng.standard_normal((n, 64), dtype=np.float32))
    pages = (n + 63) // 64
    bt = rng.permutation(pages).astype(np.int32)[None, :]
    slots = oracle.slot_mapping(bt, np.zeros(n, np.int32), np.arange(n))
    rows = torch.zeros((pages, 64, 640), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((pages, 64), dtype=torch.float32, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_fp8(to_bf16(c, "cuda"), to_bf16(k, "cuda"), torch.from_numpy(slots).cuda(), rows, scales,
                          dev_err)
    out = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    api.mla_gather_paged_fp8(rows, scales, torch.from_numpy(bt).cuda(), 0, n, out, dev_err)
    assert api.mla_check(dev_err) == 0
    want_rows, want_scales = f8.append(*f8.empty_cache(pages), c, k, slots)
    lat, rope = f8.gather(want_rows, want_scales, bt, 0, n)
    want = np.concatenate([lat, rope], axis=1).astype(np.float32)
    assert np.array_equal(_bits(out), _bf16_bits_of(want))


def test_gather_fp8_every_code_and_scale(api):
    """A cache written by hand: each token holds all 254 finite codes (twice,
    in two orders) at one of a range of scales."""
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    exps = [-120, -100, -30, -7, 0, 7, 15, 16, 17, 60, 119]
    n = len(exps)
    host_rows = np.zeros((1, 64, 640), dtype=np.uint8)
    host_scales = np.zeros((1, 64), dtype=np.float32)
    rng = np.random.default_rng(45)
    for i, e in enumerate(exps):
        host_rows[0, i, :254] = finite
        host_rows[0, i, 254:508] = rng.permutation(finite)
        host_rows[0, i, 508:512] = [0x00, 0x80, 0x01, 0x81]
        host_rows[0, i, 512:] = rng.integers(0, 256, 128, dtype=np.uint8)
        host_scales[0, i] = np.ldexp(np.float32(1.0), e)
    rows = torch.from_numpy(host_rows).cuda()
    scales = torch.from_numpy(host_scales).cuda()
    out = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_gather_paged_fp8(rows, scales, torch.zeros((1, 1), dtype=torch.int32, device="cuda"), 0, n, out, dev_err)
    assert api.mla_check(dev_err) == 0
    lat = f8.dequantize_rows(host_rows[0, :n, :512], host_scales[0, :n].astype(np.float64)).astype(np.float32)
    got = _bits(out)
    assert np.array_equal(got[:, :512], _bf16_bits_of(lat)), "dequantised latent differs"
    assert np.array_equal(got[:, 512:].view(np.uint8).reshape(n, 128), host_rows[0, :n, 512:])


def test_fp8_errors_and_empty(api):
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = torch.zeros((2, 64, 640), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    c = torch.ones((3, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((3, 64), dtype=torch.bfloat16, device="cuda")
    api.mla_kv_append_fp8(c, k, torch.tensor([0, 128, 5], dtype=torch.int64, device="cuda"), rows, scales, dev_err)
    assert int(dev_err.item()) == api.DEVERR_SLOT_OOB
    got = rows.cpu().numpy().reshape(-1, 640)
    assert np.all(got[0, :512] == f8.e4m3_encode([256.0])[0])   # all-ones row: scale 2^-8, code of 256
    assert np.all(got[1] == 0) and np.all(got[5, :512] == got[0, :512])
    assert scales.cpu().numpy().reshape(-1)[0] == 2.0 ** -8
    dev_err.zero_()
    out = torch.empty((70, 576), dtype=torch.bfloat16, device="cuda")
    api.mla_gather_paged_fp8(rows, scales, torch.tensor([[0, 7]], dtype=torch.int32, device="cuda"), 0, 70, out,
                             dev_err)
    assert int(dev_err.item()) == api.DEVERR_PAGE_OOB
    dev_err.zero_()
    api.mla_kv_append_fp8(c[:0], k[:0], torch.empty(0, dtype=torch.int64, device="cuda"), rows, scales, dev_err)
    assert api.mla_check(dev_err) == 0


# ------------------------------------------------------------------ decode over the FP8 cache (A3 + A4)
SCALE = 1.0 / math.sqrt(192)


def _check_decode_fp8(api, case, num_clusters=None, tag=""):
    dc = DeviceCase(case, with_weights=False, fp8=True)
    o, lse, plan = dc.decode(num_clusters=num_clusters)
    rows, scales = oracle_cache_fp8(case)
    ref_o, ref_lse = f8.decode(case.q_abs, case.q_r, rows, scales, case.block_table, case.seq_lens, case.q_lens,
                               SCALE)
    assert_close(to_np(o), ref_o, f"fp8 o_lat {tag}")
    assert_close(lse.cpu().numpy(), ref_lse, f"fp8 lse {tag}", max_frac=2e-3, mean_rel=5e-4)
    return plan


@pytest.mark.parametrize("num_clusters", [1, 2, 5, None])
def test_decode_fp8_ragged_lengths(api, num_clusters):
    case = wl.make_case([1, 63, 64, 65, 130, 700], [1, 1, 1, 2, 3, 1], seed=57, with_weights=False,
                        with_q_abs=True)
    _check_decode_fp8(api, case, num_clusters, f"clusters={num_clusters}")


def test_decode_fp8_split_rows_mtp_and_prefill(api):
    _check_decode_fp8(api, wl.make_case([2000, 3000], [1, 1], seed=58, with_weights=False, with_q_abs=True), 16,
                      "split")
    _check_decode_fp8(api, wl.make_case([300, 513, 322], [2, 2, 2], seed=59, with_weights=False,
                                        with_q_abs=True), None, "mtp")
    _check_decode_fp8(api, wl.make_case([250], [130], seed=60, with_weights=False, with_q_abs=True), None,
                      "prefill")


def test_decode_fp8_matches_decode_on_dequantised_bf16_cache(api):
    """The FP8 kernel sees exactly the latent values the dequantising gather
    returns (its f16 operands differ from the bf16 kernel's only in how q,
    the RoPE key and P are rounded): the bf16 kernel run on that gathered
    cache agrees within the floating tolerance."""
    case = wl.make_case([130, 700, 64], [1, 2, 1], seed=61, with_weights=False, with_q_abs=True)
    dc8 = DeviceCase(case, with_weights=False, fp8=True)
    o8, l8, _ = dc8.decode(num_clusters=3)
    dc = DeviceCase(case, with_weights=False)
    for b in range(case.B):
        n = int(case.seq_lens[b])
        rows = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
        api.mla_gather_paged_fp8(dc8.rows, dc8.scales, dc8.block_table, b, n, rows, dc8.dev_err)
        pages = case.block_table[b, :(n + 63) // 64]
        flat = dc.kv_cache.view(-1, 576)
        for j in range(n):
            flat[int(pages[j // 64]) * 64 + j % 64] = rows[j]
    o, l, _ = dc.decode(num_clusters=3)
    assert_close(to_np(o8), to_np(o).astype(np.float64), "fp8 vs bf16 kernel on the gathered cache")
    assert_close(l8.cpu().numpy(), l.cpu().numpy().astype(np.float64), "lse", max_frac=2e-3, mean_rel=5e-4)


def test_decode_fp8_flags_scales_outside_the_f16_range(api):
    """A token whose scale leaves [2^-15, 2^7] cannot be an exact f16 operand:
    the decode clamps it and sets MLA_DEVERR_FP8_RANGE; in-range tokens do not.
    (A tiny token, max|c| = 1e-3, scale 2^-18: clamping keeps the outputs finite.)"""
    case = wl.make_case([130], [1], seed=64, with_weights=False, with_q_abs=True)
    dc = DeviceCase(case, with_weights=False, fp8=True)
    o, _, _ = dc.decode(num_clusters=2)                     # all in range: no flag (checked inside)
    tiny = torch.full((1, 512), 1e-3, dtype=torch.bfloat16, device="cuda")
    api.mla_kv_append_fp8(tiny, torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda"),
                          torch.tensor([int(dc.slots_all[5])], dtype=torch.int64, device="cuda"), dc.rows, dc.scales,
                          dc.dev_err)
    assert api.mla_check(dc.dev_err) == 0                    # the append itself is exact at any scale
    plan = api.mla_decode_plan(case.seq_lens, case.q_lens, num_clusters=2)
    o2 = torch.empty_like(o)
    api.mla_decode_paged_fp8(dc.q_abs, dc.q_r, dc.rows, dc.scales, dc.block_table, plan, o2, dc.dev_err)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) & api.DEVERR_FP8_RANGE
    assert torch.isfinite(o2.float()).all()


def test_decode_fp8_page_permutation_invariance(api):
    a = wl.make_case([150, 260], [1, 2], seed=62, page_order="identity", with_weights=False, with_q_abs=True)
    b = wl.make_case([150, 260], [1, 2], seed=62, page_order="random", with_weights=False, with_q_abs=True)
    oa, la, _ = DeviceCase(a, with_weights=False, fp8=True).decode()
    ob, lb, _ = DeviceCase(b, with_weights=False, fp8=True).decode()
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_decode_fp8_bad_page_id_sets_error_word(api):
    case = wl.make_case([130], [1], seed=63, with_weights=False, with_q_abs=True)
    dc = DeviceCase(case, with_weights=False, fp8=True)
    bt = dc.block_table.clone()
    bt[0, 1] = case.num_pages + 5
    plan = api.mla_decode_plan(case.seq_lens, case.q_lens, num_clusters=2)
    o = torch.empty((1, 128, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_decode_paged_fp8(dc.q_abs, dc.q_r, dc.rows, dc.scales, bt, plan, o, dc.dev_err)
    with pytest.raises(api.MlaError):
        api.mla_check(dc.dev_err)
    assert int(dc.dev_err.item()) & api.DEVERR_PAGE_OOB


def _fp8_row_reference(case, q_abs, t, b, i):
    """One query row against its sequence's tokens, quantised by the oracle."""
    n = oracle.visible_tokens(int(case.seq_lens[b]), int(case.q_lens[b]), i)
    off = int(case.tok_off[b])
    codes, sc = f8.quantize_rows(case.c_kv[off:off + n])
    lat = f8.dequantize_rows(codes, sc)
    return oracle.attention_row(q_abs[t], case.q_r[t], lat, case.k_r[off:off + n].astype(np.float64), SCALE)


@pytest.mark.parametrize("cfg,k", [(2, 6), (3, 4)])
def test_decode_fp8_full_size_sampled_rows(api, cfg, k):
    """The MTP B64 x 8K and B16 x 64K workloads at full size, FP8 cache,
    in the bench's launch configuration; the oracle computes sampled rows,
    half of them rows that the combine merges from split pieces."""
    case = wl.workload(cfg, with_q_abs=True, with_weights=False)
    dc = DeviceCase(case, with_weights=False, fp8=True)
    o, lse, plan = dc.decode()
    index = oracle.row_index(case.seq_lens, case.q_lens)
    split = api.plan_rows(plan)["split"]
    assert split, "the full-size workloads split rows across clusters"
    rng = np.random.Generator(np.random.PCG64(99))
    pick = {0, case.T - 1} | set(int(x) for x in rng.choice(split, size=min(len(split), k // 2), replace=False))
    pick |= set(int(x) for x in rng.choice(case.T, size=k - len(pick), replace=False)) if k > len(pick) else set()
    pick = sorted(pick)
    got_o, got_l = to_np(o), lse.cpu().numpy()
    for t in pick:
        _, b, i = index[t]
        ro, rl = _fp8_row_reference(case, case.q_abs, t, b, i)
        assert_close(got_o[t], ro, f"cfg{cfg} fp8 o_lat row {t}")
        assert_close(got_l[t], rl, f"cfg{cfg} fp8 lse row {t}", max_frac=2e-3, mean_rel=5e-4)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
