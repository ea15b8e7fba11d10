"""GPU parity of the fp32 decoupled RoPE ("Tearing open DeepSeek MLA source"
page, §1: the 64-d RoPE key is cached apart from the latent; §3/§4: the
table is generated in fp32 and applied with fp32 multiply-adds) against the
oracle's float64 rotation.

Bars:
* table: each fp32 (cos, sin) within one fp32 ulp of the float64 value
  rounded to fp32, plus 2^-34 absolute: device and oracle each form the
  angle p * base^(-2i/64) in double, and a one-ulp difference in the power
  moves an angle of up to 2^16 rad by about 2^-37, which near a zero of
  cos or sin is several fp32 ulps of the tiny value;
* latent part of an appended row: bit-exact copy;
* rotated bf16 values: |gpu - ref| <= 2^-8 |ref| + 2^-20 (|x0| + |x1|) per
  element (bf16 rounding plus fp32 products of fp32-rounded cos/sin), at
  least 99% of elements equal to the oracle rounded to bf16, and the
  project-wide floating bar;
* position 0 is the identity, bit for bit.
"""
import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import assert_close, to_bf16, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_POS = 65536


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from mla_latent_kv_02_gb300 import api as a
    a.mla_version()
    return a


@pytest.fixture(scope="module")
def table(api):
    t = torch.empty((MAX_POS, 32, 2), dtype=torch.float32, device="cuda")
    api.mla_rope_table(MAX_POS, t)
    torch.cuda.synchronize()
    return t


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _check_rotated(got, x, pos, name):
    """got: bf16 results as float64 [..., 64]; x: the unrotated input; pos broadcastable."""
    ref = oracle.rope_apply(x, pos)
    x = np.asarray(x, dtype=np.float64)
    pair = np.abs(x[..., 0::2]) + np.abs(x[..., 1::2])
    slack = np.repeat(pair, 2, axis=-1) * 2.0 ** -20
    bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + slack
    assert not bad.any(), f"{name}: {int(bad.sum())} elements outside the bf16 bound"
    same = np.mean(got == wl.bf16_round(ref.astype(np.float32)))
    assert same >= 0.99, f"{name}: only {same:.4f} equal to the rounded oracle"
    assert_close(got, ref, name)


def test_rope_table_matches_oracle_to_one_ulp(table):
    got = table.cpu().numpy()
    ref = oracle.rope_table(MAX_POS).astype(np.float32)
    diff = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    ulp = np.spacing(np.abs(ref)).astype(np.float64)
    assert np.all(diff <= ulp + 2.0 ** -34), f"max diff {float((diff / ulp).max()):.2f} ulp"
    assert np.mean(got == ref) > 0.999
    # position 0: the identity rotation, exactly
    assert np.all(got[0, :, 0] == 1.0) and np.all(got[0, :, 1] == 0.0)


def test_rope_table_other_base_and_short(api):
    t = torch.empty((7, 32, 2), dtype=torch.float32, device="cuda")
    api.mla_rope_table(7, t, base=500000.0)
    ref = oracle.rope_table(7, base=500000.0).astype(np.float32)
    got = t.cpu().numpy()
    assert np.all(np.abs(got - ref) <= np.spacing(np.abs(ref)) + 2.0 ** -34)


@pytest.mark.parametrize("n", [1, 37, 1000])
def test_kv_append_rope(api, table, n):
    rng = _rng(100 + n)
    num_pages = (n + 63) // 64 + 3
    c = wl.bf16_round(rng.standard_normal((n, 512), dtype=np.float32))
    k = wl.bf16_round(rng.standard_normal((n, 64), dtype=np.float32))
    pos = rng.integers(0, MAX_POS, size=n).astype(np.int32)
    pos[0] = 0
    if n > 2:
        pos[1], pos[2] = MAX_POS - 1, 1
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    cache = torch.zeros((num_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_rope(to_bf16(c, "cuda"), to_bf16(k, "cuda"), torch.from_numpy(pos).cuda(), table,
                           torch.from_numpy(slots).cuda(), cache, dev_err)
    assert api.mla_check(dev_err) == 0
    got = to_np(cache).reshape(-1, 576).astype(np.float64)
    want = oracle.append(np.zeros((num_pages, 64, 576)), c, oracle.rope_apply(k, pos), slots).reshape(-1, 576)
    # untouched rows stay zero, latent rows are copies
    untouched = np.setdiff1d(np.arange(num_pages * 64), slots)
    assert np.all(got[untouched] == 0)
    assert np.array_equal(got[slots, :512], want[slots, :512])
    _check_rotated(got[slots, 512:], k, pos, f"k_R n={n}")
    assert np.array_equal(got[slots[0], 512:], k[0].astype(np.float64)), "position 0 must be the identity"


def test_kv_append_rope_bad_position_and_slot(api, table):
    c = torch.ones((4, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((4, 64), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((2, 64, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([-1, MAX_POS, 5, 3], dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 1, 2, 128], dtype=torch.int64, device="cuda")   # 128 is past 2 pages
    api.mla_kv_append_rope(c, k, pos, table, slots, cache, dev_err)
    with pytest.raises(api.MlaError):
        api.mla_check(dev_err)
    assert int(dev_err.item()) == api.DEVERR_POS_OOB | api.DEVERR_SLOT_OOB
    got = to_np(cache).reshape(-1, 576)
    assert np.all(got[0] == 0) and np.all(got[1] == 0) and np.all(got[2, :512] == 1) and np.all(got[3:] == 0)
    _check_rotated(got[2:3, 512:].astype(np.float64), np.ones((1, 64)), np.array([5]), "k_R row 2")


def test_kv_append_rope_empty_is_noop(api, table):
    cache = torch.zeros((1, 64, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_kv_append_rope(e, torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),
                           torch.empty(0, dtype=torch.int32, device="cuda"), table,
                           torch.empty(0, dtype=torch.int64, device="cuda"), cache, dev_err)
    assert api.mla_check(dev_err) == 0 and int(cache.abs().sum().item()) == 0


@pytest.mark.parametrize("T", [1, 3, 130])
def test_rope_q(api, table, T):
    rng = _rng(200 + T)
    q = wl.bf16_round(rng.standard_normal((T, 128, 64), dtype=np.float32))
    pos = rng.integers(0, MAX_POS, size=T).astype(np.int32)
    pos[0] = MAX_POS - 1
    if T > 1:
        pos[1] = 0
    out = torch.full((T, 128, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_rope_q(to_bf16(q, "cuda"), torch.from_numpy(pos).cuda(), table, out, dev_err)
    assert api.mla_check(dev_err) == 0
    got = to_np(out).astype(np.float64)
    _check_rotated(got, q, pos[:, None], f"q_R T={T}")
    if T > 1:
        assert np.array_equal(got[1], q[1].astype(np.float64)), "position 0 must be the identity"


def test_rope_q_bad_position_leaves_rows(api, table):
    q = torch.ones((2, 128, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((2, 128, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_rope_q(q, torch.tensor([2, MAX_POS], dtype=torch.int32, device="cuda"), table, out, dev_err)
    assert int(dev_err.item()) == api.DEVERR_POS_OOB
    got = to_np(out)
    assert np.all(np.isnan(got[1])) and np.all(np.isfinite(got[0]))


def test_rope_on_a_decode_workload_shape(api, table):
    """Cache fill and query rotation for a ragged decode batch at the
    sequences' own positions (the case's k_r / q_r arrays serve as the
    unrotated inputs)."""
    case = wl.make_case([1, 63, 64, 65, 700, 4100], [1, 1, 1, 2, 3, 1], seed=31, with_weights=False)
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    cache = torch.zeros((case.num_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_rope(to_bf16(case.c_kv, "cuda"), to_bf16(case.k_r, "cuda"), torch.from_numpy(pos).cuda(),
                           table, torch.from_numpy(slots.astype(np.int64)).cuda(), cache, dev_err)
    qpos = case.query_positions()
    q_out = torch.empty((case.T, 128, 64), dtype=torch.bfloat16, device="cuda")
    api.mla_rope_q(to_bf16(case.q_r, "cuda"), torch.from_numpy(qpos).cuda(), table, q_out, dev_err)
    assert api.mla_check(dev_err) == 0
    got = to_np(cache).reshape(-1, 576).astype(np.float64)
    assert np.array_equal(got[slots, :512], case.c_kv.astype(np.float64))
    _check_rotated(got[slots, 512:], case.k_r, pos, "k_R workload")
    _check_rotated(to_np(q_out).astype(np.float64), case.q_r, qpos[:, None], "q_R workload")
