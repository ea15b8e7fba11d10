"""GPU parity of the NVFP4 latent cache against the oracle.

Quantised codes are integer work and the dequantised values are a fixed
sequence of correctly rounded fp32 operations, so every byte of the append
and every bf16 bit of the gather must equal the oracle's: random rows,
blocks whose codes sit exactly on E2M1 midpoints, zero and saturating
blocks, and a cache written by hand with all 16 codes under normal,
subnormal and saturated block scales.  The 16-byte alignment rule of the
pages' vector gather is checked as a host-side error, never as a fault.
"""
import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import to_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
n4 = oracle.nvfp4_cache
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


def _special_rows(rng, st):
    rows = [wl.bf16_round(rng.standard_normal(512, dtype=np.float32)) for _ in range(4)]
    r = np.zeros(512, np.float32)                              # all-zero blocks
    r[16:32] = wl.bf16_round(rng.standard_normal(16, dtype=np.float32))
    rows.append(r)
    # one block exactly on E2M1 midpoints: amax = 6 * s_b * s_t with s_b = 64 (exact E4M3)
    unit = np.float32(64.0) * np.float32(st)
    r = np.zeros(512, np.float32)
    r[:16] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, -0.0, 0.5, 1.5, 3.0, 4.0],
                      np.float32) * unit
    rows.append(wl.bf16_round(r))                  # exact midpoints when s_t is a power of two
    rows.append(wl.bf16_round(rng.standard_normal(512, dtype=np.float32) * np.float32(1e4)))   # scales saturate
    rows.append(wl.bf16_round(rng.standard_normal(512, dtype=np.float32) * np.float32(1e-4)))  # subnormal scales
    rows.append(wl.bf16_round(rng.standard_normal(512, dtype=np.float32) * np.float32(1e-7)))  # scales round to 0
    out = np.stack(rows)
    assert np.array_equal(wl.bf16_round(out), out), "special rows must be bf16 values"
    return out


@pytest.mark.parametrize("st", [2.0 ** -8, 0.0173])
@pytest.mark.parametrize("n_random", [0, 1000])
def test_kv_append_nvfp4_bit_exact(api, st, n_random):
    rng = np.random.default_rng(70 + n_random)
    c = np.concatenate([_special_rows(rng, st), wl.bf16_round(rng.standard_normal((n_random, 512),
                                                                                  dtype=np.float32))])
    n = c.shape[0]
    k = wl.bf16_round(rng.standard_normal((n, 64), dtype=np.float32))
    pages = (n + 63) // 64 + 1
    slots = rng.permutation(pages * 64)[:n].astype(np.int64)
    rows = torch.zeros((pages, 64, 416), dtype=torch.uint8, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_nvfp4(to_bf16(c, "cuda"), to_bf16(k, "cuda"), torch.from_numpy(slots).cuda(), rows, st, dev_err)
    assert api.mla_check(dev_err) == 0
    want = n4.append(n4.empty_cache(pages), c, k, slots, st).reshape(-1, 416)
    got = rows.cpu().numpy().reshape(-1, 416)
    bad = np.nonzero(np.any(got != want, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ; first slots {bad[:4]}"


@pytest.mark.parametrize("st", [2.0 ** -8, 0.0173])
def test_gather_nvfp4_bit_exact(api, st):
    rng = np.random.default_rng(75)
    c = np.concatenate([_special_rows(rng, st), wl.bf16_round(rng.standard_normal((200, 512), dtype=np.float32))])
    n = c.shape[0]
    k = wl.bf16_round(rng.standard_normal((n, 64), dtype=np.float32))
    pages = (n + 63) // 64
    bt = rng.permutation(pages).astype(np.int32)[None, :]
    slots = oracle.slot_mapping(bt, np.zeros(n, np.int32), np.arange(n))
    rows = torch.zeros((pages, 64, 416), dtype=torch.uint8, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_nvfp4(to_bf16(c, "cuda"), to_bf16(k, "cuda"), torch.from_numpy(slots).cuda(), rows, st, dev_err)
    out = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    api.mla_gather_paged_nvfp4(rows, st, torch.from_numpy(bt).cuda(), 0, n, out, dev_err)
    assert api.mla_check(dev_err) == 0
    lat, rope = n4.gather(n4.append(n4.empty_cache(pages), c, k, slots, st), bt, 0, n, st)
    want = np.concatenate([lat, rope], axis=1).astype(np.float32)
    assert np.array_equal(_bits(out), _bf16_bits_of(want))


def test_gather_nvfp4_every_code_and_block_scale(api):
    """Rows written by hand: every block holds all 16 codes; block scales run
    over subnormal, normal and the largest E4M3 values."""
    scale_codes = np.array([0x00, 0x01, 0x05, 0x08, 0x30, 0x38, 0x4F, 0x66, 0x7E], dtype=np.uint8)
    n = 9
    st = 0.0173
    host = np.zeros((1, 64, 416), dtype=np.uint8)
    rng = np.random.default_rng(76)
    for i in range(n):
        codes = np.tile(np.arange(16, dtype=np.uint8), 32)
        codes = codes.reshape(32, 16)[:, rng.permutation(16)].reshape(512)
        host[0, i, :256] = n4.pack_codes(codes[None, :])[0]
        host[0, i, 256:288] = np.roll(scale_codes, i).repeat(4)[:32]
        host[0, i, 288:] = rng.integers(0, 256, 128, dtype=np.uint8)
    rows = torch.from_numpy(host).cuda()
    out = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_gather_paged_nvfp4(rows, st, torch.zeros((1, 1), dtype=torch.int32, device="cuda"), 0, n, out, dev_err)
    assert api.mla_check(dev_err) == 0
    flat = host.reshape(-1, 416)[:n]
    lat = n4.dequantize_rows(n4.unpack_codes(flat[:, :256]), flat[:, 256:288], st).astype(np.float32)
    got = _bits(out)
    assert np.array_equal(got[:, :512], _bf16_bits_of(lat))
    assert np.array_equal(got[:, 512:].view(np.uint8).reshape(n, 128), flat[:, 288:])


def test_nvfp4_misaligned_rows_is_a_host_error(api):
    """The pages' misaligned-address fault becomes MLA_ERR_MISALIGNED on the host."""
    buf = torch.zeros(2 * 64 * 416 + 16, dtype=torch.uint8, device="cuda")
    bad = buf[8:8 + 2 * 64 * 416].view(2, 64, 416)
    assert bad.data_ptr() % 16 == 8
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((10, 576), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.MlaError) as e:
        api.mla_gather_paged_nvfp4(bad, 0.01, torch.zeros((1, 1), dtype=torch.int32, device="cuda"), 0, 10, out,
                                   dev_err)
    assert e.value.status == 2
    c = torch.ones((1, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.MlaError):
        api.mla_kv_append_nvfp4(c, k, torch.zeros(1, dtype=torch.int64, device="cuda"), bad, 0.01, dev_err)
    torch.cuda.synchronize()
    assert int(dev_err.item()) == 0


def test_nvfp4_errors(api):
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = torch.zeros((2, 64, 416), dtype=torch.uint8, device="cuda")
    c = torch.ones((2, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((2, 64), dtype=torch.bfloat16, device="cuda")
    api.mla_kv_append_nvfp4(c, k, torch.tensor([3, 128], dtype=torch.int64, device="cuda"), rows, 0.01, dev_err)
    assert int(dev_err.item()) == api.DEVERR_SLOT_OOB
    assert rows.view(-1, 416)[3].any() and not rows.view(-1, 416)[4].any()
    for bad_st in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(api.MlaError):
            api.mla_kv_append_nvfp4(c, k, torch.tensor([0, 1], dtype=torch.int64, device="cuda"), rows, bad_st,
                                    dev_err)
    dev_err.zero_()
    out = torch.empty((70, 576), dtype=torch.bfloat16, device="cuda")
    api.mla_gather_paged_nvfp4(rows, 0.01, torch.tensor([[0, 9]], dtype=torch.int32, device="cuda"), 0, 70, out,
                               dev_err)
    assert int(dev_err.item()) == api.DEVERR_PAGE_OOB


def _batch_case(api, st):
    case = wl.make_case([1, 64, 65, 300, 130], [1, 1, 1, 1, 1], seed=77)
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    rows = torch.zeros((case.num_pages, 64, 416), dtype=torch.uint8, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_nvfp4(to_bf16(case.c_kv, "cuda"), to_bf16(case.k_r, "cuda"), torch.from_numpy(slots).cuda(),
                            rows, st, dev_err)
    assert api.mla_check(dev_err) == 0
    cache = n4.append(n4.empty_cache(case.num_pages), case.c_kv, case.k_r, slots, st)
    return case, rows, cache


@pytest.mark.parametrize("st", [2.0 ** -8, 0.0173])
def test_gather_nvfp4_batch_bit_exact(api, st):
    """Sequences in any order, prefixes of any length (an empty one
    included), packed into one output by one launch: every bf16 bit equals
    the oracle's per-sequence gather."""
    case, rows, cache = _batch_case(api, st)
    picks = [(3, 300), (0, 1), (1, 0), (2, 65), (4, 100), (3, 17)]
    offs = np.concatenate([[0], np.cumsum([n for _, n in picks])]).astype(np.int64)
    total = int(offs[-1])
    out = torch.full((total, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_gather_paged_nvfp4_batch(rows, st, torch.from_numpy(case.block_table).cuda(),
                                     torch.tensor([s for s, _ in picks], dtype=torch.int32, device="cuda"),
                                     torch.from_numpy(offs).cuda(), out, dev_err)
    assert api.mla_check(dev_err) == 0
    got = _bits(out)
    for i, (sid, n) in enumerate(picks):
        if n == 0:
            continue
        lat, rope = n4.gather(cache, case.block_table, sid, n, st)
        want = np.concatenate([lat, rope], axis=1).astype(np.float32)
        assert np.array_equal(got[offs[i]:offs[i + 1]], _bf16_bits_of(want)), f"entry {i} (sequence {sid})"


def test_gather_nvfp4_batch_bad_entries(api):
    """A sequence id outside the block table and a prefix longer than the
    table's pages set MLA_DEVERR_BATCH and leave their rows untouched; the
    good entries are still gathered."""
    st = 2.0 ** -8
    case, rows, cache = _batch_case(api, st)
    max_pages = case.block_table.shape[1]
    assert int(case.seq_lens[3]) > 64 * (max_pages - 1)        # sequence 3 fills every table column
    picks = [(0, 1), (99, 10), (2, 65), (3, 64 * max_pages + 5)]
    offs = np.concatenate([[0], np.cumsum([n for _, n in picks])]).astype(np.int64)
    out = torch.full((int(offs[-1]), 576), 7.0, dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_gather_paged_nvfp4_batch(rows, st, torch.from_numpy(case.block_table).cuda(),
                                     torch.tensor([s for s, _ in picks], dtype=torch.int32, device="cuda"),
                                     torch.from_numpy(offs).cuda(), out, dev_err)
    assert int(dev_err.item()) == api.DEVERR_BATCH
    o = out.float().cpu().numpy()
    assert np.all(o[offs[1]:offs[2]] == 7.0)                       # bad sequence id: untouched
    assert np.all(o[offs[3] + 64 * max_pages:offs[4]] == 7.0)      # positions past the table: untouched
    got = _bits(out)
    for i in (0, 2):
        sid, n = picks[i]
        lat, rope = n4.gather(cache, case.block_table, sid, n, st)
        want = np.concatenate([lat, rope], axis=1).astype(np.float32)
        assert np.array_equal(got[offs[i]:offs[i + 1]], _bf16_bits_of(want))
