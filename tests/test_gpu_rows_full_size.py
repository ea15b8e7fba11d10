"""Full-size parity of the cache fills and gathers the bench times, on the
MTP decode workload (B64 x 8194 tokens, 524 416 cached rows), in the
bench's launch configuration: every token is written by one launch, and
sampled outputs are checked against the oracle one by one.

* fp32 RoPE fill: latent bit-exact, the rotated key within the bf16 bound;
* FP8 fill: codes and scales bit-exact;
* NVFP4 fill: codes and block scales bit-exact; the gather of a whole
  8 194-token sequence bit-exact, and of all 64 sequences in one batched
  launch on sampled rows.
"""
import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import to_bf16, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
f8, n4 = oracle.fp8_cache, oracle.nvfp4_cache


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from mla_latent_kv_02_gb300 import api as a
    a.mla_version()
    return a


@pytest.fixture(scope="module")
def full(api):
    case = wl.workload(2, with_weights=False)
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    d = dict(case=case, pos=pos, slots=slots,
             c=to_bf16(case.c_kv, "cuda"), k=to_bf16(case.k_r, "cuda"),
             slots_t=torch.from_numpy(slots).cuda(), pos_t=torch.from_numpy(pos).cuda(),
             pick=np.random.default_rng(5).choice(pos.size, size=1500, replace=False))
    return d


def test_rope_fill_full_size(api, full):
    case, n = full["case"], full["pos"].size
    max_pos = int(case.seq_lens.max())
    table = torch.empty((max_pos, 32, 2), dtype=torch.float32, device="cuda")
    api.mla_rope_table(max_pos, table)
    cache = torch.zeros((case.num_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_rope(full["c"], full["k"], full["pos_t"], table, full["slots_t"], cache, dev_err)
    assert api.mla_check(dev_err) == 0
    flat = cache.view(-1, 576)
    pick = full["pick"]
    got = to_np(flat[torch.from_numpy(full["slots"][pick]).cuda()]).astype(np.float64)
    assert np.array_equal(got[:, :512], case.c_kv[pick].astype(np.float64))
    ref = oracle.rope_apply(case.k_r[pick], full["pos"][pick])
    x = case.k_r[pick].astype(np.float64)
    slack = np.repeat(np.abs(x[:, 0::2]) + np.abs(x[:, 1::2]), 2, axis=1) * 2.0 ** -20
    assert np.all(np.abs(got[:, 512:] - ref) <= 2.0 ** -8 * np.abs(ref) + slack)
    assert n == 524416


def test_fp8_fill_full_size(api, full):
    case = full["case"]
    rows = torch.zeros((case.num_pages, 64, 640), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((case.num_pages, 64), dtype=torch.float32, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_fp8(full["c"], full["k"], full["slots_t"], rows, scales, dev_err)
    assert api.mla_check(dev_err) == 0
    pick = full["pick"]
    sl = torch.from_numpy(full["slots"][pick]).cuda()
    got_rows = rows.view(-1, 640)[sl].cpu().numpy()
    got_sc = scales.view(-1)[sl].cpu().numpy().astype(np.float64)
    codes, sc = f8.quantize_rows(case.c_kv[pick])
    assert np.array_equal(got_rows[:, :512], codes)
    assert np.array_equal(got_rows[:, 512:], f8.bf16_bytes(case.k_r[pick]))
    assert np.array_equal(got_sc, sc)


def test_nvfp4_fill_and_gather_full_size(api, full):
    case = full["case"]
    st = 2.0 ** -8
    rows = torch.zeros((case.num_pages, 64, 416), dtype=torch.uint8, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_kv_append_nvfp4(full["c"], full["k"], full["slots_t"], rows, st, dev_err)
    assert api.mla_check(dev_err) == 0
    pick = full["pick"]
    got = rows.view(-1, 416)[torch.from_numpy(full["slots"][pick]).cuda()].cpu().numpy()
    codes, sb = n4.quantize_rows(case.c_kv[pick], st)
    assert np.array_equal(got[:, :256], n4.pack_codes(codes))
    assert np.array_equal(got[:, 256:288], sb)
    # gather sequence 37 whole, bit for bit
    b = 37
    n = int(case.seq_lens[b])
    out = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    api.mla_gather_paged_nvfp4(rows, st, torch.from_numpy(case.block_table).cuda(), b, n, out, dev_err)
    assert api.mla_check(dev_err) == 0
    off = int(case.tok_off[b])
    c2, s2 = n4.quantize_rows(case.c_kv[off:off + n], st)
    want = np.concatenate([n4.dequantize_rows(c2, s2, st), case.k_r[off:off + n].astype(np.float64)], axis=1)
    want_bits = (np.ascontiguousarray(want, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().astype(np.uint16), want_bits)
    del out
    # every sequence whole in one batched launch (the bench's launch); sampled rows bit for bit
    lens = case.seq_lens.astype(np.int64)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    allout = torch.empty((int(offs[-1]), 576), dtype=torch.bfloat16, device="cuda")
    api.mla_gather_paged_nvfp4_batch(rows, st, torch.from_numpy(case.block_table).cuda(),
                                     torch.arange(case.B, dtype=torch.int32, device="cuda"),
                                     torch.from_numpy(offs).cuda(), allout, dev_err)
    assert api.mla_check(dev_err) == 0
    g = np.sort(np.random.default_rng(6).choice(int(offs[-1]), size=1500, replace=False))
    seq_of = np.searchsorted(offs, g, side="right") - 1
    tok = case.tok_off[seq_of] + (g - offs[seq_of])          # the token's row in the case's inputs
    c3, s3 = n4.quantize_rows(case.c_kv[tok], st)
    want = np.concatenate([n4.dequantize_rows(c3, s3, st), case.k_r[tok].astype(np.float64)], axis=1)
    want_bits = (np.ascontiguousarray(want, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = allout[torch.from_numpy(g).cuda()].view(torch.int16).cpu().numpy().astype(np.uint16)
    assert np.array_equal(got, want_bits)
