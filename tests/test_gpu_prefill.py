"""GPU parity of the decompress branch (path A of the "Tearing open DeepSeek
MLA source" page, §4; the 256-token threshold of its §3) against the oracle:
the expansion K_c = c·W_UK^T, V_c = c·W_UV, and the causal attention over the
expanded cache, whose output must equal the absorbed path's out (steps
A2-A5) within the floating tolerance.  Cases span several query tiles, a
ragged last tile, N not a multiple of 128, a chunk that fills the whole
cache, a mixed batch dispatched per sequence, and the full-size chunked
prefill workload on sampled rows.
"""
import math

import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

from _helpers import DeviceCase, assert_close, to_bf16, to_np

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


def test_branch_threshold(api):
    assert api.mla_prefill_threshold() == 256
    assert api.mla_branch_for(255) == 0 and api.mla_branch_for(256) == 1 and api.mla_branch_for(1) == 0


@pytest.mark.parametrize("n", [1, 130, 256, 257, 300, 2600])
def test_expand_kv(api, n):
    case = wl.make_case([n], [1], seed=80 + n)
    rows = torch.cat([to_bf16(case.c_kv, "cuda"), to_bf16(case.k_r, "cuda")], dim=1).contiguous()
    # one buffer [K_c | V_c | guard]: the stores of a ragged last tile must stay inside each head's n rows
    buf = torch.full((2 * 128 * n * 128 + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    k_c = buf[:128 * n * 128].view(128, n, 128)
    v_c = buf[128 * n * 128:2 * 128 * n * 128].view(128, n, 128)
    k_c.fill_(float("nan"))
    v_c.fill_(float("nan"))
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_expand_kv(rows, to_bf16(case.w_uk, "cuda"), to_bf16(case.w_uv, "cuda"), k_c, v_c, dev_err)
    assert api.mla_check(dev_err) == 0
    assert bool((buf[2 * 128 * n * 128:] == 7.0).all()), "a store wrote past V_c"
    rk, rv = oracle.expand_kv(case.c_kv, case.w_uk, case.w_uv)
    assert_close(to_np(k_c), rk.transpose(1, 0, 2), f"K_c n={n}")   # head-major on the device
    assert_close(to_np(v_c), rv.transpose(1, 0, 2), f"V_c n={n}")


def _decompress(api, case, dc, b):
    """Run the branch for sequence b of a device case; returns out [q_len, 128, 128]."""
    n, q = int(case.seq_lens[b]), int(case.q_lens[b])
    r0 = int(case.q_start[b])
    ws = torch.empty(api.mla_prefill_workspace_size(n), dtype=torch.uint8, device="cuda")
    out = torch.full((q, 128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.mla_prefill_decompress(dc.q_c[r0:r0 + q], dc.q_r[r0:r0 + q], dc.kv_cache, dc.block_table, b, n, dc.w_uk,
                               dc.w_uv, ws, out, dc.dev_err)
    assert api.mla_check(dc.dev_err) == 0
    return out


@pytest.mark.parametrize("seq,q", [(300, 260), (700, 300), (300, 300), (1000, 512)])
def test_decompress_matches_the_absorbed_oracle(api, seq, q):
    case = wl.make_case([seq], [q], seed=90 + q)
    dc = DeviceCase(case)
    out = _decompress(api, case, dc, 0)
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, oracle.append(
        np.zeros((case.num_pages, 64, 576)), case.c_kv, case.k_r,
        oracle.slot_mapping(case.block_table, *case.positions())), case.block_table, case.seq_lens, case.q_lens,
        SCALE)
    assert_close(to_np(out), ref["out"], f"decompress out seq={seq} q={q}")


@pytest.mark.parametrize("seq,q", [(600, 256), (900, 768), (1100, 1024)])
def test_decompress_many_query_tiles(api, seq, q):
    """2, 6 and 8 query tiles of 128 rows per head, each with its own causal
    key range; the first and last row of every tile against the oracle."""
    case = wl.make_case([seq], [q], seed=70 + q)
    dc = DeviceCase(case)
    got = to_np(_decompress(api, case, dc, 0))
    assert np.all(np.isfinite(got))
    rows = sorted({r for t in range(0, q, 128) for r in (t, min(t + 127, q - 1))} | {q - 1})
    cache = oracle.append(np.zeros((case.num_pages, 64, 576), dtype=np.float32), case.c_kv, case.k_r,
                          oracle.slot_mapping(case.block_table, *case.positions()))
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, cache, case.block_table, case.seq_lens,
                          case.q_lens, SCALE, rows=rows)
    assert_close(got[rows], ref["out"][rows], f"decompress out seq={seq} q={q}")


def test_decompress_equals_path_a_rows(api):
    """A few rows against the oracle's own path A (decompress, then attend)."""
    case = wl.make_case([400], [270], seed=97)
    dc = DeviceCase(case)
    got = to_np(_decompress(api, case, dc, 0))
    for i in (0, 127, 128, 269):
        n = oracle.visible_tokens(400, 270, i)
        ref, _ = oracle.naive_attention_row(case.q_c[i], case.q_r[i], case.c_kv[:n], case.k_r[:n], case.w_uk,
                                            case.w_uv, SCALE)
        assert_close(got[i], ref, f"row {i}")


def test_mixed_batch_dispatch(api):
    """q_lens 1, 2, 300: the first two sequences go through A2-A5, the third
    through the decompress branch; together they give the oracle's out."""
    case = wl.make_case([200, 150, 600], [1, 2, 300], seed=98)
    dc = DeviceCase(case)
    T = case.T
    out = torch.full((T, 128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    absorbed = [b for b in range(case.B) if api.mla_branch_for(int(case.q_lens[b])) == 0]
    assert absorbed == [0, 1]
    q_abs = torch.empty((T, 128, 512), dtype=torch.bfloat16, device="cuda")
    api.mla_absorb_q(dc.q_c, dc.w_uk, q_abs, dc.dev_err)
    sub = wl.make_case([200, 150], [1, 2], seed=98)       # the absorbed sequences' plan
    o_lat = torch.empty((3, 128, 512), dtype=torch.bfloat16, device="cuda")
    plan = api.mla_decode_plan(sub.seq_lens, sub.q_lens)
    api.mla_decode_paged(q_abs[:3], dc.q_r[:3], dc.kv_cache, dc.block_table[:2], plan, o_lat, dc.dev_err)
    api.mla_up_v(o_lat, dc.w_uv, out[:3], dc.dev_err)
    out[3:] = _decompress(api, case, dc, 2)
    assert api.mla_check(dc.dev_err) == 0
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, oracle.append(
        np.zeros((case.num_pages, 64, 576)), case.c_kv, case.k_r,
        oracle.slot_mapping(case.block_table, *case.positions())), case.block_table, case.seq_lens, case.q_lens,
        SCALE)
    assert_close(to_np(out), ref["out"], "mixed batch out")


def test_decompress_full_size_chunked_prefill_sampled_rows(api):
    """B4 x (16384 cached + 512-token chunk), every sequence through the
    decompress branch (the bench's launch configuration); sampled rows against
    the oracle (the absorbed form, pinned equal to path A)."""
    case = wl.workload(4)
    dc = DeviceCase(case)
    rng = np.random.default_rng(99)
    got = np.empty((case.T, 128, 128))
    for b in range(case.B):
        r0 = int(case.q_start[b])
        got[r0:r0 + 512] = to_np(_decompress(api, case, dc, b))
    assert np.all(np.isfinite(got))
    rows = sorted({0, 511, 512 + 300, case.T - 1} | {int(x) for x in rng.choice(case.T, size=3, replace=False)})
    cache = oracle.append(np.zeros((case.num_pages, 64, 576), dtype=np.float32), case.c_kv, case.k_r,
                          oracle.slot_mapping(case.block_table, *case.positions()))
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, cache, case.block_table, case.seq_lens,
                          case.q_lens, SCALE, rows=rows)
    assert_close(got[rows], ref["out"][rows], "chunked prefill decompress out")


def test_decompress_rejects_bad_arguments(api):
    case = wl.make_case([100], [50], seed=91)
    dc = DeviceCase(case)
    ws = torch.empty(api.mla_prefill_workspace_size(100), dtype=torch.uint8, device="cuda")
    out = torch.empty((50, 128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.MlaError):          # M > N
        api.mla_prefill_decompress(dc.q_c, dc.q_r, dc.kv_cache, dc.block_table, 0, 40, dc.w_uk, dc.w_uv, ws, out,
                                   dc.dev_err)
    with pytest.raises(api.MlaError):          # workspace too small
        api.mla_prefill_decompress(dc.q_c, dc.q_r, dc.kv_cache, dc.block_table, 0, 100, dc.w_uk, dc.w_uv, ws[:100],
                                   out, dc.dev_err)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0


def _decompress_batch(api, case, dc, seqs):
    """The branch for the sequences `seqs` of a device case in one batched call;
    returns out [T, 128, 128] with the chunks' rows written (others NaN)."""
    n = [int(case.seq_lens[b]) for b in seqs]
    ws = torch.empty(api.mla_prefill_batch_workspace_size(n), dtype=torch.uint8, device="cuda")
    out = torch.full((case.T, 128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.mla_prefill_decompress_batch(dc.q_c, dc.q_r, dc.kv_cache, dc.block_table, seqs,
                                     [int(case.q_start[b]) for b in seqs], [int(case.q_lens[b]) for b in seqs], n,
                                     dc.w_uk, dc.w_uv, ws, out, dc.dev_err)
    assert api.mla_check(dc.dev_err) == 0
    return out


def test_decompress_batch_equals_per_sequence_calls(api):
    """Three qualifying sequences of different lengths (several query tiles,
    ragged tiles, a chunk that fills its cache) around an absorbed one: the
    batched call (one gather, one expansion, one attention launch over the
    packed arrays) gives, row for row, the bits of one call per sequence,
    writes nothing else, and matches the oracle on sampled rows."""
    case = wl.make_case([700, 200, 300, 1000], [300, 1, 300, 512], seed=101)
    dc = DeviceCase(case)
    seqs = [b for b in range(case.B) if api.mla_branch_for(int(case.q_lens[b])) == 1]
    assert seqs == [0, 2, 3]
    got = _decompress_batch(api, case, dc, seqs)
    for b in seqs:
        r0, q = int(case.q_start[b]), int(case.q_lens[b])
        one = _decompress(api, case, dc, b)
        assert torch.equal(got[r0:r0 + q], one), f"sequence {b}"
    absorbed_rows = int(case.q_start[1])
    assert torch.isnan(got[absorbed_rows].float()).all(), "the batched call wrote an absorbed sequence's row"
    rows = sorted({0, 299, 300 + 1, 301 + 150, 601, 601 + 255, 601 + 256, case.T - 1})
    cache = oracle.append(np.zeros((case.num_pages, 64, 576), dtype=np.float32), case.c_kv, case.k_r,
                          oracle.slot_mapping(case.block_table, *case.positions()))
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, cache, case.block_table, case.seq_lens,
                          case.q_lens, SCALE, rows=rows)
    assert_close(to_np(got)[rows], ref["out"][rows], "batched decompress out")


def test_decompress_batch_full_size_chunked_prefill(api):
    """The chunked-prefill workload (B4 x (16384 + 512)) through one batched
    call: the same bits as the per-sequence calls, and sampled rows against
    the oracle."""
    case = wl.workload(4)
    dc = DeviceCase(case)
    got = _decompress_batch(api, case, dc, list(range(case.B)))
    for b in (0, case.B - 1):
        r0 = int(case.q_start[b])
        assert torch.equal(got[r0:r0 + 512], _decompress(api, case, dc, b)), f"sequence {b}"
    rows = [3, 700, 1300, case.T - 2]
    cache = oracle.append(np.zeros((case.num_pages, 64, 576), dtype=np.float32), case.c_kv, case.k_r,
                          oracle.slot_mapping(case.block_table, *case.positions()))
    ref = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, cache, case.block_table, case.seq_lens,
                          case.q_lens, SCALE, rows=rows)
    assert_close(to_np(got)[rows], ref["out"][rows], "batched chunked prefill out")


def test_decompress_batch_rejects_bad_arguments(api):
    case = wl.make_case([300, 300], [260, 260], seed=102)
    dc = DeviceCase(case)
    ws = torch.empty(api.mla_prefill_batch_workspace_size([300, 300]), dtype=torch.uint8, device="cuda")
    out = torch.empty((case.T, 128, 128), dtype=torch.bfloat16, device="cuda")
    ok = dict(seq_ids=[0, 1], q_starts=[0, 260], q_lens=[260, 260], n_tokens=[300, 300])

    def call(**kw):
        a = dict(ok, **kw)
        api.mla_prefill_decompress_batch(dc.q_c, dc.q_r, dc.kv_cache, dc.block_table, a["seq_ids"], a["q_starts"],
                                         a["q_lens"], a["n_tokens"], dc.w_uk, dc.w_uv, a.get("ws", ws), out,
                                         dc.dev_err)

    for bad in (dict(seq_ids=[0, 2]), dict(q_lens=[301, 260]), dict(q_lens=[0, 260]), dict(n_tokens=[300, 5000]),
                dict(q_starts=[-1, 260]), dict(ws=ws[:1024])):
        with pytest.raises(api.MlaError):
            call(**bad)
    with pytest.raises(api.MlaError):
        api.mla_prefill_batch_workspace_size([10] * 65)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
