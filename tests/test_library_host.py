"""Host-side tests of libmla (no GPU): the library builds and loads, exports
every symbol include/mla.h declares, and its host logic (byte formula, page
pool, slot mapping, split planner, argument validation) is right."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
from mla_latent_kv_02_gb300 import _build, _lib
from mla_latent_kv_02_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def api():
    if _build.is_stale():
        _build.build()
    from mla_latent_kv_02_gb300 import api as a
    a.mla_version()
    return a


def header_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function(api):
    names = header_functions()
    assert len(names) >= 20
    h = C.CDLL(_lib.path())
    missing = [n for n in names if not hasattr(h, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_kv_bytes_matches_oracle(api):
    for args in [(60, 512, 64, 2, 1, 1), (1, 512, 64, 2, 64, 1), (60, 512, 64, 2, 131072, 1), (61, 512, 0, 1, 7, 3)]:
        assert api.mla_kv_bytes(*args) == oracle.kv_bytes(*args)


@pytest.mark.parametrize("args", [(0, 512, 64, 2, 1, 1), (60, 512, -1, 2, 1, 1), (60, 512, 64, 2, 0, 1),
                                  (60, 512, 64, 2, 1, 0), (2**40, 2**20, 0, 2**10, 2**10, 1)])
def test_kv_bytes_rejects_invalid(api, args):
    with pytest.raises(api.MlaError) as e:
        api.mla_kv_bytes(*args)
    assert e.value.status == 1


def test_config_default(api):
    c = api.mla_config_default()
    assert (c.num_heads, c.head_dim_c, c.latent_dim, c.rope_dim, c.page_size) == (128, 128, 512, 64, 64)
    assert abs(c.scale - 192 ** -0.5) < 1e-7
    lib = _lib.lib()
    assert lib.mla_config_validate(C.byref(c)) == 0
    c.page_size = 16
    assert lib.mla_config_validate(C.byref(c)) == 3


def test_pool_alloc_free(api):
    p = api.MlaPool(8)
    a = p.alloc(3)
    assert list(a) == [0, 1, 2] and p.available() == 5
    with pytest.raises(api.MlaError) as e:
        p.alloc(6)
    assert e.value.status == 7 and p.available() == 5
    p.free([1])
    assert list(p.alloc(2)) == [1, 3]
    with pytest.raises(api.MlaError):
        p.free([1, 1])          # repeated
    with pytest.raises(api.MlaError):
        p.free([7])             # not allocated
    with pytest.raises(api.MlaError):
        p.free([9])             # out of range
    assert p.available() == 4   # failed frees change nothing
    p.close()


def test_slot_mapping_matches_oracle(api):
    case = wl.make_case([1, 63, 64, 65, 700], [1, 1, 1, 2, 3], seed=3, with_weights=False)
    seq, pos = case.positions()
    got = api.mla_slot_mapping(case.block_table, seq, pos)
    assert np.array_equal(got, oracle.slot_mapping(case.block_table, seq, pos))


def test_slot_mapping_rejects_unmapped(api):
    bt = np.array([[3, -1]], dtype=np.int32)
    with pytest.raises(api.MlaError):
        api.mla_slot_mapping(bt, [0], [64])
    with pytest.raises(api.MlaError):
        api.mla_slot_mapping(bt, [1], [0])


def _plan_segments(buf, info):
    from mla_latent_kv_02_gb300.api import mla_decode_plan_bytes  # noqa: F401
    nc, ns, nsr = info.num_clusters, info.num_segments, info.num_split_rows
    seg_off = buf[16:16 + nc + 1]
    seg_base = (16 + nc + 1 + 7) // 8 * 8
    segs = buf[seg_base:seg_base + 8 * ns].reshape(ns, 8)
    split = buf[seg_base + 8 * ns: seg_base + 8 * ns + 4 * nsr].reshape(nsr, 4)
    return seg_off, segs, split


@pytest.mark.parametrize("seq_lens,q_lens,nc", [
    ([8194] * 64, [2] * 64, 76), ([65536] * 16, [1] * 16, 76), ([1024], [1], 76), ([1, 63, 64, 65], [1, 1, 1, 2], 3),
    ([16896] * 4, [512] * 4, 76), ([100, 200], [0, 2], 1)])
def test_planner_covers_every_tile_once(api, seq_lens, q_lens, nc):
    buf, info = api.mla_decode_plan_host(seq_lens, q_lens, nc)
    assert info.magic == 0x504C4D41 and buf[0] == np.int32(np.uint32(0x504C4D41).view(np.int32))
    seg_off, segs, split = _plan_segments(buf, info)
    rows = oracle.row_index(seq_lens, q_lens)
    assert info.T == len(rows)
    need = {t: (oracle.visible_tokens(seq_lens[b], q_lens[b], i) + 63) // 64 for t, b, i in rows}
    assert info.total_tiles == sum(need.values())
    covered = {t: [] for t in need}
    for s in segs:
        row, b, pb, pe, vis = s[:5]
        assert rows[row][1] == b and vis == oracle.visible_tokens(seq_lens[b], q_lens[b], rows[row][2])
        covered[row].extend(range(pb, pe))
    for t, n in need.items():
        assert sorted(covered[t]) == list(range(n)), t
    # contiguous, balanced ranges
    assert seg_off[0] == 0 and seg_off[-1] == info.num_segments and np.all(np.diff(seg_off) >= 1)
    per = [sum(int(s[3] - s[2]) for s in segs[seg_off[c]:seg_off[c + 1]]) for c in range(info.num_clusters)]
    assert info.num_clusters <= nc
    # Lanes (uniform multi-token decode): each cluster serves one in-sequence
    # row index; within a lane every cluster but the last holds the same count.
    lane_of = [{rows[int(s[0])][2] for s in segs[seg_off[c]:seg_off[c + 1]]} for c in range(info.num_clusters)]
    q = set(x for x in q_lens if x > 0)
    laned = len(q) == 1 and min(q) >= 2 and nc // min(q) >= 1
    if laned:
        assert all(len(l) == 1 for l in lane_of)
        lanes = [next(iter(l)) for l in lane_of]
        assert lanes == sorted(lanes)
        groups = [[per[c] for c in range(len(per)) if lanes[c] == j] for j in sorted(set(lanes))]
    else:
        groups = [per]
    for g in groups:
        assert max(g) - min(g[:-1] or g) <= 0
    # split rows: exactly the rows with several pieces, slots contiguous
    pieces = {}
    for s in segs:
        pieces.setdefault(int(s[0]), []).append(int(s[5]))
    multi = {r: p for r, p in pieces.items() if len(p) > 1}
    assert info.num_split_rows == len(multi) == split.shape[0]
    for row, s0, n, _ in split:
        assert multi[row] == list(range(s0, s0 + n))
    assert all(p == [-1] for r, p in pieces.items() if r not in multi)
    assert info.num_partials == sum(len(p) for p in multi.values())


def test_planner_lanes_align_the_rows_of_a_sequence(api):
    # Multi-token decode: cluster c of lane j reads the same pages of the same
    # sequences as cluster c of lane 0 (up to the one-tile difference between
    # the rows' visible lengths), so the rows of a sequence share page reads.
    seq_lens, q_lens, nc = [8194] * 64, [2] * 64, 76
    buf, info = api.mla_decode_plan_host(seq_lens, q_lens, nc)
    seg_off, segs, _ = _plan_segments(buf, info)
    rows = oracle.row_index(seq_lens, q_lens)
    lanes = {}
    for c in range(info.num_clusters):
        work = [(int(s[1]), p) for s in segs[seg_off[c]:seg_off[c + 1]] for p in range(int(s[2]), int(s[3]))]
        lane = rows[int(segs[seg_off[c]][0])][2]
        lanes.setdefault(lane, []).append(work)
    assert sorted(lanes) == [0, 1] and len(lanes[0]) == len(lanes[1]) == nc // 2
    for w0, w1 in zip(lanes[0], lanes[1]):
        assert w0 == w1


def test_planner_rejects_bad_lengths(api):
    with pytest.raises(api.MlaError):
        api.mla_decode_plan_host([0], [0], 4)
    with pytest.raises(api.MlaError):
        api.mla_decode_plan_host([5], [6], 4)
    with pytest.raises(api.MlaError):
        api.mla_decode_plan_host([5], [1], 0)


def test_plan_bytes_bound_holds(api):
    for seq_lens, q_lens in [([8194] * 64, [2] * 64), ([3] * 50, [3] * 50), ([10**6], [1])]:
        for nc in (1, 7, 76, 200):
            buf, info = api.mla_decode_plan_host(seq_lens, q_lens, nc)
            assert info.plan_bytes <= buf.nbytes
            assert api.mla_decode_workspace_size(nc) >= info.num_partials * (128 * 512 * 4 + 128 * 4)


def test_device_calls_validate_before_any_launch(api):
    """Arguments are rejected on the host before anything touches CUDA."""
    lib = _lib.lib()
    P = C.c_void_p
    ok = P(0x10000)
    odd = P(0x10008)
    err = P(0x20000)
    # null inputs
    assert lib.mla_kv_append(None, ok, ok, 1, ok, 4, err, None) == 1
    # misaligned bf16 pointer (16-byte rule)
    assert lib.mla_kv_append(odd, ok, ok, 1, ok, 4, err, None) == 2
    assert lib.mla_absorb_q(ok, odd, ok, 4, err, None) == 2
    assert lib.mla_up_v(ok, ok, None, 4, err, None) == 1
    assert lib.mla_cache_init(ok, 0, None) == 1
    # n == 0 / T == 0 are no-ops
    assert lib.mla_kv_append(None, None, None, 0, None, 0, None, None) == 0
    assert lib.mla_absorb_q(None, None, None, 0, None, None) == 0
    # decode: a zeroed info is not a plan
    info = _lib.mla_plan_info()
    assert lib.mla_decode_paged(ok, ok, ok, 4, ok, 4, ok, C.byref(info), C.c_float(0.07), ok, 1 << 20,
                                ok, None, err, None) == 1
    # decode: block table narrower than the plan needs; bad scale
    buf, pinfo = api.mla_decode_plan_host([700], [1], 4)
    assert lib.mla_decode_paged(ok, ok, ok, 64, ok, 2, ok, C.byref(pinfo), C.c_float(0.07), ok, 1 << 30,
                                ok, None, err, None) == 1
    assert lib.mla_decode_paged(ok, ok, ok, 64, ok, 11, ok, C.byref(pinfo), C.c_float(-1.0), ok, 1 << 30,
                                ok, None, err, None) == 1
    assert lib.mla_decode_paged(ok, odd, ok, 64, ok, 11, ok, C.byref(pinfo), C.c_float(0.07), ok, 1 << 30,
                                ok, None, err, None) == 2
    # workspace too small for the plan's partials
    buf, pinfo = api.mla_decode_plan_host([7000], [1], 8)
    assert pinfo.num_partials > 0
    assert lib.mla_decode_paged(ok, ok, ok, 200, ok, 110, ok, C.byref(pinfo), C.c_float(0.07), ok, 16,
                                ok, None, err, None) == 1
    assert "workspace" in lib.mla_last_error().decode()


def test_rope_calls_validate_before_any_launch(api):
    """RoPE entry points reject bad arguments on the host (nothing is enqueued)."""
    lib = _lib.lib()
    P = C.c_void_p
    ok = P(0x10000)
    odd8 = P(0x10004)    # 4-byte but not 8-byte aligned
    odd16 = P(0x10008)   # 8-byte but not 16-byte aligned
    err = P(0x20000)
    f = C.c_float
    # table: base must be finite and > 1; max_pos within [0, 2^24]; 0 rows is a no-op
    assert lib.mla_rope_table(16, f(1.0), ok, None) == 1
    assert lib.mla_rope_table(16, f(float("inf")), ok, None) == 1
    assert lib.mla_rope_table(16, f(float("nan")), ok, None) == 1
    assert lib.mla_rope_table((1 << 24) + 1, f(10000.0), ok, None) == 1
    assert lib.mla_rope_table(-1, f(10000.0), ok, None) == 1
    assert lib.mla_rope_table(16, f(10000.0), None, None) == 1
    assert lib.mla_rope_table(16, f(10000.0), odd8, None) == 2
    assert lib.mla_rope_table(16, f(10000.0), odd16, None) == 2
    assert lib.mla_rope_table(0, f(10000.0), None, None) == 0
    # append with rotation
    assert lib.mla_kv_append_rope(ok, ok, ok, ok, 64, ok, -1, ok, 4, err, None) == 1
    assert lib.mla_kv_append_rope(None, None, None, None, 0, None, 0, None, 0, None, None) == 0
    assert lib.mla_kv_append_rope(ok, ok, None, ok, 64, ok, 1, ok, 4, err, None) == 1
    assert lib.mla_kv_append_rope(ok, odd16, ok, ok, 64, ok, 1, ok, 4, err, None) == 2
    assert lib.mla_kv_append_rope(ok, ok, ok, odd8, 64, ok, 1, ok, 4, err, None) == 2
    assert lib.mla_rope_q(ok, ok, odd16, 64, P(0x90000), 1, err, None) == 2
    assert lib.mla_kv_append_rope(ok, ok, ok, ok, 0, ok, 1, ok, 4, err, None) == 1
    assert lib.mla_kv_append_rope(ok, ok, ok, ok, 64, ok, 1, ok, 0, err, None) == 1
    # query rotation: alignment, max_pos, overlap of input and output
    assert lib.mla_rope_q(None, None, None, 0, None, 0, None, None) == 0
    assert lib.mla_rope_q(ok, ok, ok, 64, ok, -1, err, None) == 1
    assert lib.mla_rope_q(odd16, ok, ok, 64, P(0x90000), 1, err, None) == 2
    assert lib.mla_rope_q(ok, ok, ok, 0, P(0x90000), 1, err, None) == 1
    assert lib.mla_rope_q(ok, ok, ok, 64, P(0x10000 + 16384 - 16), 1, err, None) == 1   # overlaps by 16 B
    assert "overlap" in lib.mla_last_error().decode()


def test_nvfp4_calls_validate_before_any_launch(api):
    lib = _lib.lib()
    P = C.c_void_p
    ok, odd, err = P(0x10000), P(0x10008), P(0x20000)
    f = C.c_float
    assert lib.mla_kv_append_nvfp4(None, None, None, 0, f(0.01), None, 0, None, None) == 0
    assert lib.mla_kv_append_nvfp4(ok, ok, ok, -1, f(0.01), ok, 4, err, None) == 1
    assert lib.mla_kv_append_nvfp4(ok, ok, ok, 1, f(0.0), ok, 4, err, None) == 1
    assert lib.mla_kv_append_nvfp4(ok, ok, ok, 1, f(float("nan")), ok, 4, err, None) == 1
    assert lib.mla_kv_append_nvfp4(ok, ok, ok, 1, f(0.01), odd, 4, err, None) == 2
    assert lib.mla_gather_paged_nvfp4(odd, f(0.01), 4, ok, 2, 0, 10, ok, err, None) == 2
    assert lib.mla_gather_paged_nvfp4(ok, f(0.01), 4, ok, 2, 0, 10, odd, err, None) == 2
    assert lib.mla_gather_paged_nvfp4(ok, f(0.01), 4, ok, 1, 0, 65, ok, err, None) == 1
    assert lib.mla_gather_paged_nvfp4(ok, f(-2.0), 4, ok, 2, 0, 10, ok, err, None) == 1
    assert lib.mla_gather_paged_nvfp4(None, f(0.01), 4, ok, 2, 0, 0, None, None, None) == 0
    # batched gather: rows, B, max_pages, seq_ids, out_offsets, nb, total, out
    g = lib.mla_gather_paged_nvfp4_batch
    assert g(None, f(0.01), 4, None, 1, 1, None, None, 0, 0, None, None, None) == 0
    assert g(ok, f(0.01), 4, ok, 2, 2, ok, ok, -1, 10, ok, err, None) == 1
    assert g(ok, f(0.01), 4, ok, 2, 2, ok, ok, 1, -10, ok, err, None) == 1
    assert g(ok, f(0.0), 4, ok, 2, 2, ok, ok, 1, 10, ok, err, None) == 1
    assert g(ok, f(0.01), 4, ok, 0, 2, ok, ok, 1, 10, ok, err, None) == 1
    assert g(ok, f(0.01), 4, ok, 2, 2, None, ok, 1, 10, ok, err, None) == 1
    assert g(odd, f(0.01), 4, ok, 2, 2, ok, ok, 1, 10, ok, err, None) == 2
    assert g(ok, f(0.01), 4, ok, 2, 2, ok, P(0x10004), 1, 10, ok, err, None) == 2
    assert g(ok, f(0.01), 4, ok, 2, 2, ok, ok, 1, 10, odd, err, None) == 2


def test_fp8_and_decompress_calls_validate_before_any_launch(api):
    lib = _lib.lib()
    P = C.c_void_p
    ok, odd, err = P(0x10000), P(0x10008), P(0x20000)
    f = C.c_float
    # FP8 decode: a zeroed info is not a plan; the scales pointer is required and 16-byte aligned
    info = _lib.mla_plan_info()
    assert lib.mla_decode_paged_fp8(ok, ok, ok, ok, 4, ok, 4, ok, C.byref(info), f(0.07), ok, 1 << 20, ok, None,
                                    err, None) == 1
    buf, pinfo = api.mla_decode_plan_host([700], [1], 4)
    assert lib.mla_decode_paged_fp8(ok, ok, ok, None, 64, ok, 11, ok, C.byref(pinfo), f(0.07), ok, 1 << 30, ok, None,
                                    err, None) == 1
    assert lib.mla_decode_paged_fp8(ok, ok, ok, odd, 64, ok, 11, ok, C.byref(pinfo), f(0.07), ok, 1 << 30, ok, None,
                                    err, None) == 2
    # FP8 append / gather
    assert lib.mla_kv_append_fp8(ok, ok, ok, 1, ok, odd, 4, err, None) == 2
    assert lib.mla_kv_append_fp8(ok, ok, ok, -1, ok, ok, 4, err, None) == 1
    assert lib.mla_gather_paged_fp8(ok, ok, 4, ok, 1, 0, 65, ok, err, None) == 1
    # expansion and prefill attention
    assert lib.mla_expand_kv(None, 0, None, None, None, None, None, None) == 0
    assert lib.mla_expand_kv(ok, -1, ok, ok, ok, ok, err, None) == 1
    assert lib.mla_expand_kv(ok, 10, ok, ok, odd, ok, err, None) == 2
    assert lib.mla_prefill_attention(ok, ok, 0, ok, ok, ok, 10, f(0.07), ok, err, None) == 0
    assert lib.mla_prefill_attention(ok, ok, 11, ok, ok, ok, 10, f(0.07), ok, err, None) == 1   # M > N
    assert lib.mla_prefill_attention(ok, ok, 5, ok, ok, ok, 10, f(-1.0), ok, err, None) == 1
    assert lib.mla_prefill_attention(ok, odd, 5, ok, ok, ok, 10, f(0.07), ok, err, None) == 2
    # the whole branch: M > N, short workspace
    ws = C.c_size_t()
    assert lib.mla_prefill_workspace_size(100, C.byref(ws)) == 0
    assert ws.value == (100 * 1152 + 15) // 16 * 16 + 2 * 100 * 128 * 128 * 2
    assert lib.mla_prefill_decompress(ok, ok, 60, ok, 4, ok, 2, 0, 50, ok, ok, f(0.07), ok, ws.value, ok, err,
                                      None) == 1
    assert lib.mla_prefill_decompress(ok, ok, 20, ok, 4, ok, 2, 0, 100, ok, ok, f(0.07), ok, 100, ok, err,
                                      None) == 1
    assert "workspace" in lib.mla_last_error().decode()
    assert lib.mla_branch_for(300) == 1 and lib.mla_branch_for(10) == 0 and lib.mla_prefill_threshold() == 256
