#!/usr/bin/env python3
"""Benchmark of the absorbed paged MLA decode path on GB300.

One step = one pass of the whole hot path over one batch:
  A1 mla_kv_append (this step's new tokens) -> A2 mla_absorb_q ->
  A3+A4 mla_decode_paged (split-KV + combine) -> A5 mla_up_v.

Default workload: MTP-style decode, batch 64, 8192 cached tokens + 2 query
tokens per sequence (128 query rows), 128 heads, d_c 512, d_r 64, page 64,
random page tables, seed 0.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2] [--impl mla|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_latent_kv_02_gb300 import workloads as wl  # noqa: E402

E2E_SLOTS = 2     # steps in flight in the end-to-end loop (3 measured the same)
METRIC = "MLA decode tokens/s and achieved KV HBM TB/s (% roofline), B=64 ctx 8K"
SCALE = 1.0 / math.sqrt(192)
FLOPS_PER_VISIBLE = 128 * (2 * 576 + 2 * 512)   # per (query row, visible token), all heads


def workload_stats(case):
    """Algorithmic work of one decode step (A3): flops and bytes."""
    visible = 0
    for b in range(case.B):
        n, q = int(case.seq_lens[b]), int(case.q_lens[b])
        visible += sum(n - q + i + 1 for i in range(q))
    kv_tokens = int(case.seq_lens[case.q_lens > 0].astype(np.int64).sum())
    T = case.T
    flops = visible * FLOPS_PER_VISIBLE
    bytes_ = kv_tokens * 1152 + T * 128 * 576 * 2 + T * 128 * 512 * 2
    return dict(T=T, visible=visible, kv_tokens=kv_tokens, flops=flops, bytes=bytes_,
                kv_bytes=kv_tokens * 1152)


# DRAM traffic (read + write) per decode launch from an ncu capture, keyed by
# the sha1 prefix of the decode kernel source it was taken on and the
# workload.  Captured at half batch and scaled by the query rows (see
# profiles/decode_kernel_mtp2_b32_ncu.md); any other source reads as null.
MEASURED_TRAFFIC = {("86c8047d28f0", 2): 664.54e6}


def decode_traffic(workload: int, batch):
    import hashlib
    src = os.path.join(ROOT, "mla_latent_kv_02_gb300", "csrc", "decode_paged.cu")
    try:
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()[:12]
    except OSError:
        return None
    if batch is not None:
        return None
    return MEASURED_TRAFFIC.get((sha, workload))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int, device=None) -> float:
    """Max of a float over all ranks (identity when not distributed)."""
    if ws <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}",
                 "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 5:
                continue
            try:
                s, m = float(parts[1]), float(parts[2])
                r = int(parts[4], 16)
            except ValueError:
                continue
            sm.append(s)
            mx.append(m)
            for bit, name in REASON_BITS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle baseline
def cpu_baseline(case, budget_s: float, max_rows: int = 128, check=None):
    """The oracle as it stands on a bounded sample of rows of the same workload.

    check: the timed GPU step's outputs on some rows ({rows, split, o_lat,
    out, lse}); those rows are computed first and compared with it (the
    parity of the timed run, with the tolerances of the parity tests)."""
    import oracle  # test infrastructure: only the CPU-baseline leg imports it
    t0 = time.perf_counter()
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    cache = oracle.append(np.zeros((case.num_pages, 64, 576), dtype=np.float32), case.c_kv, case.k_r, slots)
    setup = time.perf_counter() - t0
    first = list(check["rows"]) if check else []
    order = first + [r for r in range(case.T) if r not in set(first)]
    ref = {}
    rows_done = 0
    t1 = time.perf_counter()
    while rows_done < min(max(max_rows, len(first)), case.T):
        r = order[rows_done]
        res = oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, cache, case.block_table,
                              case.seq_lens, case.q_lens, SCALE, rows=[r])
        if r in first:
            ref[r] = (res["o_lat"][r], res["out"][r], res["lse"][r])
        rows_done += 1
        if time.perf_counter() - t1 > budget_s and rows_done >= len(first):
            break
    el = time.perf_counter() - t1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    blas = None
    try:
        from threadpoolctl import threadpool_info
        blas = sum(int(x.get("num_threads", 0)) for x in threadpool_info() if x.get("user_api") == "blas") or None
    except Exception:
        pass
    out = dict(value=rows_done / el, unit="tokens/s", cores=int(blas or cores), kind="oracle",
               sample=f"{rows_done} of {case.T} query rows (A2+A3+A5 in float64 NumPy, all 128 heads); "
                      f"cache placement {setup:.1f}s untimed", seconds=el)
    if check:
        def stats(gpu, want):
            d = np.abs(np.asarray(gpu, dtype=np.float64) - want)
            return dict(max_err_frac=float(d.max() / max(np.abs(want).max(), 1e-300)),
                        mean_rel=float(d.sum() / max(np.abs(want).sum(), 1e-300)))
        rows = list(check["rows"])
        par = dict(rows=rows, split_rows_checked=sorted(set(rows) & set(check["split"])),
                   o_lat=stats(check["o_lat"], np.stack([ref[r][0] for r in rows])),
                   out=stats(check["out"], np.stack([ref[r][1] for r in rows])),
                   lse=stats(check["lse"], np.stack([ref[r][2] for r in rows])),
                   tolerance="max|err| <= 2e-2 max|ref| and sum|err|/sum|ref| <= 5e-3 (o_lat, out); "
                             "2e-3 and 5e-4 (lse)")
        par["passed"] = bool(all(par[x]["max_err_frac"] <= 2e-2 and par[x]["mean_rel"] <= 5e-3
                                 for x in ("o_lat", "out"))
                             and par["lse"]["max_err_frac"] <= 2e-3 and par["lse"]["mean_rel"] <= 5e-4)
        out["parity"] = par
    return out


# ------------------------------------------------------------------ GPU arm
def _time_launches(torch, stream, fn, reps=5, warmup=3, per_rep=1):
    """Average device time (us) of one fn() launch: `reps` launches back to
    back between two CUDA events on `stream`, queued behind a short device
    sleep so that host-side call overhead leaves no gaps between them."""
    for i in range(warmup):
        fn(i)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000 + 60_000 * reps * per_rep)   # ~30 us of queue time per launch at 2 GHz
    a.record(stream)
    for i in range(reps):
        fn(i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps * 1e3


def measure_rows(api, torch, dev, stream, case, c_old, k_old, slots_old, pos_old, q_r, kv, dev_err, hbm_gbs,
                 plan=None, q_abs=None, st=None, peaks=None):
    """HBM-bound kernels outside the timed step, each timed alone (outside the
    step's timed region; inputs larger than L2): the bulk cache fill (A1 over
    the whole context), the same fill with the RoPE key rotated on the way in,
    the query RoPE rotation for this step's rows and for a prefill-sized block
    of rows, the quantising FP8 fill and the decode step over the FP8 cache.
    Algorithmic bytes: every operand read once, every output written once; a
    RoPE table row is counted once per distinct position."""
    n = int(c_old.shape[0])
    max_pos = int(case.seq_lens.max())
    table = torch.empty((max_pos, 32, 2), dtype=torch.float32, device=dev)
    api.mla_rope_table(max_pos, table)
    d_pos = torch.from_numpy(np.ascontiguousarray(pos_old, dtype=np.int32)).to(dev)
    distinct = int(np.unique(pos_old).size)
    out = {}

    def entry(name, us, nbytes, **extra):
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = dict(us=round(us, 2), bytes=int(nbytes), gbs=round(gbs, 1), peak=hbm_gbs,
                         frac=round(gbs / hbm_gbs, 4), **extra)

    us = _time_launches(torch, stream, lambda i: api.mla_kv_append(c_old, k_old, slots_old, kv, dev_err))
    entry("kv_append_bulk", us, n * (1152 + 8 + 1152), tokens=n)
    us = _time_launches(torch, stream, lambda i: api.mla_kv_append_rope(c_old, k_old, d_pos, table, slots_old, kv,
                                                                          dev_err))
    entry("kv_append_rope_bulk", us, n * (1152 + 8 + 4 + 1152) + distinct * 256, tokens=n)
    # this step's query rows: cycle through copies that together exceed L2
    qpos = torch.from_numpy(case.query_positions()).to(dev)
    T = int(q_r.shape[0])
    copies = max(2, -(-(256 << 20) // (2 * q_r.numel() * 2)))
    q_in = q_r.unsqueeze(0).repeat(copies, 1, 1, 1)
    q_out = torch.empty_like(q_in)
    us = _time_launches(torch, stream, lambda i: api.mla_rope_q(q_in[i % copies], qpos, table, q_out[i % copies],
                                                                  dev_err), reps=copies)
    entry("rope_q_step", us, T * (128 * 128 * 2 + 4) + int(np.unique(case.query_positions()).size) * 256,
          rows=T * 128, l2="%d input copies cycled (%.0f MB)" % (copies, 2 * q_in.numel() * 2 / 2 ** 20))
    del q_in, q_out
    Tp = 8192
    qp = torch.randn((Tp, 128, 64), generator=torch.Generator(device=dev).manual_seed(5), device=dev).to(
        torch.bfloat16)
    pp = torch.arange(Tp, dtype=torch.int32, device=dev) % max_pos
    qo = torch.empty_like(qp)
    us = _time_launches(torch, stream, lambda i: api.mla_rope_q(qp, pp, table, qo, dev_err))
    entry("rope_q_prefill8192", us, Tp * (128 * 128 * 2 + 4) + min(Tp, max_pos) * 256, rows=Tp * 128)
    del qp, qo
    if plan is not None:
        # FP8 (E4M3) cache: quantising fill of the whole context, then the
        # decode step over it (the same plan), against the same roofline as
        # the bf16 decode: flops unchanged, KV bytes 644 per token.
        rows = torch.empty((case.num_pages, 64, 640), dtype=torch.uint8, device=dev)
        scales = torch.ones((case.num_pages, 64), dtype=torch.float32, device=dev)
        rows.zero_()
        us = _time_launches(torch, stream, lambda i: api.mla_kv_append_fp8(c_old, k_old, slots_old, rows, scales,
                                                                             dev_err))
        entry("kv_append_fp8_bulk", us, n * (1152 + 8 + 644), tokens=n)
        new_idx = case.new_token_index()
        seq, pos = case.positions()
        slots_new = torch.from_numpy(api.mla_slot_mapping(case.block_table, seq, pos)[new_idx]).to(dev)
        c_new = torch.from_numpy(np.ascontiguousarray(case.c_kv[new_idx])).to(device=dev, dtype=torch.bfloat16)
        k_new = torch.from_numpy(np.ascontiguousarray(case.k_r[new_idx])).to(device=dev, dtype=torch.bfloat16)
        api.mla_kv_append_fp8(c_new, k_new, slots_new, rows, scales, dev_err)
        bt = torch.from_numpy(case.block_table).to(dev)
        o8 = torch.empty((q_abs.shape[0], 128, 512), dtype=torch.bfloat16, device=dev)
        l8 = torch.empty((q_abs.shape[0], 128), dtype=torch.float32, device=dev)
        us = _time_launches(torch, stream, lambda i: api.mla_decode_paged_fp8(q_abs, q_r, rows, scales, bt, plan, o8,
                                                                               dev_err, lse=l8, scale=SCALE))
        fbytes = st["kv_tokens"] * 644 + st["T"] * 128 * (576 + 512) * 2
        t_f = st["flops"] / (peaks["bf16_tflops"] * 1e12)
        t_b = fbytes / (peaks["hbm_gbs"] * 1e9)
        tf = st["flops"] / (us * 1e-6) / 1e12
        out["decode_paged_fp8"] = dict(us=round(us, 2), bytes=int(fbytes), gbs=round(fbytes / (us * 1e-6) / 1e9, 1),
                                       tflops=round(tf, 1), bound="tensor" if t_f >= t_b else "hbm",
                                       frac=round(max(t_f, t_b) / (us * 1e-6), 4),
                                       peak_source=peaks["source"] + " (burst)")
        del rows, scales
        # NVFP4 cache (E2M1 codes, E4M3 block scales, fp32 tensor scale):
        # quantising fill of the whole context, then the dequantising gather
        # of every sequence, as B launches queued back to back and as one
        # batched launch; 416 B read and 1152 B written per token.
        st_nv = 2.0 ** -8
        rows4 = torch.zeros((case.num_pages, 64, 416), dtype=torch.uint8, device=dev)
        us = _time_launches(torch, stream, lambda i: api.mla_kv_append_nvfp4(c_old, k_old, slots_old, rows4, st_nv,
                                                                               dev_err))
        entry("kv_append_nvfp4_bulk", us, n * (1152 + 8 + 416), tokens=n)
        gl = [int(x) for x in case.seq_lens]
        outs = [torch.empty((m, 576), dtype=torch.bfloat16, device=dev) for m in gl]

        def gather_all(i):
            for b2, m in enumerate(gl):
                api.mla_gather_paged_nvfp4(rows4, st_nv, bt, b2, m, outs[b2], dev_err)

        us = _time_launches(torch, stream, gather_all, reps=3, warmup=2, per_rep=len(gl))
        tot = sum(gl)
        gbytes = tot * (416 + 1152) + sum((m + 63) // 64 * 4 for m in gl)
        entry("gather_nvfp4_per_sequence", us, gbytes, tokens=tot, launches=len(gl))
        # the same gather of every sequence as one batched launch into a packed output
        del outs
        offs = torch.from_numpy(np.concatenate([[0], np.cumsum(gl)]).astype(np.int64)).to(dev)
        sids = torch.arange(len(gl), dtype=torch.int32, device=dev)
        packed = torch.empty((tot, 576), dtype=torch.bfloat16, device=dev)
        us = _time_launches(torch, stream, lambda i: api.mla_gather_paged_nvfp4_batch(rows4, st_nv, bt, sids, offs,
                                                                                      packed, dev_err))
        entry("gather_nvfp4_batch", us, gbytes + len(gl) * 12, tokens=tot, launches=1)
        del rows4, packed
    if api.mla_check(dev_err) != 0:
        raise RuntimeError("device error word set while timing the cache-fill, RoPE and FP8 kernels")
    # put the unrotated keys back (the cache holds them for the step above)
    api.mla_kv_append(c_old, k_old, slots_old, kv, dev_err)
    return out


def measure_decompress(api, torch, dev, stream, peaks):
    """The decompress branch on its own workload (B4 x 16384 cached + a
    512-token chunk, q_len >= the 256-token threshold): per-kernel times of
    one sequence (gather, K/V expansion, attention), the whole branch for the
    batch in one batched call, and steps A2-A5 of the absorbed path on the
    same inputs."""
    case = wl.workload(4, seed=0)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device=dev, dtype=torch.bfloat16)

    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = torch.empty((case.num_pages, 64, 576), dtype=torch.bfloat16, device=dev)
    seq, pos = case.positions()
    api.mla_kv_append(bf(case.c_kv), bf(case.k_r), torch.from_numpy(api.mla_slot_mapping(case.block_table, seq, pos)).to(dev),
                      kv, err)
    bt = torch.from_numpy(case.block_table).to(dev)
    q_c, q_r, w_uk, w_uv = bf(case.q_c), bf(case.q_r), bf(case.w_uk), bf(case.w_uv)
    T, N, M = case.T, int(case.seq_lens[0]), int(case.q_lens[0])
    ws = torch.empty(api.mla_prefill_workspace_size(N), dtype=torch.uint8, device=dev)
    rows = ws[:N * 1152].view(torch.bfloat16).view(N, 576)
    k_c = ws[N * 1152:N * 1152 + N * 32768].view(torch.bfloat16).view(128, N, 128)
    v_c = ws[N * 1152 + N * 32768:N * 1152 + 2 * N * 32768].view(torch.bfloat16).view(128, N, 128)
    out = torch.empty((T, 128, 128), dtype=torch.bfloat16, device=dev)
    g_us = _time_launches(torch, stream, lambda i: api.mla_gather_paged(kv, bt, 0, N, rows, err))
    e_us = _time_launches(torch, stream, lambda i: api.mla_expand_kv(rows, w_uk, w_uv, k_c, v_c, err))
    a_us = _time_launches(torch, stream, lambda i: api.mla_prefill_attention(q_c[:M], q_r[:M], rows, k_c, v_c, out[:M],
                                                                               err))

    # the whole branch for the batch: one gather, one expansion and one
    # attention launch over every sequence's packed cache
    n_all = [int(x) for x in case.seq_lens]
    ws_all = torch.empty(api.mla_prefill_batch_workspace_size(n_all), dtype=torch.uint8, device=dev)
    seqs = list(range(case.B))
    starts = [int(x) for x in case.q_start[:case.B]]
    qls = [int(x) for x in case.q_lens]

    def branch(i):
        api.mla_prefill_decompress_batch(q_c, q_r, kv, bt, seqs, starts, qls, n_all, w_uk, w_uv, ws_all, out, err)

    d_us = _time_launches(torch, stream, branch, reps=3, warmup=2, per_rep=3)
    q_abs = torch.empty((T, 128, 512), dtype=torch.bfloat16, device=dev)
    o_lat = torch.empty((T, 128, 512), dtype=torch.bfloat16, device=dev)
    out2 = torch.empty_like(out)
    plan = api.mla_decode_plan(case.seq_lens, case.q_lens, device=dev)

    def absorbed(i):
        api.mla_absorb_q(q_c, w_uk, q_abs, err)
        api.mla_decode_paged(q_abs, q_r, kv, bt, plan, o_lat, err, scale=SCALE)
        api.mla_up_v(o_lat, w_uv, out2, err)

    b_us = _time_launches(torch, stream, absorbed, reps=3, warmup=2, per_rep=4)
    if api.mla_check(err) != 0:
        raise RuntimeError("device error word set while timing the decompress branch")
    exp_fl = N * 128 * 2 * 512 * 256
    vis = M * (N - M) + M * (M + 1) // 2
    att_fl = vis * 128 * 2 * 320
    pk = peaks["bf16_tflops"]
    return {
        "workload": case.name, "threshold": api.mla_prefill_threshold(),
        "gather_us": round(g_us, 2),
        "expand_us": round(e_us, 1), "expand_tflops": round(exp_fl / e_us / 1e6, 1),
        "expand_frac": round(exp_fl / e_us / 1e6 / pk, 4),
        "attention_us": round(a_us, 1), "attention_tflops": round(att_fl / a_us / 1e6, 1),
        "attention_frac": round(att_fl / a_us / 1e6 / pk, 4),
        "branch_us_batch": round(d_us, 1), "absorbed_a2_a5_us_batch": round(b_us, 1),
        "branch_tflops": round(case.B * (exp_fl + att_fl) / d_us / 1e6, 1),
        "peak_tflops": pk, "peak_source": peaks["source"] + " (burst)",
    }


def parity_rows(api, plan, T, k=8):
    """Rows checked against the oracle: the first and last row, then rows the
    combine merges from split pieces, then rows at cluster-range boundaries."""
    r = api.plan_rows(plan)
    pick = [0, T - 1]
    for x in r["split"][::max(1, len(r["split"]) // max(1, k // 2))] + r["boundary"]:
        if len(pick) >= k:
            break
        if x not in pick:
            pick.append(int(x))
    return sorted(set(pick)), r["split"]


def measure_configs(api, torch, dev, stream, peaks, main_w, main_st, main_dec_us, main_step_us, num_clusters,
                    reps=6):
    """Every workload of the scope table, each in the bench's launch
    configuration (all clusters, inputs resident): the decode (decode +
    combine launches) and the whole step A1 -> A5, each launch timed alone
    with CUDA events after a write of 256 MB that flushes L2 (workloads 0, 1
    and 4 would otherwise find their cache in L2); the roofline of the
    decode.  The main workload's entry repeats the timed run's figures.
    (Every workload's rows are checked against the oracle at full size by
    the GPU parity tests; the main workload's timed step also by the CPU
    baseline leg here.)"""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    table = {}
    for w in sorted(wl.WORKLOADS):
        case = wl.workload(w, seed=0)
        st = workload_stats(case)
        t_f = st["flops"] / (peaks["bf16_tflops"] * 1e12)
        t_b = st["bytes"] / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if t_f >= t_b else "hbm"
        t_roof_us = max(t_f, t_b) * 1e6
        if w == main_w:
            dec_us, step_us = main_dec_us, main_step_us
        else:
            def bf(x):
                return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device=dev, dtype=torch.bfloat16)
            err = torch.zeros(1, dtype=torch.int32, device=dev)
            kv = torch.empty((case.num_pages, 64, 576), dtype=torch.bfloat16, device=dev)
            api.mla_cache_init(kv)
            seq, pos = case.positions()
            slots = api.mla_slot_mapping(case.block_table, seq, pos)
            new_idx = case.new_token_index()
            old = np.ones(slots.shape[0], dtype=bool)
            old[new_idx] = False
            if old.any():
                api.mla_kv_append(bf(case.c_kv[old]), bf(case.k_r[old]), torch.from_numpy(slots[old]).to(dev), kv,
                                  err)
            c_new, k_new = bf(case.c_kv[new_idx]), bf(case.k_r[new_idx])
            s_new = torch.from_numpy(slots[new_idx]).to(dev)
            bt = torch.from_numpy(case.block_table).to(dev)
            q_c, q_r, w_uk, w_uv = bf(case.q_c), bf(case.q_r), bf(case.w_uk), bf(case.w_uv)
            T = case.T
            q_abs = torch.empty((T, 128, 512), dtype=torch.bfloat16, device=dev)
            o_lat = torch.empty((T, 128, 512), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((T, 128), dtype=torch.float32, device=dev)
            out = torch.empty((T, 128, 128), dtype=torch.bfloat16, device=dev)
            plan = api.mla_decode_plan(case.seq_lens, case.q_lens, device=dev, num_clusters=num_clusters)

            def decode():
                api.mla_decode_paged(q_abs, q_r, kv, bt, plan, o_lat, err, lse=lse, scale=SCALE)

            def whole():
                api.mla_kv_append(c_new, k_new, s_new, kv, err)
                api.mla_absorb_q(q_c, w_uk, q_abs, err)
                decode()
                api.mla_up_v(o_lat, w_uv, out, err)

            def timed(fn):
                for _ in range(3):
                    fn()
                ts = []
                for _ in range(reps):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    torch.cuda.synchronize(dev)
                    ts.append(a.elapsed_time(b) * 1e3)
                return statistics.median(ts)

            step_us = timed(whole)
            dec_us = timed(decode)
            if api.mla_check(err) != 0:
                raise RuntimeError(f"device error word set while timing workload {w}")
            del kv, q_abs, o_lat, out
            torch.cuda.empty_cache()
        table[case.name] = dict(
            rows=case.T, bound=bound, t_roof_us=round(t_roof_us, 2), decode_us=round(dec_us, 2),
            frac=round(t_roof_us / dec_us, 4), kv_tb_per_s=round(st["kv_bytes"] / (dec_us * 1e-6) / 1e12, 4),
            tflops=round(st["flops"] / (dec_us * 1e-6) / 1e12, 1), step_us=round(step_us, 2),
            step_tokens_per_s=round(case.T / (step_us * 1e-6), 1),
            timing="main timed run" if w == main_w else "median of %d launches, L2 flushed before each" % reps)
    del flush
    return table


def run_mla(args):
    import torch
    from mla_latent_kv_02_gb300 import api

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    case = wl.workload(args.workload, seed=0, batch=args.batch)
    st = workload_stats(case)
    T = case.T

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device=dev, dtype=torch.bfloat16)

    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = torch.empty((case.num_pages, 64, 576), dtype=torch.bfloat16, device=dev)
    api.mla_cache_init(kv)
    bt = torch.from_numpy(case.block_table).to(dev)
    seq, pos = case.positions()
    slots_all = api.mla_slot_mapping(case.block_table, seq, pos)
    new_idx = case.new_token_index()
    old_mask = np.ones(slots_all.shape[0], dtype=bool)
    old_mask[new_idx] = False
    old_idx = np.nonzero(old_mask)[0]
    c_old, k_old = bf(case.c_kv[old_idx]), bf(case.k_r[old_idx])
    slots_old = torch.from_numpy(slots_all[old_idx]).to(dev)
    if old_idx.size:
        api.mla_kv_append(c_old, k_old, slots_old, kv, dev_err)
    c_new, k_new = bf(case.c_kv[new_idx]), bf(case.k_r[new_idx])
    slots_new = torch.from_numpy(slots_all[new_idx]).to(dev)
    q_c, q_r = bf(case.q_c), bf(case.q_r)
    w_uk, w_uv = bf(case.w_uk), bf(case.w_uv)
    q_abs = torch.empty((T, 128, 512), dtype=torch.bfloat16, device=dev)
    o_lat = torch.empty((T, 128, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, 128), dtype=torch.float32, device=dev)
    out = torch.empty((T, 128, 128), dtype=torch.bfloat16, device=dev)
    plan = api.mla_decode_plan(case.seq_lens, case.q_lens, device=dev)
    launches_per_step = 4 + (1 if plan.info.num_split_rows > 0 else 0)

    def step(ev=None):
        api.mla_kv_append(c_new, k_new, slots_new, kv, dev_err)
        api.mla_absorb_q(q_c, w_uk, q_abs, dev_err)
        if ev is not None:
            ev[0].record(stream)
        api.mla_decode_paged(q_abs, q_r, kv, bt, plan, o_lat, dev_err, lse=lse, scale=SCALE)
        if ev is not None:
            ev[1].record(stream)
        api.mla_up_v(o_lat, w_uv, out, dev_err)

    for _ in range(args.warmup):
        step()
    if api.mla_check(dev_err) != 0:
        raise RuntimeError("device error word set during warm-up")

    K = args.steps
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    import tempfile
    clocks = ClockSampler(local, os.path.join(tempfile.gettempdir(), f"mla_bench_clocks_{os.getpid()}_r{rank}.csv"))
    barrier(ws)
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(2_000_000)   # untimed: lets the first launches queue up behind it
    e0.record(stream)
    for i in range(K):
        step(dec_ev[i])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    ms_total = e0.elapsed_time(e1)
    ms_total = reduce_max(ms_total, ws, dev)
    dec_ms = [a.elapsed_time(b) for a, b in dec_ev]
    dec_avg = sum(dec_ms) / len(dec_ms)
    if api.mla_check(dev_err) != 0:
        raise RuntimeError("device error word set during the timed steps")
    # the step's other kernels, each timed alone after the timed region on
    # the same inputs (launched back to back, warm as inside the step)
    step_kernels = {
        "a1_kv_append_us": round(_time_launches(torch, stream, lambda i: api.mla_kv_append(c_new, k_new, slots_new, kv,
                                                                                           dev_err), reps=20), 2),
        "a2_absorb_q_us": round(_time_launches(torch, stream, lambda i: api.mla_absorb_q(q_c, w_uk, q_abs, dev_err),
                                               reps=20), 2),
        "a3_a4_decode_us": round(dec_avg * 1e3, 2),
        "a5_up_v_us": round(_time_launches(torch, stream, lambda i: api.mla_up_v(o_lat, w_uv, out, dev_err), reps=20), 2),
    }
    step_kernels["outside_decode_us"] = round(ms_total / K * 1e3 - dec_avg * 1e3, 2)
    if api.mla_check(dev_err) != 0:
        raise RuntimeError("device error word set while timing the step's kernels")

    # ---- end to end through the API: pinned host inputs in, result out, plan rebuilt each step.
    # E2E_SLOTS steps in flight, as a serving loop runs: the host plans and
    # enqueues the next steps before it waits for step i's result and reads it; the copies
    # in and the copies out run on two streams of their own (double-buffered
    # device inputs and outputs), so that step i+1's inputs never queue behind
    # step i's result and both overlap the neighbouring steps' kernels.
    h_q_c = torch.from_numpy(case.q_c).to(torch.bfloat16).pin_memory()
    h_q_r = torch.from_numpy(case.q_r).to(torch.bfloat16).pin_memory()
    h_c_new = c_new.cpu().pin_memory()
    h_k_new = k_new.cpu().pin_memory()
    h_slots = slots_new.cpu().pin_memory()
    h_out = [torch.empty((T, 128, 128), dtype=torch.bfloat16).pin_memory() for _ in range(E2E_SLOTS)]
    d_in = [(torch.empty_like(q_c), torch.empty_like(q_r), torch.empty_like(c_new), torch.empty_like(k_new),
             torch.empty_like(slots_new)) for _ in range(E2E_SLOTS)]
    d_out = [torch.empty((T, 128, 128), dtype=torch.bfloat16, device=dev) for _ in range(E2E_SLOTS)]
    h2d = sum(t.numel() * t.element_size() for t in (h_q_c, h_q_r, h_c_new, h_k_new, h_slots))
    d2h = h_out[0].numel() * h_out[0].element_size()
    in_stream = torch.cuda.Stream(device=dev)
    out_stream = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(E2E_SLOTS)]     # inputs of slot s landed
    ev_used = [torch.cuda.Event() for _ in range(E2E_SLOTS)]   # the kernels of slot s are done with its buffers
    ev_done = [torch.cuda.Event() for _ in range(E2E_SLOTS)]   # slot s's result is on the host
    for e in ev_used:
        e.record(stream)
    checksum = [0.0]
    e2e_plans = [api.mla_decode_plan(case.seq_lens, case.q_lens, device=dev, num_clusters=plan.num_clusters)
                 for _ in range(E2E_SLOTS)]

    def e2e_issue(i):
        sl = i % E2E_SLOTS
        dq_c, dq_r, dc_new, dk_new, dslots = d_in[sl]
        with torch.cuda.stream(in_stream):
            in_stream.wait_event(ev_used[sl])
            dq_c.copy_(h_q_c, non_blocking=True)
            dq_r.copy_(h_q_r, non_blocking=True)
            dc_new.copy_(h_c_new, non_blocking=True)
            dk_new.copy_(h_k_new, non_blocking=True)
            dslots.copy_(h_slots, non_blocking=True)
            # the plan is rebuilt every step into its slot's pinned buffer
            # (that slot's previous step has finished: its result was
            # collected) and uploaded with the inputs, off the compute stream
            p = api.mla_decode_plan(case.seq_lens, case.q_lens, device=dev, into=e2e_plans[sl], stream=in_stream)
            ev_in[sl].record(in_stream)
        stream.wait_event(ev_in[sl])
        api.mla_kv_append(dc_new, dk_new, dslots, kv, dev_err)
        api.mla_absorb_q(dq_c, w_uk, q_abs, dev_err)
        api.mla_decode_paged(q_abs, dq_r, kv, bt, p, o_lat, dev_err, lse=lse, scale=SCALE)
        api.mla_up_v(o_lat, w_uv, d_out[sl], dev_err)
        ev_used[sl].record(stream)
        with torch.cuda.stream(out_stream):
            out_stream.wait_event(ev_used[sl])
            h_out[sl].copy_(d_out[sl], non_blocking=True)
            ev_done[sl].record(out_stream)

    def e2e_collect(i):
        ev_done[i % E2E_SLOTS].synchronize()
        checksum[0] += float(h_out[i % E2E_SLOTS][0, 0, 0])   # the host reads this step's result

    def e2e_run(n):
        for i in range(n):
            e2e_issue(i)
            if i >= E2E_SLOTS - 1:
                e2e_collect(i - (E2E_SLOTS - 1))
        for i in range(max(0, n - (E2E_SLOTS - 1)), n):
            e2e_collect(i)

    e2e_run(max(E2E_SLOTS, args.warmup))
    barrier(ws)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    e2e_run(K)
    e2e_s = reduce_max(time.perf_counter() - t0, ws, dev)
    if api.mla_check(dev_err) != 0:
        raise RuntimeError("device error word set during the end-to-end steps")

    peaks = load_peaks()
    # the timed step's outputs on the rows the CPU baseline will check (split and boundary rows first)
    check_rows, check_split = parity_rows(api, plan, T)
    gpu_rows = dict(rows=check_rows, split=check_split, o_lat=o_lat.float().cpu().numpy()[check_rows],
                    out=out.float().cpu().numpy()[check_rows], lse=lse.cpu().numpy()[check_rows])
    rows = measure_rows(api, torch, dev, stream, case, c_old, k_old, slots_old, pos[old_idx], q_r, kv, dev_err,
                        peaks["hbm_gbs"], plan=plan, q_abs=q_abs, st=st, peaks=peaks) if old_idx.size else {}
    step_s = ms_total / 1e3 / K
    tokens = T * ws
    value = tokens / step_s
    dec_s = dec_avg / 1e3
    t_flops = st["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_bytes = st["bytes"] / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_flops >= t_bytes else "hbm"
    if bound == "tensor":
        achieved, peak, unit = st["flops"] / dec_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = st["bytes"] / dec_s / 1e9, peaks["hbm_gbs"], "GB/s"

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/512) weights, random page tables)",
        "config": {
            "workload": case.name,
            "batch": case.B, "query_tokens_per_seq": int(case.q_lens.max()),
            "context_tokens": int(case.seq_lens.max()), "rows": T, "heads": 128, "d_c": 512, "d_r": 64,
            "page_size": 64, "kv_bytes_per_step": st["kv_bytes"],
            "l2": "inputs larger than L2 (%.0f MB of KV streamed per step)" % (st["kv_bytes"] / 1e6),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "decode_clusters": plan.num_clusters, "split_rows": int(plan.info.num_split_rows),
        },
        "kv_tb_per_s": round(st["kv_bytes"] / dec_s / 1e12, 4),
        "decode_us": round(dec_avg * 1e3, 2),
        "step_kernels": step_kernels,
        "roofline": {
            "kernel": "mla_decode_paged (decode + combine launches)",
            "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": decode_traffic(args.workload, args.batch),
            "peak_source": peaks["source"] + " (burst)",
            "t_roof_us": round(max(t_flops, t_bytes) * 1e6, 2),
            "frac_of_t_roof": round(max(t_flops, t_bytes) / dec_s, 4),
            "algorithmic": {"flops": st["flops"], "bytes": st["bytes"]},
        },
        "e2e": {"value": round(tokens * K / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps_in_flight": E2E_SLOTS},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "parity": None,
        "rows": rows,
    }
    if not args.no_configs:
        # free this workload's device buffers before the others are built
        del kv, c_old, k_old, q_abs, o_lat, out, d_in, d_out
        torch.cuda.empty_cache()
        line["configs"] = measure_configs(api, torch, dev, stream, peaks, args.workload, st, dec_avg * 1e3,
                                          ms_total / K * 1e3, plan.num_clusters)
    if not args.no_decompress:
        line["decompress_branch"] = measure_decompress(api, torch, dev, stream, peaks)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_budget, check=gpu_rows)
        line["cpu_baseline"].pop("seconds", None)
        line["parity"] = line["cpu_baseline"].pop("parity", None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm: the CPU oracle
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    case = wl.workload(args.workload, seed=0)
    import oracle
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    cache = oracle.append(np.zeros((case.num_pages, 64, 576), dtype=np.float32), case.c_kv, case.k_r, slots)
    rows_per_step = max(1, min(case.T, args.ref_rows))

    def step(i):
        rows = [(i * rows_per_step + k) % case.T for k in range(rows_per_step)]
        oracle.mla_step(case.q_c, case.q_r, case.w_uk, case.w_uv, cache, case.block_table,
                        case.seq_lens, case.q_lens, SCALE, rows=rows)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": case.name, "batch": case.B, "rows": case.T},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} query rows per step of {case.T}"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=2, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None, help="keep only the first N sequences (profiling cases)")
    ap.add_argument("--impl", default="mla", choices=["mla", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decompress", action="store_true", help="skip the decompress-branch measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table")
    ap.add_argument("--ref-rows", type=int, default=2, help="query rows per reference-arm step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "mla":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_mla(args)


if __name__ == "__main__":
    main()
