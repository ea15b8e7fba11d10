"""Shared test helpers: upload a seeded case, build both caches, compare."""
from __future__ import annotations

import numpy as np

import oracle
from mla_latent_kv_02_gb300 import workloads as wl

# Floating-point bar for bf16 storage with fp32 accumulation.
MAX_ERR_FRAC = 2e-2      # max|gpu - ref| <= 2e-2 * max|ref|
MEAN_REL = 5e-3          # sum|gpu - ref| / sum|ref| <= 5e-3


def err_stats(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(gpu - ref)
    return float(d.max() / max(np.abs(ref).max(), 1e-300)), float(d.sum() / max(np.abs(ref).sum(), 1e-300))


def assert_close(gpu, ref, name, max_frac=MAX_ERR_FRAC, mean_rel=MEAN_REL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite GPU values"
    mx, mr = err_stats(gpu, ref)
    assert mx <= max_frac and mr <= mean_rel, f"{name}: max_err/max_ref={mx:.3e} mean_rel={mr:.3e}"
    return mx, mr


def oracle_cache(case: wl.Case) -> np.ndarray:
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    empty = np.zeros((case.num_pages, wl.PAGE, wl.D_QK), dtype=np.float32)
    return oracle.append(empty, case.c_kv, case.k_r, slots)


def oracle_cache_fp8(case: wl.Case):
    """The oracle's FP8 cache of a case: (rows uint8, scales float64)."""
    seq, pos = case.positions()
    slots = oracle.slot_mapping(case.block_table, seq, pos)
    return oracle.fp8_cache.append(*oracle.fp8_cache.empty_cache(case.num_pages), case.c_kv, case.k_r, slots)


def to_bf16(x, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device=device, dtype=torch.bfloat16)


def to_np(t):
    import torch
    return t.detach().to(dtype=torch.float32).cpu().numpy()


class DeviceCase:
    """A case on the GPU; the paged cache is filled through mla_kv_append.

    The cached context is appended in one bulk call and this step's query
    tokens in a second call (step A1 of the path).
    """

    def __init__(self, case: wl.Case, device="cuda:0", with_weights=True, fp8=False):
        import torch
        from mla_latent_kv_02_gb300 import api
        self.case = case
        self.device = torch.device(device)
        dev = self.device
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.fp8 = fp8
        if fp8:
            self.rows = torch.zeros((case.num_pages, wl.PAGE, 640), dtype=torch.uint8, device=dev)
            self.scales = torch.ones((case.num_pages, wl.PAGE), dtype=torch.float32, device=dev)
        else:
            self.kv_cache = torch.empty((case.num_pages, wl.PAGE, wl.D_QK), dtype=torch.bfloat16, device=dev)
            api.mla_cache_init(self.kv_cache)
        self.block_table = torch.from_numpy(case.block_table).to(dev)
        seq, pos = case.positions()
        slots = api.mla_slot_mapping(case.block_table, seq, pos)
        new = np.zeros(slots.shape[0], dtype=bool)
        new[case.new_token_index()] = True
        self.slots_all = slots
        old_idx = np.nonzero(~new)[0]
        new_idx = case.new_token_index()
        for idx in (old_idx, new_idx):
            if idx.size == 0:
                continue
            if fp8:
                api.mla_kv_append_fp8(to_bf16(case.c_kv[idx], dev), to_bf16(case.k_r[idx], dev),
                                      torch.from_numpy(slots[idx]).to(dev), self.rows, self.scales, self.dev_err)
            else:
                api.mla_kv_append(to_bf16(case.c_kv[idx], dev), to_bf16(case.k_r[idx], dev),
                                  torch.from_numpy(slots[idx]).to(dev), self.kv_cache, self.dev_err)
        self.q_c = to_bf16(case.q_c, dev)
        self.q_r = to_bf16(case.q_r, dev)
        self.q_abs = to_bf16(case.q_abs, dev) if case.q_abs is not None else None
        if with_weights and case.w_uk is not None:
            self.w_uk = to_bf16(case.w_uk, dev)
            self.w_uv = to_bf16(case.w_uv, dev)
        torch.cuda.synchronize(dev)

    def decode(self, q_abs=None, num_clusters=None):
        import torch
        from mla_latent_kv_02_gb300 import api
        case = self.case
        q_abs = self.q_abs if q_abs is None else q_abs
        plan = api.mla_decode_plan(case.seq_lens, case.q_lens, device=self.device, num_clusters=num_clusters)
        T = case.T
        o = torch.full((T, wl.H, wl.D_C), float("nan"), dtype=torch.bfloat16, device=self.device)
        lse = torch.full((T, wl.H), float("nan"), dtype=torch.float32, device=self.device)
        if self.fp8:
            api.mla_decode_paged_fp8(q_abs, self.q_r, self.rows, self.scales, self.block_table, plan, o,
                                     self.dev_err, lse=lse)
        else:
            api.mla_decode_paged(q_abs, self.q_r, self.kv_cache, self.block_table, plan, o, self.dev_err, lse=lse)
        word = api.mla_check(self.dev_err)
        assert word == 0
        return o, lse, plan
