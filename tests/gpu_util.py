"""Helpers shared by the GPU tests: move seeded workloads to the device and
compare library results with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances for bf16 inputs with fp32 accumulation (outputs vs the fp64 oracle).
TOL_O = 1e-2
TOL_LSE = 1e-3


def dev_bf16(a, device="cuda:0"):
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)


def dev_i32(a, device="cuda:0"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class VerifyDev:
    def __init__(self, wl, device="cuda:0"):
        self.wl = wl
        self.q = dev_bf16(wl.q, device)
        self.k = dev_bf16(wl.k_pages, device)
        self.v = dev_bf16(wl.v_pages, device)
        self.ppt = dev_i32(wl.prefix_page_table, device)
        self.dpt = dev_i32(wl.draft_page_table, device)
        self.lens = dev_i32(wl.prefix_lens, device)

    def args(self):
        return (self.q, self.k, self.v, self.ppt, self.dpt, self.lens, self.wl.topk, self.wl.S)


class PrefillDev:
    def __init__(self, wl, device="cuda:0"):
        self.wl = wl
        self.q = dev_bf16(wl.q, device)
        self.k = dev_bf16(wl.k_pages, device)
        self.v = dev_bf16(wl.v_pages, device)
        self.pt = dev_i32(wl.page_table, device)


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref_o, ref_lse, rows=None, tol_o=TOL_O,
            tol_lse=TOL_LSE):
    """Element-wise check; returns (max|do|, max|dlse|).  -inf lse must match exactly."""
    d = ref_o.shape[-1]
    go = o_gpu.float().reshape(-1, d)
    gl = lse_gpu.float().reshape(-1)
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), device=go.device)
        go = go[idx]
        gl = gl[idx]
    go = go.cpu().numpy().astype(np.float64)
    gl = gl.cpu().numpy().astype(np.float64)
    assert go.shape == ref_o.shape, (go.shape, ref_o.shape)
    assert np.all(np.isfinite(go)), "non-finite output"
    err_o = float(np.abs(go - ref_o).max()) if go.size else 0.0
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gl), fin), "lse finiteness differs from the oracle"
    assert np.all(gl[~fin] == -np.inf)
    err_l = float(np.abs(gl[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
    assert err_o <= tol_o, f"max|do| = {err_o:.3e} > {tol_o}"
    assert err_l <= tol_lse, f"max|dlse| = {err_l:.3e} > {tol_lse}"
    return err_o, err_l


def sample_rows(n_rows: int, k: int, seed: int, always=()):
    rng = np.random.default_rng(seed)
    pick = set(int(x) for x in rng.choice(n_rows, size=min(k, n_rows), replace=False))
    pick.update(int(a) % n_rows for a in always)
    return np.array(sorted(pick), dtype=np.int64)


class TreeDev:
    def __init__(self, wl, device="cuda:0"):
        self.wl = wl
        self.q = dev_bf16(wl.q, device)
        self.k = dev_bf16(wl.k_pages, device)
        self.v = dev_bf16(wl.v_pages, device)
        self.ppt = dev_i32(wl.prefix_page_table, device)
        self.tpt = dev_i32(wl.tree_page_table, device)
        self.lens = dev_i32(wl.prefix_lens, device)
        self.parents = dev_i32(wl.parents, device)

    def args(self):
        return (self.q, self.k, self.v, self.ppt, self.tpt, self.lens, self.parents)
