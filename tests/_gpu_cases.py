"""Helpers for the GPU tests: move a seeded workload to cuda:0, run one entry
point of the library through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import block_causal_paged_gb300 as bca

# Acceptance bar for outputs against the fp64 oracle on the same bf16 inputs.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def assert_close(got_bf16: torch.Tensor, ref: np.ndarray, mask=None, what=""):
    got = got_bf16.detach().cpu().double().numpy()
    if mask is not None:
        got, ref = got[mask], ref[mask]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def dims_for_decode(case, scale=0.0):
    return bca.dims(case.B, case.D, case.Hq, case.Hkv, case.d, case.pool.page_size,
                    case.pool.num_pages, case.pool.max_pages_per_seq, scale)


class DecodeRun:
    def __init__(self, case, dev="cuda"):
        self.case = case
        self.q = case.q.to(dev)
        self.k_blk = case.k_blk.to(dev)
        self.v_blk = case.v_blk.to(dev)
        self.k_pool = case.pool.k_pool.to(dev)
        self.v_pool = case.pool.v_pool.to(dev)
        self.page_table = case.pool.page_table.to(dev)
        self.prefix_len = torch.tensor(case.prefix_len, dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.d = dims_for_decode(case)
        self.ws = bca.new_workspace(self.d, bca.OP_DECODE, device=dev)

    def run(self, commit=False, ws=None):
        ws = self.ws if ws is None else ws
        bca.bca_decode(self.d, self.q, self.k_blk, self.v_blk, self.k_pool, self.v_pool,
                       self.page_table, self.prefix_len, self.out, commit, ws)
        torch.cuda.synchronize()
        return self.out

    def status(self):
        return bca.read_device_status(self.ws)
