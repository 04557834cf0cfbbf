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

    def run(self, commit=False, ws=None, extend=False):
        ws = self.ws if ws is None else ws
        fn = bca.bca_extend if extend else bca.bca_decode
        fn(self.d, self.q, self.k_blk, self.v_blk, self.k_pool, self.v_pool, self.page_table,
           self.prefix_len, self.out, commit, ws)
        torch.cuda.synchronize()
        return self.out

    def status(self):
        return bca.read_device_status(self.ws)


class PrefillRun:
    def __init__(self, case, dev="cuda", write_pages=True):
        self.case = case
        self.q, self.k, self.v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
        self.cu = case.cu_seqlens.to(dev)
        self.k_pool = case.pool.k_pool.to(dev) if write_pages else None
        self.v_pool = case.pool.v_pool.to(dev) if write_pages else None
        self.page_table = case.pool.page_table.to(dev)
        self.out = torch.empty_like(self.q)
        self.d = bca.dims(len(case.seq_lens), case.D, case.Hq, case.Hkv, case.d,
                          case.pool.page_size, case.pool.num_pages, case.pool.max_pages_per_seq)
        self.ws = bca.new_workspace(self.d, bca.OP_PREFILL, device=dev)

    def run(self):
        c = self.case
        bca.bca_prefill(self.d, self.q, self.k, self.v, self.cu, sum(c.seq_lens), max(c.seq_lens),
                        self.k_pool, self.v_pool, self.page_table, self.out, self.ws)
        torch.cuda.synchronize()
        return self.out

    def status(self):
        return bca.read_device_status(self.ws)


class MulticanvasRun:
    def __init__(self, case, dev="cuda", pass_positions=True, promote=True):
        self.case = case
        self.q = case.q_live.to(dev)
        self.k = case.k_live.to(dev)
        self.v = case.v_live.to(dev)
        self.live_pos = case.live_pos.to(dev) if pass_positions else None
        self.live_count = case.live_count.to(dev) if pass_positions else None
        self.k_pool = case.pool.k_pool.to(dev)
        self.v_pool = case.pool.v_pool.to(dev)
        self.page_table = case.pool.page_table.to(dev)
        self.kv_pos = case.kv_pos.to(dev)
        self.arena_len = case.arena_len.to(dev)
        self.commit_rows = case.commit_rows.to(dev) if promote else None
        self.commit_count = case.commit_count.to(dev) if promote else None
        self.out = torch.zeros_like(self.q)
        self.d = bca.dims(case.B, case.canvas_len, case.Hq, case.Hkv, case.d,
                          case.pool.page_size, case.pool.num_pages, case.pool.max_pages_per_seq)
        self.ws = bca.new_workspace(self.d, bca.OP_MULTICANVAS, device=dev)

    def run(self, window=0):
        c = self.case
        bca.bca_multicanvas(self.d, self.q, self.k, self.v, self.live_pos, self.live_count,
                            c.q_live.shape[1], c.prompt_len, c.n_canvas, self.k_pool, self.v_pool,
                            self.page_table, self.kv_pos, self.arena_len, self.commit_rows,
                            self.commit_count, c.commit_rows.shape[1], self.out, self.ws,
                            window=window)
        torch.cuda.synchronize()
        return self.out

    def status(self):
        return bca.read_device_status(self.ws)
