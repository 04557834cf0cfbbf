"""The seeded synthetic inputs follow their stated recipe (shapes, value
ranges, distributions, page-table structure), so that the figures quoted on
them (the bench's prefix sums, the rows' workloads) describe what ran.
Small head counts keep the tensors cheap where only the structure matters."""
import math

import numpy as np
import pytest
import torch

import workloads


def test_serving_prefixes():
    """64 prefixes, 64 * round(exp(U[ln 128, ln 32768]) / 64) in [128, 32768];
    seed 0 sums to 399,936 tokens (the bench's decode workload) and, at
    token granularity, to 399,993 (the extend workload)."""
    P = workloads.prefix_loguniform_blocks(64, 128, 32768, 64, seed=0)
    assert len(P) == 64 and all(p % 64 == 0 and 128 <= p <= 32768 for p in P)
    assert sum(P) == 399936
    assert sum(workloads.prefix_loguniform_blocks(64, 128, 32768, 1, seed=0)) == 399993
    assert workloads.prefix_loguniform_blocks(64, 128, 32768, 64, seed=1) != P


def test_log_uniform_distribution():
    """ln of the draws is uniform on [ln 128, ln 32768] (step 1, many draws)."""
    scipy_stats = pytest.importorskip("scipy.stats")
    x = np.log(np.array(workloads.prefix_loguniform_blocks(20000, 128, 32768, 1, seed=3), float))
    lo, hi = math.log(128), math.log(32768)
    assert scipy_stats.kstest(x, "uniform", args=(lo, hi - lo)).pvalue > 1e-3


def test_block_decode_prefixes():
    """8 prefixes uniform over {512, 576, ..., 4096}; seed 0 sums to 16,384."""
    P = workloads.prefix_uniform_blocks(8, 512, 4096, 64, seed=0)
    assert all(p % 64 == 0 and 512 <= p <= 4096 for p in P)
    assert sum(P) == 16384
    many = workloads.prefix_uniform_blocks(5700, 512, 4096, 64, seed=4)
    assert set(many) == set(range(512, 4097, 64))


@pytest.mark.parametrize("S", [16, 64])
def test_pool_pages(S):
    """ceil(cap / S) distinct physical pages per sequence, none shared, ids in
    [0, num_pages), the pool twice the need, unused entries -1, slots NaN."""
    cap = [0, 1, 100, 3000, 64]
    pool = workloads.build_paged_pool(cap, Hkv=2, d=16, page_size=S, seed=5)
    need = [-(-c // S) for c in cap]
    assert pool.num_pages == max(sum(need), math.ceil(2.0 * sum(need)))
    pt = pool.page_table.numpy()
    used = np.concatenate([pt[b, :n] for b, n in enumerate(need)])
    assert len(set(used.tolist())) == used.size == sum(need)
    assert used.min() >= 0 and used.max() < pool.num_pages
    for b, n in enumerate(need):
        assert (pt[b, n:] == -1).all()
    assert torch.isnan(pool.k_pool.float()).all() and torch.isnan(pool.v_pool.float()).all()


def test_multicanvas_structure():
    """The multicanvas row's structure (16 sequences, prompt 1024, 3 canvases
    of 256): every position below the last canvas's end stored exactly once,
    in the arena or as a live row; the arena is the prompt in order, then
    promoted rows; each canvas keeps 30-100 % of its rows live; about 25 % of
    each canvas's live rows are promoted, at least one."""
    c = workloads.make_multicanvas_case(16, 1024, 3, 256, Hq=2, Hkv=1, d=16, seed=0)
    total = 1024 + 3 * 256
    for b in range(c.B):
        n = int(c.live_count[b])
        live = c.live_pos[b, :n].tolist()
        arena = c.arena_pos[b].tolist()
        assert sorted(live + arena) == list(range(total))
        assert arena[:1024] == list(range(1024))
        assert int(c.arena_len[b]) == len(arena)
        rows = c.commit_rows[b, :int(c.commit_count[b])].tolist()
        assert len(set(rows)) == len(rows) and all(0 <= r < n for r in rows)
        for k in range(3):
            lo, hi = 1024 + 256 * k, 1024 + 256 * (k + 1)
            n_live = sum(lo <= p < hi for p in live)
            assert 0.3 * 256 - 1 <= n_live <= 256
            n_com = sum(lo <= live[r] < hi for r in rows)
            assert n_com == max(1, round(0.25 * n_live))


def test_confidence_logits():
    """N(0, 3^2) logits with one token of every fourth row lifted by 6 to 14."""
    x = workloads.confidence_logits(64, 4096, seed=2, dtype=torch.float32)
    assert x.shape == (64, 4096)
    body = x[1::4].flatten()
    assert abs(float(body.std()) - 3.0) < 0.1 and abs(float(body.mean())) < 0.1
    top = x[0::4].max(dim=1).values
    assert (top > 6.0).all()
