"""GPU parity of bca_qkv_post (norms + RoPE + cache write) against the fp64
oracle.  Query and key outputs are within one bf16 ulp of the oracle's fp64
value (the kernel rounds its fp32 result once: |err| <= 2^-8 |x| + 2^-16);
values and every cache write are bit-exact."""
import numpy as np
import pytest
import torch

import block_causal_paged_gb300 as bca
import oracle
import workloads

pytestmark = pytest.mark.gpu


class Run:
    def __init__(self, c, dev="cuda"):
        self.c = c
        self.qkv = c.qkv.to(dev)
        self.positions = c.positions.to(dev)
        self.qw, self.kw = c.q_norm_w.to(dev), c.k_norm_w.to(dev)
        self.write_pos = c.write_pos.to(dev)
        self.k_pool, self.v_pool = c.pool.k_pool.to(dev), c.pool.v_pool.to(dev)
        self.page_table = c.pool.page_table.to(dev)
        self.kv_pos = torch.full((c.pool.num_pages, c.pool.page_size), -7, dtype=torch.int32,
                                 device=dev)
        self.q = torch.empty((c.B, c.n, c.Hq, c.d), dtype=torch.bfloat16, device=dev)
        self.k = torch.empty((c.B, c.n, c.Hkv, c.d), dtype=torch.bfloat16, device=dev)
        self.v = torch.empty_like(self.k)
        self.d = bca.dims(c.B, c.n, c.Hq, c.Hkv, c.d, c.pool.page_size, c.pool.num_pages,
                          c.pool.max_pages_per_seq)
        self.ws = bca.new_workspace(self.d, bca.OP_COMMIT, device=dev)

    def run(self, norms=True, theta=1e6, eps=1e-6, write=True, arena=False):
        bca.bca_qkv_post(self.d, self.qkv, self.positions, self.q, self.k, self.v, self.ws,
                         q_norm_w=self.qw if norms else None, k_norm_w=self.kw if norms else None,
                         eps=eps, rope_theta=theta, write_pos=self.write_pos if write else None,
                         k_pool=self.k_pool, v_pool=self.v_pool, page_table=self.page_table,
                         kv_pos=self.kv_pos if arena else None)
        torch.cuda.synchronize()

    def status(self):
        return bca.read_device_status(self.ws)


def _check(r, norms=True, theta=1e6, eps=1e-6):
    c = r.c
    q, k, v = oracle.qkv_post(c.qkv, c.positions, c.Hq, c.Hkv,
                              q_norm_w=c.q_norm_w if norms else None,
                              k_norm_w=c.k_norm_w if norms else None, eps=eps, rope_theta=theta)
    for name, got, ref in (("q", r.q, q), ("k", r.k, k)):
        g = got.float().cpu().numpy().astype(np.float64)
        err = np.abs(g - ref)
        bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -16
        assert (err <= bound).all(), f"{name}: worst excess {(err - bound).max():.3g}"
    want_v = c.qkv[:, :, c.Hq + c.Hkv:].contiguous()
    assert torch.equal(r.v.cpu().view(torch.int16), want_v.view(torch.int16))


def _check_cache(r, arena=False):
    c = r.c
    S = c.pool.page_size
    kp, vp = c.pool.k_pool.clone(), c.pool.v_pool.clone()
    kv_pos = torch.full((c.pool.num_pages, S), -7, dtype=torch.int32)
    kc, vc = r.k.cpu(), r.v.cpu()
    for b in range(c.B):
        for t in range(c.n):
            p = int(c.write_pos[b, t])
            if p < 0:
                continue
            page = int(c.pool.page_table[b, p // S])
            kp[page, :, p % S] = kc[b, t]
            vp[page, :, p % S] = vc[b, t]
            kv_pos[page, p % S] = int(c.positions[b, t])
    assert torch.equal(r.k_pool.cpu().view(torch.int16), kp.view(torch.int16))
    assert torch.equal(r.v_pool.cpu().view(torch.int16), vp.view(torch.int16))
    if arena:
        assert torch.equal(r.kv_pos.cpu(), kv_pos)


@pytest.mark.parametrize("d", [128, 64])
def test_block_after_prefix_with_commit(cuda_lib, d):
    c = workloads.make_qkv_post_case(5, 64, 8, 2, d, prefix_len=[0, 64, 320, 1024, 4032], seed=d)
    r = Run(c)
    r.run()
    assert r.status() == 0
    _check(r)
    _check_cache(r)


def test_arena_mode_random_positions(cuda_lib):
    """Live rows at scattered absolute positions up to 2^20 (the angle
    reduction), written to arena slots with their positions."""
    c = workloads.make_qkv_post_case(3, 40, 6, 2, 128, seed=3, pos_max=1 << 20)
    r = Run(c)
    r.run(arena=True)
    assert r.status() == 0
    _check(r)
    _check_cache(r, arena=True)


@pytest.mark.parametrize("norms,theta", [(False, 1e6), (True, 0.0), (False, 0.0), (True, 10000.0)])
def test_norm_and_rope_switches(cuda_lib, norms, theta):
    c = workloads.make_qkv_post_case(2, 9, 32, 8, 128, prefix_len=[7, 1000], seed=4)
    r = Run(c)
    r.run(norms=norms, theta=theta, write=False)
    _check(r, norms=norms, theta=theta)
    assert torch.equal(r.k_pool.cpu().view(torch.int16), c.pool.k_pool.view(torch.int16))


def test_skipped_and_bad_cache_writes(cuda_lib):
    c = workloads.make_qkv_post_case(3, 16, 8, 2, 64, prefix_len=[0, 16, 48], seed=5)
    c.write_pos[0, :8] = -1                       # not written
    r = Run(c)
    r.run()
    assert r.status() == 0
    _check_cache(r)
    r.write_pos[1, 3] = c.pool.max_pages_per_seq * c.pool.page_size  # past the page table
    r.run()
    assert r.status() == bca.ERR_DEVICE_BAD_LENGTH
    r.write_pos[1, 3] = 16
    r.page_table[2, 3] = c.pool.num_pages + 1     # a page outside the pool
    r.run()
    assert r.status() == bca.ERR_DEVICE_PAGE_OOB


def test_serving_block_b64(cuda_lib):
    """Batch 64 blocks of 64 tokens, 32/8 heads, d = 128, after the serving
    prefixes, committed: the bench workload, every output compared."""
    P = workloads.prefix_loguniform_blocks(64, 128, 32768, 64, seed=0)
    c = workloads.make_qkv_post_case(64, 64, 32, 8, 128, prefix_len=P, seed=0)
    r = Run(c)
    r.run()
    assert r.status() == 0
    _check(r)


@pytest.mark.parametrize("scale,eps", [(1e-3, 1e-6), (3e-4, 1e-5)])
def test_small_rows_where_epsilon_matters(cuda_lib, scale, eps):
    """Rows small enough that the norm's epsilon is as large as (or larger
    than) the mean of the squares: the kernel follows the oracle's
    x * w / sqrt(mean(x^2) + eps), and the same comparison with eps dropped
    from the oracle fails, so the term is really exercised."""
    c = workloads.make_qkv_post_case(4, 16, 8, 2, 128, prefix_len=[0, 64, 320, 4032], seed=9,
                                     qkv_scale=scale)
    r = Run(c)
    r.run(eps=eps)
    assert r.status() == 0
    _check(r, eps=eps)
    q0, _, _ = oracle.qkv_post(c.qkv, c.positions, c.Hq, c.Hkv, q_norm_w=c.q_norm_w,
                               k_norm_w=c.k_norm_w, eps=0.0, rope_theta=1e6)
    g = r.q.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -8 * np.abs(q0) + 2.0 ** -16
    assert (np.abs(g - q0) > bound).mean() > 0.5


def test_long_token_ranges_per_sm(cuda_lib):
    """65536 tokens (8 x 8192) of 2/1 heads, d = 64: every SM's share runs to
    hundreds of tokens, so each consumer warp reloads its window of token
    metadata several times; rows of 4 heads leave a partial work unit per
    token.  Outputs against the oracle, the cache writes and kv_pos
    (arena mode) bit-exact."""
    c = workloads.make_qkv_post_case(8, 8192, 2, 1, 64, prefix_len=[0, 64, 128, 0, 512, 64, 0, 1024],
                                     seed=11)
    r = Run(c)
    r.run(arena=True)
    assert r.status() == 0
    _check(r)
    S = c.pool.page_size
    wp = c.write_pos.long()
    pages = torch.gather(c.pool.page_table.long(), 1, wp // S)
    kp, vp = c.pool.k_pool.clone(), c.pool.v_pool.clone()
    kv_pos = torch.full((c.pool.num_pages, S), -7, dtype=torch.int32)
    kp[pages.flatten(), :, (wp % S).flatten()] = r.k.cpu().reshape(-1, c.Hkv, c.d)
    vp[pages.flatten(), :, (wp % S).flatten()] = r.v.cpu().reshape(-1, c.Hkv, c.d)
    kv_pos[pages.flatten(), (wp % S).flatten()] = c.positions.flatten().int()
    assert torch.equal(r.k_pool.cpu().view(torch.int16), kp.view(torch.int16))
    assert torch.equal(r.v_pool.cpu().view(torch.int16), vp.view(torch.int16))
    assert torch.equal(r.kv_pos.cpu(), kv_pos)
