"""GPU parity with pages of 32, 64 and 256 tokens.

The cache takes any page size that is a multiple of 16 up to 256 ("Paged
Attention": position p lives in page page_table[b][p / S], slot p % S); the
kernels still move 16-row boxes, several per page.  Every entry point that
reads or writes pages, against the oracle; every written page bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_cases import DecodeRun, MulticanvasRun, PrefillRun, assert_close

pytestmark = pytest.mark.gpu

SIZES = [32, 64, 256]


def _check_commit(case, r, n):
    S = case.pool.page_size
    for name, pool, blk in (("k", r.k_pool, case.k_blk), ("v", r.v_pool, case.v_blk)):
        src = (case.pool.k_pool if name == "k" else case.pool.v_pool).view(torch.int16).numpy()
        want = oracle.commit(src, case.pool.page_table, case.prefix_len,
                             blk.view(torch.int16).numpy(), n, S)
        assert np.array_equal(pool.cpu().view(torch.int16).numpy(), want), f"{name} pool, S={S}"


@pytest.mark.parametrize("S", SIZES)
@pytest.mark.parametrize("D", [64, 32])
def test_decode_with_commit(cuda_lib, S, D):
    """D = 64 runs on CTA pairs, D = 32 on single CTAs (32/8 heads, d = 128);
    prefixes end mid-page, so the block is committed into a partly filled
    page (and, for the empty prefix, at slot 0)."""
    P = [0, 768, 1344, 4096]
    case = workloads.make_decode_case(P, D=D, Hq=32, Hkv=8, d=128, page_size=S, seed=S + D)
    r = DecodeRun(case)
    out = r.run(commit=True)
    assert r.status() == 0
    ref = oracle.decode(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix)
    assert_close(out, ref, what=f"decode S={S} D={D}")
    _check_commit(case, r, D)


@pytest.mark.parametrize("S", SIZES)
def test_extend_with_commit(cuda_lib, S):
    """9 new tokens after prefixes of any length: the new rows start mid-page
    and cross page boundaries (P = S - 4)."""
    P = [5, S - 4, 3 * S + 1, 1000]
    n = 9
    case = workloads.make_decode_case(P, D=n, Hq=32, Hkv=8, d=128, page_size=S, seed=S)
    r = DecodeRun(case)
    out = r.run(commit=True, extend=True)
    assert r.status() == 0
    ref = oracle.extend(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix)
    assert_close(out, ref, what=f"extend S={S}")
    _check_commit(case, r, n)


@pytest.mark.parametrize("S", SIZES)
def test_prefill_page_write(cuda_lib, S):
    lens = [300, 512, 70]
    case = workloads.make_prefill_case(lens, D=64, Hq=32, Hkv=8, d=128, page_size=S, seed=S)
    r = PrefillRun(case)
    out = r.run()
    assert r.status() == 0
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, case.D)
    assert_close(out, ref, what=f"prefill S={S}")
    cu = case.cu_seqlens.tolist()
    for name, pool_dev, pool_src, src in (("k", r.k_pool, case.pool.k_pool, case.k),
                                          ("v", r.v_pool, case.pool.v_pool, case.v)):
        want = pool_src.view(torch.int16).numpy().copy()
        for b, L in enumerate(lens):
            blk = src[cu[b]:cu[b + 1]].view(torch.int16).numpy()[None]
            want = oracle.commit(want, case.pool.page_table[b:b + 1], [0], blk, L, S)
        assert np.array_equal(pool_dev.cpu().view(torch.int16).numpy(), want), f"{name}, S={S}"


@pytest.mark.parametrize("S", SIZES)
def test_multicanvas_with_promotion(cuda_lib, S):
    """Arena keys gathered through pages of S tokens with their stored
    positions; the promoted rows appended at arena_len, bit-exact."""
    c = workloads.make_multicanvas_case(3, 200, 3, 96, Hq=32, Hkv=8, d=128, page_size=S,
                                        seed=S, shuffle_live=True)
    r = MulticanvasRun(c)
    out = r.run()
    assert r.status() == 0
    m = np.arange(c.q_live.shape[1])[None, :] < c.live_count.numpy()[:, None]
    ref = oracle.multicanvas(c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k,
                             c.arena_v, c.arena_pos, c.prompt_len, c.canvas_len)
    assert_close(out.cpu()[torch.from_numpy(m)], ref[m], what=f"multicanvas S={S}")
    k = c.pool.k_pool.view(torch.int16).numpy().copy()
    v = c.pool.v_pool.view(torch.int16).numpy().copy()
    kv_pos = c.kv_pos.numpy().copy()
    for b in range(c.B):
        n = int(c.commit_count[b])
        rows = c.commit_rows[b, :n].long()
        A = int(c.arena_len[b])
        pt = c.pool.page_table[b:b + 1]
        k = oracle.commit(k, pt, [A], c.k_live[b, rows].view(torch.int16).numpy()[None], n, S)
        v = oracle.commit(v, pt, [A], c.v_live[b, rows].view(torch.int16).numpy()[None], n, S)
        for i in range(n):
            e = A + i
            kv_pos[int(pt[0, e // S]), e % S] = int(c.live_pos[b, int(rows[i])])
    assert np.array_equal(r.k_pool.cpu().view(torch.int16).numpy(), k)
    assert np.array_equal(r.v_pool.cpu().view(torch.int16).numpy(), v)
    assert np.array_equal(r.kv_pos.cpu().numpy(), kv_pos)
    assert np.array_equal(r.arena_len.cpu().numpy(), (c.arena_len + c.commit_count).numpy())
