"""GPU parity of bca_multicanvas (live rows over an arena) and its promotion."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_cases import MulticanvasRun, assert_close

pytestmark = pytest.mark.gpu


def _ref(c, window=0):
    return oracle.multicanvas(c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k,
                              c.arena_v, c.arena_pos, c.prompt_len, c.canvas_len, window=window)


def _live_mask(c):
    n = c.q_live.shape[1]
    return (np.arange(n)[None, :] < c.live_count.numpy()[:, None])


def _expected_promotion(c):
    S = c.pool.page_size
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
    return k, v, kv_pos, (c.arena_len + c.commit_count).numpy()


@pytest.mark.parametrize("seed", [0, 1])
def test_multicanvas_b16(cuda_lib, seed):
    """Batch 16, prompt 1024, 3 canvases of 256 with 30-100% live rows, 32/8
    heads, d = 128; then 25% of each canvas's live rows are promoted."""
    c = workloads.multicanvas_b16(seed=seed)
    r = MulticanvasRun(c)
    out = r.run()
    assert r.status() == 0
    m = _live_mask(c)
    assert_close(out.cpu()[torch.from_numpy(m)], _ref(c)[m], what=f"multicanvas seed {seed}")
    k, v, kv_pos, alen = _expected_promotion(c)
    assert np.array_equal(r.k_pool.cpu().view(torch.int16).numpy(), k)
    assert np.array_equal(r.v_pool.cpu().view(torch.int16).numpy(), v)
    assert np.array_equal(r.kv_pos.cpu().numpy(), kv_pos)
    assert np.array_equal(r.arena_len.cpu().numpy(), alen)


def _degenerate_case():
    """Four sequences: one with no live rows (nothing to attend to or
    promote), one whose arena is empty (its live rows see only each other),
    two ordinary ones."""
    c = workloads.make_multicanvas_case(4, 128, 3, 64, Hq=32, Hkv=8, d=128, seed=9)
    c.live_count[1] = 0
    c.commit_count[1] = 0
    c.arena_len[2] = 0
    c.arena_k[2], c.arena_v[2], c.arena_pos[2] = c.arena_k[2][:0], c.arena_v[2][:0], c.arena_pos[2][:0]
    return c


def test_no_live_rows_and_empty_arena(cuda_lib):
    c = _degenerate_case()
    r = MulticanvasRun(c)
    out = r.run()
    assert r.status() == 0
    m = _live_mask(c)
    assert_close(out.cpu()[torch.from_numpy(m)], _ref(c)[m], what="no live rows / empty arena")
    k, v, kv_pos, alen = _expected_promotion(c)
    assert np.array_equal(r.k_pool.cpu().view(torch.int16).numpy(), k)
    assert np.array_equal(r.v_pool.cpu().view(torch.int16).numpy(), v)
    assert np.array_equal(r.kv_pos.cpu().numpy(), kv_pos)
    assert np.array_equal(r.arena_len.cpu().numpy(), alen)
    # the same under a narrow sliding window (band kernel)
    c = _degenerate_case()
    r = MulticanvasRun(c, promote=False)
    out = r.run(window=64)
    assert r.status() == 0
    assert_close(out.cpu()[torch.from_numpy(m)], _ref(c, 64)[m], what="window 64, degenerate")


def test_multicanvas_small_shapes(cuda_lib):
    c = workloads.make_multicanvas_case(3, 40, 4, 24, Hq=6, Hkv=2, d=64, seed=5)
    r = MulticanvasRun(c)
    out = r.run()
    assert r.status() == 0
    m = _live_mask(c)
    assert_close(out.cpu()[torch.from_numpy(m)], _ref(c)[m], what="small multicanvas")


def test_live_order_equivariance(cuda_lib):
    """Listing the live rows in another order permutes the outputs."""
    a = workloads.make_multicanvas_case(2, 64, 3, 64, Hq=8, Hkv=2, d=128, seed=9)
    b = workloads.make_multicanvas_case(2, 64, 3, 64, Hq=8, Hkv=2, d=128, seed=9,
                                        shuffle_live=True)
    oa = MulticanvasRun(a, promote=False).run().cpu()
    ob = MulticanvasRun(b, promote=False).run().cpu()
    for s in range(2):
        n = int(a.live_count[s])
        ia = {int(p): i for i, p in enumerate(a.live_pos[s, :n])}
        for i, p in enumerate(b.live_pos[s, :n]):
            err = (ob[s, i].float() - oa[s, ia[int(p)]].float()).abs().max()
            assert err <= 2e-2


def test_all_rows_live_one_canvas_is_block_decode(cuda_lib):
    """With every row live and one canvas, the live-position list may be
    omitted (row r at prompt_len + r) and the step equals a block decode."""
    c = workloads.make_multicanvas_case(2, 128, 1, 64, Hq=8, Hkv=2, d=128, active_lo=1.0,
                                        active_hi=1.0, seed=4)
    r = MulticanvasRun(c, pass_positions=False, promote=False)
    out = r.run()
    assert r.status() == 0
    ref = oracle.decode(c.q_live, c.k_live, c.v_live, c.arena_k, c.arena_v)
    assert_close(out, ref, what="one canvas, all live")


def test_sliding_window_five_canvases(cuda_lib):
    """"Advancement 11": a 1024-token sliding-window layer over a 1024-token
    prompt and 5 canvases of 256 (positions up to 2304): later canvases lose
    the start of the prompt."""
    c = workloads.make_multicanvas_case(4, 1024, 5, 256, Hq=32, Hkv=8, d=128, seed=21)
    r = MulticanvasRun(c)
    out = r.run(window=1024)
    assert r.status() == 0
    m = _live_mask(c)
    assert_close(out.cpu()[torch.from_numpy(m)], _ref(c, 1024)[m], what="window 1024, 5 canvases")


@pytest.mark.parametrize("window", [1, 64, 200])
def test_sliding_window_small(cuda_lib, window):
    c = workloads.make_multicanvas_case(3, 300, 4, 96, Hq=6, Hkv=2, d=64, seed=22)
    r = MulticanvasRun(c)
    out = r.run(window=window)
    assert r.status() == 0
    m = _live_mask(c)
    assert_close(out.cpu()[torch.from_numpy(m)], _ref(c, window)[m], what=f"window {window}")


def test_wide_window_equals_no_window(cuda_lib):
    c = workloads.make_multicanvas_case(2, 200, 3, 64, Hq=8, Hkv=2, d=128, seed=23,
                                        commit_frac=0.0)
    a = MulticanvasRun(c).run().clone()
    b = MulticanvasRun(c).run(window=10 ** 6).clone()
    m = torch.from_numpy(_live_mask(c))
    assert torch.equal(a.cpu()[m], b.cpu()[m])


def test_device_error_bad_arena_page_is_reported(cuda_lib):
    """A page id outside the pool in a sequence's arena is reported in the
    status word; the kernels skip it and the outputs stay finite."""
    import block_causal_paged_gb300 as bca
    c = workloads.make_multicanvas_case(3, 40, 4, 24, Hq=6, Hkv=2, d=64, seed=5)
    r = MulticanvasRun(c, promote=False)
    r.page_table[1, 0] = c.pool.num_pages + 3
    out = r.run()
    assert r.status() == bca.ERR_DEVICE_PAGE_OOB
    assert torch.isfinite(out.float()).all()


def test_device_error_bad_arena_length_is_reported(cuda_lib):
    import block_causal_paged_gb300 as bca
    c = workloads.make_multicanvas_case(3, 40, 4, 24, Hq=6, Hkv=2, d=64, seed=5)
    r = MulticanvasRun(c, promote=False)
    r.arena_len[2] = c.pool.max_pages_per_seq * c.pool.page_size + 16
    r.run()
    assert r.status() == bca.ERR_DEVICE_BAD_LENGTH
