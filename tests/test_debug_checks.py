"""BCA_DEBUG=1: host-side checks of lengths, positions and page tables
before a launch (the page table used with stricter error checking, "Paged
Attention").

The entry points are called through the C ABI with host arrays for the
lengths and page tables (the checks copy them to the host anyway) and
placeholder tensor pointers: a refused request returns before any launch.
Requests the checks accept go on to the device, so they are only issued
where there is no GPU (there the call then fails on the missing device,
with an error that is not one of the checks' codes)."""
import ctypes

import numpy as np
import pytest

import block_causal_paged_gb300 as bca

FAKE = 1 << 20       # 16-byte aligned placeholder for tensors never touched
WS = 1 << 30         # workspace size that passes every size check
CHECK_CODES = {bca.ERR_INVALID_ARG, bca.ERR_CAPACITY, bca.ERR_PAGE_RANGE, bca.ERR_PAGE_SHARED}


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture
def debug_env(monkeypatch):
    bca.load()
    monkeypatch.setenv("BCA_DEBUG", "1")
    yield
    monkeypatch.delenv("BCA_DEBUG", raising=False)


def _p(a):
    return a.ctypes.data


def _decode(d, pt, plen, commit=1, extend=False):
    lib = bca.load()
    fn = lib.bca_extend if extend else lib.bca_decode
    return fn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, _p(pt), _p(plen), FAKE, commit, FAKE,
              WS, None)


def _pool(B, max_pages, num_pages, seed=0):
    """Each sequence its own pages, drawn without repetition."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)[:B * max_pages]
    return perm.reshape(B, max_pages).astype(np.int32)


def test_decode_refusals(debug_env):
    B, D, S, maxp, npg = 3, 64, 16, 12, 64
    d = bca.dims(B, D, 8, 2, 128, S, npg, maxp)
    pt = _pool(B, maxp, npg)
    ok = np.array([0, 64, 128], np.int32)
    # a prefix that is not a whole number of blocks (decode), negative, too long
    assert _decode(d, pt, np.array([0, 65, 128], np.int32)) == bca.ERR_INVALID_ARG
    assert _decode(d, pt, np.array([0, -64, 128], np.int32)) == bca.ERR_INVALID_ARG
    assert _decode(d, pt, np.array([0, 64, maxp * S - D + 64], np.int32)) == bca.ERR_CAPACITY
    # a page id outside the pool in a used entry; an unused entry may hold anything
    bad = pt.copy()
    bad[1, 3] = npg
    assert _decode(d, bad, ok) == bca.ERR_PAGE_RANGE
    unused = pt.copy()
    unused[0, maxp - 1] = -5
    if not _has_gpu():
        assert _decode(d, unused, ok) not in CHECK_CODES
    # a page the commit writes (sequence 2, positions 128..191 = entries 8..11)
    # also read by sequence 1
    shared = pt.copy()
    shared[1, 0] = pt[2, 9]
    assert _decode(d, shared, ok) == bca.ERR_PAGE_SHARED
    # the same page read by two sequences (a shared prefix) is allowed; not
    # when the commit writes it
    prefix = pt.copy()
    prefix[1, 0] = pt[2, 0]
    if not _has_gpu():
        assert _decode(d, prefix, ok, commit=0) not in CHECK_CODES
    # one page twice in one sequence's used entries
    twice = pt.copy()
    twice[2, 1] = pt[2, 0]
    assert _decode(d, twice, ok, commit=0) == bca.ERR_PAGE_SHARED


def test_extend_any_prefix(debug_env):
    B, n, S, maxp, npg = 2, 9, 16, 8, 32
    d = bca.dims(B, n, 8, 2, 128, S, npg, maxp)
    pt = _pool(B, maxp, npg, seed=1)
    if not _has_gpu():
        assert _decode(d, pt, np.array([5, 100], np.int32), extend=True) not in CHECK_CODES
    assert _decode(d, pt, np.array([5, maxp * S - n + 1], np.int32), extend=True) == bca.ERR_CAPACITY


def test_prefill_refusals(debug_env):
    B, S, maxp, npg = 3, 16, 8, 48
    d = bca.dims(B, 64, 8, 2, 128, S, npg, maxp)
    pt = _pool(B, maxp, npg, seed=2)
    lib = bca.load()

    def call(cu, total, max_len, pages=pt):
        return lib.bca_prefill(ctypes.byref(d), FAKE, FAKE, FAKE, _p(cu), total, max_len, FAKE,
                               FAKE, _p(pages), FAKE, FAKE, WS, None)

    cu = np.array([0, 64, 192, 320], np.int32)
    assert call(np.array([1, 64, 192, 320], np.int32), 320, 128) == bca.ERR_INVALID_ARG
    assert call(np.array([0, 128, 64, 320], np.int32), 320, 128) == bca.ERR_INVALID_ARG  # decreasing
    assert call(cu, 321, 128) == bca.ERR_INVALID_ARG                                      # total
    assert call(cu, 320, 100) == bca.ERR_INVALID_ARG                                      # max_seqlen
    shared = pt.copy()
    shared[0, 1] = pt[1, 0]   # prefill writes every page of every sequence
    assert call(cu, 320, 128, shared) == bca.ERR_PAGE_SHARED
    if not _has_gpu():
        assert call(cu, 320, 128) not in CHECK_CODES


def test_commit_and_qkv_post_refusals(debug_env):
    B, n, S, maxp, npg = 2, 16, 16, 4, 16
    d = bca.dims(B, n, 8, 2, 64, S, npg, maxp)
    pt = _pool(B, maxp, npg, seed=3)
    lib = bca.load()

    def commit(start, pages=pt, k=n):
        return lib.bca_commit_kv(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, _p(pages), _p(start), k,
                                 FAKE, WS, None)

    assert commit(np.array([-1, 0], np.int32)) == bca.ERR_INVALID_ARG
    assert commit(np.array([0, maxp * S - n + 1], np.int32)) == bca.ERR_CAPACITY
    bad = pt.copy()
    bad[0, 0] = -1
    assert commit(np.array([0, 16], np.int32), bad) == bca.ERR_PAGE_RANGE

    def qkv(wp, pages=pt):
        return lib.bca_qkv_post(ctypes.byref(d), FAKE, FAKE, None, None, 1e-6, 0.0, FAKE, FAKE,
                                FAKE, _p(wp), FAKE, FAKE, _p(pages), None, FAKE, WS, None)

    wp = np.stack([np.arange(n), 16 + np.arange(n)]).astype(np.int32)
    dup = wp.copy()
    dup[1, 5] = dup[1, 4]     # two tokens write one slot
    assert qkv(dup) == bca.ERR_INVALID_ARG
    far = wp.copy()
    far[0, 0] = maxp * S
    assert qkv(far) == bca.ERR_CAPACITY
    cross = pt.copy()
    cross[1, 1] = pt[0, 0]    # both sequences write into one page
    assert qkv(wp, cross) == bca.ERR_PAGE_SHARED
    skipped = wp.copy()
    skipped[0, :] = -1        # negative positions are not written and not checked
    if not _has_gpu():
        assert qkv(skipped, cross) not in CHECK_CODES


def test_multicanvas_refusals(debug_env):
    B, C, S, maxp, npg = 2, 32, 16, 8, 32
    d = bca.dims(B, C, 8, 2, 128, S, npg, maxp)
    pt = _pool(B, maxp, npg, seed=4)
    lib = bca.load()
    max_live, max_commit = 48, 8

    def call(live, arena, rows=None, count=None, pages=pt):
        return lib.bca_multicanvas(ctypes.byref(d), FAKE, FAKE, FAKE, None, _p(live), max_live, 16,
                                   2, FAKE, FAKE, _p(pages), FAKE, _p(arena),
                                   None if rows is None else _p(rows),
                                   None if count is None else _p(count), max_commit, FAKE, FAKE,
                                   WS, None)

    live = np.array([40, 48], np.int32)
    arena = np.array([16, 40], np.int32)
    assert call(np.array([49, 0], np.int32), arena) == bca.ERR_INVALID_ARG
    assert call(live, np.array([16, maxp * S + 1], np.int32)) == bca.ERR_CAPACITY
    rows = np.zeros((B, max_commit), np.int32)
    rows[0, :3] = [0, 5, 5]   # a live row promoted twice
    assert call(live, arena, rows, np.array([3, 0], np.int32)) == bca.ERR_INVALID_ARG
    rows[0, :3] = [0, 5, 7]
    assert call(live, np.array([16, maxp * S - 2], np.int32), rows,
                np.array([0, 3], np.int32)) == bca.ERR_CAPACITY
    shared = pt.copy()
    shared[1, 0] = pt[0, 1]   # sequence 0's promotion writes entry 1, read by sequence 1
    assert call(live, arena, rows, np.array([3, 0], np.int32), shared) == bca.ERR_PAGE_SHARED
    if not _has_gpu():
        assert call(live, arena, rows, np.array([3, 0], np.int32)) not in CHECK_CODES


def test_checks_are_off_without_the_variable(monkeypatch):
    """Without BCA_DEBUG the host does not read the page table: the same bad
    request goes on to the device (where its accesses are checked and
    skipped).  Issued only where there is no GPU."""
    if _has_gpu():
        pytest.skip("would launch with placeholder tensors")
    monkeypatch.delenv("BCA_DEBUG", raising=False)
    B, D, S, maxp, npg = 2, 64, 16, 8, 16
    d = bca.dims(B, D, 8, 2, 128, S, npg, maxp)
    pt = _pool(B, maxp, npg, seed=5)
    pt[0, 0] = npg + 3
    assert _decode(d, pt, np.array([0, 64], np.int32)) not in CHECK_CODES
