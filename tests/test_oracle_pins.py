"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test names what it pins against: brute-force enumeration written from a
different (but equivalent) statement of the rule, PyTorch SDPA in fp64 for the
special cases the pages reduce to, closed forms, the pages' worked examples
(tests/golden/), and invariants the pages state.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    meta, grid = {}, []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0].isupper() and len(parts) == 2 and parts[1].lstrip("-").isdigit():
            meta[parts[0]] = int(parts[1])
        else:
            grid.append(parts)
    return meta, np.array(grid)


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


# ---------------------------------------------------------------------------
# 1. brute force: per-row enumeration with the "key limit" statement of the rule
# ---------------------------------------------------------------------------

def _brute(q, k, v, q_pos, k_pos, P0, D, scale):
    """A query at position p sees exactly the keys at positions below
    limit(p) = P0 if p < P0 else P0 + D * (floor((p - P0) / D) + 1)
    (earlier blocks and its own block, nothing later)."""
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((Tq, Hq, d))
    for i in range(Tq):
        p = int(q_pos[i])
        limit = P0 if p < P0 else P0 + D * ((p - P0) // D + 1)
        keys = [j for j in range(k.shape[0]) if int(k_pos[j]) < limit]
        for h in range(Hq):
            g = h // G
            s = [scale * math.fsum(float(q[i, h, c]) * float(k[j, g, c]) for c in range(d))
                 for j in keys]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            z = math.fsum(w)
            for c in range(d):
                out[i, h, c] = math.fsum(w[t] * float(v[keys[t], g, c]) for t in range(len(keys))) / z
    return out


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_random_positions(seed):
    rng = np.random.default_rng(seed)
    Hkv, G, d = 2, int(rng.integers(1, 4)), 8
    Hq = Hkv * G
    D = int(rng.integers(1, 6))
    P0 = int(rng.integers(0, 10))
    Tk = int(rng.integers(4, 24))
    k_pos = rng.permutation(Tk + 5)[:Tk]             # distinct, unordered positions
    q_pos = rng.choice(k_pos, size=min(Tk, 7), replace=False)
    q, k, v = _rand((q_pos.size, Hq, d), seed), _rand((Tk, Hkv, d), seed + 100), \
        _rand((Tk, Hkv, d), seed + 200)
    # some query might see no key only if it had no key at or before its block;
    # every query position is also a key position, so it always sees itself
    scale = 0.37
    got = oracle.attention(q, k, v, q_pos, k_pos, P0, D, scale=scale)
    ref = _brute(q.numpy(), k.numpy(), v.numpy(), q_pos, k_pos, P0, D, scale)
    assert np.abs(got - ref).max() < 1e-12


def test_default_scale_is_inverse_sqrt_d():
    q, k, v = _rand((3, 2, 16), 1), _rand((5, 1, 16), 2), _rand((5, 1, 16), 3)
    pos = np.arange(5)
    a = oracle.attention(q, k, v, pos[2:], pos, 0, 1)
    b = _brute(q.numpy(), k.numpy(), v.numpy(), pos[2:], pos, 0, 1, 1 / 4.0)
    assert np.abs(a - b).max() < 1e-12


# ---------------------------------------------------------------------------
# 2. library special cases: PyTorch SDPA in fp64
# ---------------------------------------------------------------------------

def _sdpa(q, k, v, **kw):
    """q [T, Hq, d], k/v [Tk, Hkv, d] -> SDPA with contiguous GQA groups."""
    G = q.shape[1] // k.shape[1]
    qh = q.transpose(0, 1)
    kh = k.repeat_interleave(G, dim=1).transpose(0, 1)
    vh = v.repeat_interleave(G, dim=1).transpose(0, 1)
    return F.scaled_dot_product_attention(qh, kh, vh, **kw).transpose(0, 1)


@pytest.mark.parametrize("T,Hq,Hkv,d", [(19, 4, 2, 16), (33, 6, 3, 8)])
def test_block_size_one_prefill_is_causal(T, Hq, Hkv, d):
    q, k, v = _rand((T, Hq, d), 3), _rand((T, Hkv, d), 4), _rand((T, Hkv, d), 5)
    got = oracle.prefill(q, k, v, [0, T], D=1)
    ref = _sdpa(q, k, v, is_causal=True).numpy()
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("T", [8, 24])
def test_single_block_prefill_is_unmasked(T):
    q, k, v = _rand((T, 4, 16), 6), _rand((T, 2, 16), 7), _rand((T, 2, 16), 8)
    got = oracle.prefill(q, k, v, [0, T], D=T)
    ref = _sdpa(q, k, v).numpy()
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("T,D", [(24, 4), (40, 8), (30, 5)])
def test_prefill_matches_sdpa_with_block_lower_triangular_mask(T, D):
    q, k, v = _rand((T, 4, 16), 9), _rand((T, 1, 16), 10), _rand((T, 1, 16), 11)
    nb = T // D
    # allowed iff key block <= query block: lower-triangular blocks of ones
    allowed = torch.kron(torch.tril(torch.ones(nb, nb)), torch.ones(D, D)).bool()
    got = oracle.prefill(q, k, v, [0, T], D=D)
    ref = _sdpa(q, k, v, attn_mask=allowed).numpy()
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("P,D", [(0, 16), (48, 16), (37, 1), (64, 64)])
def test_decode_attends_whole_prefix_and_block(P, D):
    """The decode queries see every prefix key and every key of their block,
    i.e. plain unmasked attention over prefix ++ block (block size 1 is the
    ordinary single-token causal decode step)."""
    B, Hq, Hkv, d = 2, 4, 2, 32
    q, kb, vb = _rand((B, D, Hq, d), 12), _rand((B, D, Hkv, d), 13), _rand((B, D, Hkv, d), 14)
    kp, vp = _rand((B, P, Hkv, d), 15), _rand((B, P, Hkv, d), 16)
    got = oracle.decode(q, kb, vb, list(kp), list(vp))
    for b in range(B):
        ref = _sdpa(q[b], torch.cat([kp[b], kb[b]]), torch.cat([vp[b], vb[b]])).numpy()
        assert np.abs(got[b] - ref).max() < 1e-12


# ---------------------------------------------------------------------------
# 3. closed forms
# ---------------------------------------------------------------------------

def test_two_token_softmax_by_hand():
    # q.k0 = 0, q.k1 = ln 3 -> weights (1/4, 3/4); one-hot values read them out
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[0.0, 0.0]], [[math.log(3.0), 0.0]]])
    v = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    out = oracle.attention(q, k, v, [1], [0, 1], P0=0, D=2, scale=1.0)
    assert np.allclose(out[0, 0], [0.25, 0.75], atol=1e-15, rtol=0)
    # with block size 1 the query at position 0 sees only key 0
    out0 = oracle.attention(q, k, v, [0], [0, 1], P0=0, D=1, scale=1.0)
    assert np.array_equal(out0[0, 0], [1.0, 0.0])


def test_constant_values_give_constant_output():
    T, D = 20, 4
    q, k = _rand((T, 4, 8), 17), _rand((T, 2, 8), 18)
    v = torch.full((T, 2, 8), 0.625, dtype=torch.float64)
    out = oracle.prefill(q, k, v, [0, T], D=D)
    assert np.abs(out - 0.625).max() < 1e-14


def test_one_hot_values_recover_weights():
    T, D, d = 12, 3, 16
    q, k = _rand((T, 2, d), 19), _rand((T, 1, d), 20)
    v = torch.zeros((T, 1, d), dtype=torch.float64)
    for j in range(T):
        v[j, 0, j] = 1.0
    out = oracle.prefill(q, k, v, [0, T], D=D)
    scale = 1 / math.sqrt(d)
    for i in range(T):
        visible = (i // D + 1) * D
        for h in range(2):
            s = scale * (k[:visible, 0] @ q[i, h]).numpy()
            w = np.exp(s - s.max())
            w /= w.sum()
            assert np.abs(out[i, h, :visible] - w).max() < 1e-14
            assert np.all(out[i, h, visible:T] == 0.0)


# ---------------------------------------------------------------------------
# 4. the pages' worked examples
# ---------------------------------------------------------------------------

def test_background_figure_tile_grid():
    meta, grid = _golden("background_tiles_d2_b2.txt")
    T = meta["D"] * meta["BLOCKS"]
    pos = np.arange(T)
    got = oracle.tile_classes(pos, pos, 0, meta["D"], meta["TILE"], meta["TILE"])
    assert (got == grid).all()
    assert (got == "F").sum() == 6 and (got == "S").sum() == 3 and (got == "P").sum() == 0


def test_kv_cache_worked_example():
    meta, grid = _golden("kv_cache_d4_prompt10.txt")
    D, prompt = meta["D"], meta["PROMPT"]
    cached = (prompt // D) * D               # completed blocks only
    assert cached == meta["CACHED_TOKENS"]
    assert cached // D == meta["COMPLETED_BLOCKS"] == meta["NEXT_ACTIVE_BLOCK"]
    assert prompt - cached + meta["MASKED_IN_NEXT_BLOCK"] == D
    T = meta["MAX_PREFILL"]
    pos = np.arange(T)
    got = oracle.tile_classes(pos, pos, 0, D, meta["TILE"], meta["TILE"])
    assert (got == grid).all()
    # decoding B2 against the cached B0, B1 equals rows 8..11 of the prefill
    # over the 12 tokens B0 B1 B2 (the block sees itself bidirectionally)
    q, k, v = _rand((12, 2, 8), 21), _rand((12, 1, 8), 22), _rand((12, 1, 8), 23)
    dec = oracle.decode(q[cached:].unsqueeze(0), k[cached:].unsqueeze(0),
                        v[cached:].unsqueeze(0), [k[:cached]], [v[:cached]])
    pre = oracle.prefill(q, k, v, [0, 12], D=D)
    assert np.abs(dec[0] - pre[cached:]).max() < 1e-13


@pytest.mark.parametrize("T,D", [(64, 4), (256, 64), (96, 16)])
def test_aligned_tiles_have_no_partial_tile(T, D):
    """"FlexAttention with Aligned Tiles": with tile size equal to the block
    size every tile is fully included or fully excluded."""
    pos = np.arange(T)
    got = oracle.tile_classes(pos, pos, 0, D, D, D)
    assert (got == "P").sum() == 0
    n = T // D
    assert (got == "F").sum() == n * (n + 1) // 2


def test_prefill_8192_tile_counts_at_128():
    """4 x 8192 prefill, D = 64, 128 x 128 tiles: per (sequence, head) the
    lower triangle is full, the diagonal partial (its upper-right 64 x 64
    quadrant masked) and the upper triangle skipped."""
    pos = np.arange(8192)
    got = oracle.tile_classes(pos, pos, 0, 64, 128, 128)
    assert (got == "F").sum() == 2016
    assert (got == "P").sum() == 64
    assert (got == "S").sum() == 2016
    mask = oracle.block_causal_mask(np.arange(128), np.arange(128), 0, 64)
    assert mask[:64, 64:].sum() == 0 and mask.sum() == 3 * 64 * 64


# ---------------------------------------------------------------------------
# 5. invariants the pages state
# ---------------------------------------------------------------------------

def test_key_storage_order_does_not_matter():
    """"Advancement 10": masks address keys by position, so compacting or
    reordering the cache leaves the result unchanged."""
    rng = np.random.default_rng(3)
    Tk, P0, D = 30, 6, 4
    k_pos = np.arange(Tk)
    q_pos = np.arange(P0, Tk)
    q, k, v = _rand((q_pos.size, 4, 8), 24), _rand((Tk, 2, 8), 25), _rand((Tk, 2, 8), 26)
    a = oracle.attention(q, k, v, q_pos, k_pos, P0, D)
    perm = rng.permutation(Tk)
    b = oracle.attention(q, k[perm], v[perm], q_pos, k_pos[perm], P0, D)
    assert np.abs(a - b).max() < 1e-13


def test_appending_blocks_leaves_completed_rows_unchanged():
    """"Background": a completed block's representation cannot change."""
    D, T = 4, 16
    q, k, v = _rand((T + 2 * D, 2, 8), 27), _rand((T + 2 * D, 1, 8), 28), _rand((T + 2 * D, 1, 8), 29)
    short = oracle.prefill(q[:T], k[:T], v[:T], [0, T], D=D)
    long = oracle.prefill(q, k, v, [0, T + 2 * D], D=D)
    assert np.array_equal(short, long[:T])


def test_within_block_permutation_equivariance():
    """No positional op inside the kernel ("Advancement 10": rotary phases are
    baked into Q/K before the call): permuting a block's rows (queries and its
    own keys/values together) permutes the outputs."""
    B, D, P = 1, 8, 16
    q, kb, vb = _rand((B, D, 4, 8), 30), _rand((B, D, 2, 8), 31), _rand((B, D, 2, 8), 32)
    kp, vp = _rand((B, P, 2, 8), 33), _rand((B, P, 2, 8), 34)
    perm = torch.randperm(D, generator=torch.Generator().manual_seed(5))
    a = oracle.decode(q, kb, vb, list(kp), list(vp))
    b = oracle.decode(q[:, perm], kb[:, perm], vb[:, perm], list(kp), list(vp))
    assert np.abs(a[:, perm.numpy()] - b).max() < 1e-13


@pytest.mark.parametrize("j", [0, 2, 5])
def test_decode_of_block_equals_prefill_rows(j):
    D, nblk = 4, 6
    T = D * nblk
    q, k, v = _rand((T, 4, 8), 35), _rand((T, 2, 8), 36), _rand((T, 2, 8), 37)
    pre = oracle.prefill(q, k, v, [0, T], D=D)
    s = j * D
    dec = oracle.decode(q[s:s + D][None], k[s:s + D][None], v[s:s + D][None], [k[:s]], [v[:s]])
    assert np.abs(dec[0] - pre[s:s + D]).max() < 1e-13


def test_multicanvas_one_full_canvas_is_block_decode():
    c = workloads.make_multicanvas_case(2, 32, 1, 16, 4, 2, 16, active_lo=1.0, active_hi=1.0,
                                        seed=3, fill_bits_value=None)
    assert (c.live_count == 16).all()
    got = oracle.multicanvas(c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k,
                             c.arena_v, c.arena_pos, 32, 16)
    ref = oracle.decode(c.q_live, c.k_live, c.v_live, c.arena_k, c.arena_v)
    assert np.abs(got - ref).max() < 1e-13


def test_multicanvas_matches_per_canvas_prefix_attention():
    """"Advancement 13": canvas c attends exactly the contiguous prefix of
    positions below prompt + C*(c+1); evaluate it with unmasked SDPA on the
    logically ordered prefix."""
    c = workloads.make_multicanvas_case(2, 24, 3, 8, 4, 2, 16, seed=4, fill_bits_value=None)
    got = oracle.multicanvas(c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k,
                             c.arena_v, c.arena_pos, 24, 8)
    for b in range(2):
        n = int(c.live_count[b])
        pos = torch.cat([c.arena_pos[b], c.live_pos[b, :n].long()])
        keys = torch.cat([c.arena_k[b], c.k_live[b, :n]]).double()
        vals = torch.cat([c.arena_v[b], c.v_live[b, :n]]).double()
        order = torch.argsort(pos)
        assert torch.equal(pos[order], torch.arange(24 + 24))
        keys, vals = keys[order], vals[order]
        for r in range(n):
            p = int(c.live_pos[b, r])
            lim = 24 + 8 * ((p - 24) // 8 + 1)
            ref = _sdpa(c.q_live[b, r:r + 1].double(), keys[:lim], vals[:lim]).numpy()
            assert np.abs(got[b, r] - ref[0]).max() < 1e-13


def test_multicanvas_arena_order_invariance():
    c = workloads.make_multicanvas_case(1, 16, 2, 8, 2, 1, 8, seed=5, fill_bits_value=None)
    args = (c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count)
    a = oracle.multicanvas(*args, c.arena_k, c.arena_v, c.arena_pos, 16, 8)
    perm = torch.randperm(c.arena_k[0].shape[0], generator=torch.Generator().manual_seed(1))
    b = oracle.multicanvas(*args, [c.arena_k[0][perm]], [c.arena_v[0][perm]],
                           [c.arena_pos[0][perm]], 16, 8)
    assert np.abs(a - b).max() < 1e-13


@pytest.mark.parametrize("W", [1, 5, 17, 40])
def test_sliding_window_multicanvas_is_a_windowed_prefix(W):
    """"Advancement 11": a sliding-window layer band-masks the entries outside
    the window.  With positions 0..N-1 in logical order, a live row at p sees
    the contiguous slice [max(0, p - W + 1), lim(p)); evaluate it with
    unmasked SDPA on that slice."""
    c = workloads.make_multicanvas_case(2, 24, 3, 8, 4, 2, 16, seed=6, fill_bits_value=None)
    got = oracle.multicanvas(c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k,
                             c.arena_v, c.arena_pos, 24, 8, window=W)
    for b in range(2):
        n = int(c.live_count[b])
        pos = torch.cat([c.arena_pos[b], c.live_pos[b, :n].long()])
        keys = torch.cat([c.arena_k[b], c.k_live[b, :n]]).double()
        vals = torch.cat([c.arena_v[b], c.v_live[b, :n]]).double()
        order = torch.argsort(pos)
        assert torch.equal(pos[order], torch.arange(24 + 24))
        keys, vals = keys[order], vals[order]
        for r in range(n):
            p = int(c.live_pos[b, r])
            lim = 24 + 8 * ((p - 24) // 8 + 1)
            lo = max(0, p - W + 1)
            ref = _sdpa(c.q_live[b, r:r + 1].double(), keys[lo:lim], vals[lo:lim]).numpy()
            assert np.abs(got[b, r] - ref[0]).max() < 1e-13


def test_window_wider_than_every_distance_is_no_band():
    c = workloads.make_multicanvas_case(2, 24, 3, 8, 4, 2, 16, seed=7, fill_bits_value=None)
    args = (c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k, c.arena_v,
            c.arena_pos, 24, 8)
    assert np.array_equal(oracle.multicanvas(*args), oracle.multicanvas(*args, window=48),
                          equal_nan=True)
    band = oracle.sliding_window_mask([10, 11], [0, 5, 9, 10, 11, 12], 3)
    assert band.tolist() == [[0, 0, 1, 1, 1, 1], [0, 0, 1, 1, 1, 1]]


# ---------------------------------------------------------------------------
# 6. commit: a bit copy, checked against an independent flat-index scatter
# ---------------------------------------------------------------------------

def test_commit_is_bit_copy_and_keeps_other_slots():
    c = workloads.tiny_decode(fill_bits_value=workloads.BF16_CANARY_BITS)
    S = c.pool.page_size
    pool_bits = c.pool.k_pool.view(torch.int16).numpy()
    blk_bits = c.k_blk.view(torch.int16).numpy()
    start = np.array(c.prefix_len)
    new = oracle.commit(pool_bits, c.pool.page_table, start, blk_bits, c.D, S)
    # independent: flatten (page, slot) and assign through torch indexing
    ref = torch.from_numpy(pool_bits.copy()).permute(0, 2, 1, 3).reshape(-1, 1, 64)
    p = torch.arange(c.D) + c.prefix_len[0]
    flat = c.pool.page_table[0, p // S].long() * S + p % S
    ref[flat] = torch.from_numpy(blk_bits[0])
    ref = ref.reshape(8, S, 1, 64).permute(0, 2, 1, 3).numpy()
    assert np.array_equal(new, ref)
    # the commit lands in the 4th logical page; every other slot keeps its bits
    page4 = int(c.pool.page_table[0, 3])
    changed = np.any(new != pool_bits, axis=(1, 2, 3))
    assert changed.nonzero()[0].tolist() == [page4]


def test_bf16_round_matches_torch():
    x = _rand((1000,), 40).float().numpy().astype(np.float64) * 7.0
    got = oracle.bf16_round(x)
    ref = torch.from_numpy(x).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref)
