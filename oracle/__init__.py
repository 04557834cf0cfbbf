"""fp64 CPU oracle for block-causal paged attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``, never by the product package.
It shares no code with the CUDA path; the only thing both sides use is the
seeded input generator in ``workloads``, which holds none of the method's
arithmetic.

Each entry point below states the passage it follows.  Every one of them
reduces to the same definition (``attention``): softmax attention in double
precision under the block rule

    blk(p) = -1 if p < P0 else floor((p - P0) / D);   j visible to i  iff  blk(j) <= blk(i)

("Inference for Interpretable Text-Diffusion Models", "Background", first
bullet; "Inference: Fewer, smaller forwards", "Advancement 1" and
"Advancement 13").  Keys are given in *logical* order with explicit
positions; paging is a storage detail the oracle never sees.

``confidence`` (the top prediction of a position and its probability under
the softmax over the vocabulary) is the one entry point that is not an
attention.

Pins (tests/test_oracle_*.py) tie this code to things other than itself:
brute-force per-row enumeration, PyTorch SDPA in fp64 for the special cases
the pages reduce to (block size 1 = causal; one block = unmasked), closed
forms, the pages' worked examples (tests/golden/) and the invariants the
pages state.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Sequence

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64p = ctypes.POINTER(ctypes.c_int64)
        dp = ctypes.POINTER(ctypes.c_double)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_block_causal_mask.argtypes = [i64p, ctypes.c_int64, i64p, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, u8p]
        lib.oracle_block_causal_mask.restype = ctypes.c_int
        lib.oracle_masked_attention.argtypes = [dp, dp, dp, u8p, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_double, dp, dp, ctypes.c_int]
        lib.oracle_masked_attention.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(x) -> np.ndarray:
    """Exact conversion of a bf16/fp32 tensor (torch or numpy) to fp64."""
    if hasattr(x, "detach"):
        import torch  # only for tensors handed in by the caller
        return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ---------------------------------------------------------------------------
# The definition
# ---------------------------------------------------------------------------

def block_index(p, P0: int, D: int):
    """blk(p): -1 inside the completed prefix, else the diffusion block (canvas) number."""
    p = np.asarray(p, dtype=np.int64)
    return np.where(p < P0, -1, (p - P0) // D)


def block_causal_mask(q_pos, k_pos, P0: int, D: int) -> np.ndarray:
    """Dense [Tq, Tk] uint8 mask of the block rule (1 = the key is visible)."""
    qp, kp = _i64(q_pos), _i64(k_pos)
    mask = np.empty((qp.size, kp.size), dtype=np.uint8)
    rc = _lib().oracle_block_causal_mask(_ptr(qp, ctypes.c_int64), qp.size, _ptr(kp, ctypes.c_int64),
                                         kp.size, int(P0), int(D), _ptr(mask, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("oracle_block_causal_mask: bad arguments")
    return mask


def sliding_window_mask(q_pos, k_pos, window: int) -> np.ndarray:
    """Dense [Tq, Tk] uint8 band of a sliding-window layer (1 = kept).

    "Inference: Fewer, smaller forwards", "Advancement 11": arena entries keep
    their absolute positions, so sliding-window layers can band-mask the
    entries that fall outside the 1024-token window.  Reading: the window of a
    query at position q holds the `window` most recent positions up to q,
    i.e. a key at position k is kept iff q - k < window (keys after q, which
    only the query's own canvas holds, are kept).  window <= 0: no band.
    """
    qp, kp = _i64(q_pos), _i64(k_pos)
    if window <= 0:
        return np.ones((qp.size, kp.size), dtype=np.uint8)
    return (qp[:, None] - kp[None, :] < window).astype(np.uint8)


def attention(q, k, v, q_pos, k_pos, P0: int, D: int, scale: float | None = None,
              nthreads: int | None = None, return_lse: bool = False, mask=None):
    """Block-causal attention of one sequence in fp64.

    q [Tq, Hq, d], k/v [Tk, Hkv, d] (any float dtype, converted exactly);
    q_pos/k_pos absolute positions; query head h reads kv head h // (Hq // Hkv).
    ``scale`` defaults to 1/sqrt(d).  ``mask`` overrides the block rule with an
    explicit [Tq, Tk] 0/1 matrix (used only by tests of the mask itself).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    if scale is None or scale == 0.0:
        scale = 1.0 / math.sqrt(d)
    if mask is None:
        mask = block_causal_mask(q_pos, k_pos, P0, D)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    out = np.empty((Tq, Hq, d), dtype=np.float64)
    lse = np.empty((Tq, Hq), dtype=np.float64)
    rc = _lib().oracle_masked_attention(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        _ptr(mask, ctypes.c_uint8), Tq, Tk, Hq, Hkv, d, float(scale),
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_masked_attention failed ({rc})")
    return (out, lse) if return_lse else out


# ---------------------------------------------------------------------------
# Entry points of the path, each reduced to the definition
# ---------------------------------------------------------------------------

def decode(q, k_blk, v_blk, k_prefix: Sequence, v_prefix: Sequence, scale=None,
           nthreads=None, seqs: Sequence[int] | None = None):
    """One diffusion-block decode step for a batch.

    "Inference for Interpretable Text-Diffusion Models", "KV Cache", step 2:
    the active block is processed against the cache of completed blocks.
    q [B, D, Hq, d] are the block's queries at positions P_b .. P_b+D-1;
    the keys are the logical prefix 0 .. P_b-1 (k_prefix[b], [P_b, Hkv, d])
    followed by the block's own D keys (k_blk[b]).  P0 = P_b, so the prefix
    is fully visible and the block is visible to itself in both directions.
    Returns fp64 [B, D, Hq, d] (rows of sequences not in ``seqs`` are NaN).
    """
    q, k_blk, v_blk = _f64(q), _f64(k_blk), _f64(v_blk)
    B, D = q.shape[0], q.shape[1]
    out = np.full(q.shape, np.nan, dtype=np.float64)
    for b in (range(B) if seqs is None else seqs):
        kp, vp = _f64(k_prefix[b]), _f64(v_prefix[b])
        P = kp.shape[0]
        keys = np.concatenate([kp, k_blk[b]], axis=0)
        vals = np.concatenate([vp, v_blk[b]], axis=0)
        k_pos = np.arange(P + D, dtype=np.int64)
        q_pos = P + np.arange(D, dtype=np.int64)
        out[b] = attention(q[b], keys, vals, q_pos, k_pos, P0=P, D=D, scale=scale,
                           nthreads=nthreads)
    return out


def extend(q, k_new, v_new, k_prefix: Sequence, v_prefix: Sequence, scale=None,
           nthreads=None, seqs: Sequence[int] | None = None):
    """Short causal extend of a batch over its cached prefix.

    "Introspective Diffusion Language Model", "3.3 I-DLM Serving Stack" and
    Appendix D: each step appends a few causal query tokens (2N - 1 for
    fixed-query introspective decoding, at most 9 in the short-extend case)
    that attend the whole paged prefix and, among themselves, strictly
    causally.  q [B, n, Hq, d] are the new tokens at positions P_b .. P_b+n-1;
    keys are the logical prefix 0 .. P_b-1 (k_prefix[b]) followed by the n
    new keys (k_new[b]).  The causal rule is the block rule with blocks of
    one token (P0 = P_b, D = 1): key j is visible to query i iff j <= i.
    Unlike a diffusion block, P_b need not be a multiple of anything.
    Returns fp64 [B, n, Hq, d] (rows of sequences not in ``seqs`` are NaN).
    """
    q, k_new, v_new = _f64(q), _f64(k_new), _f64(v_new)
    B, n = q.shape[0], q.shape[1]
    out = np.full(q.shape, np.nan, dtype=np.float64)
    for b in (range(B) if seqs is None else seqs):
        kp, vp = _f64(k_prefix[b]), _f64(v_prefix[b])
        P = kp.shape[0]
        keys = np.concatenate([kp, k_new[b]], axis=0)
        vals = np.concatenate([vp, v_new[b]], axis=0)
        k_pos = np.arange(P + n, dtype=np.int64)
        q_pos = P + np.arange(n, dtype=np.int64)
        out[b] = attention(q[b], keys, vals, q_pos, k_pos, P0=P, D=1, scale=scale,
                           nthreads=nthreads)
    return out


def prefill(q, k, v, cu_seqlens, D: int, scale=None, nthreads=None,
            q_rows: dict | None = None):
    """Block-causal prefill of packed sequences.

    "Inference for Interpretable Text-Diffusion Models", "KV Cache", step 1 and
    the prefill BlockMask figure: every token of the prompt attends with the
    block rule, P0 = 0.  q [total_T, Hq, d], k/v [total_T, Hkv, d],
    cu_seqlens [B+1].  ``q_rows`` optionally maps a sequence index to the
    local query rows to evaluate (others are NaN); by default all rows.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = _i64(cu_seqlens)
    out = np.full(q.shape, np.nan, dtype=np.float64)
    for b in range(cu.size - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        T = e - s
        if q_rows is not None and b not in q_rows:
            continue
        rows = np.arange(T) if q_rows is None else np.asarray(q_rows[b], dtype=np.int64)
        if rows.size == 0:
            continue
        k_pos = np.arange(T, dtype=np.int64)
        res = attention(q[s + rows], k[s:e], v[s:e], rows, k_pos, P0=0, D=D, scale=scale,
                        nthreads=nthreads)
        out[s + rows] = res
    return out


def multicanvas(q_live, k_live, v_live, live_pos, live_count, k_arena: Sequence,
                v_arena: Sequence, arena_pos: Sequence, prompt_len: int, canvas_len: int,
                scale=None, nthreads=None, seqs: Sequence[int] | None = None, window: int = 0):
    """Multi-canvas shrinking-window attention.

    "Inference: Fewer, smaller forwards", "Advancement 1", "Advancement 9",
    "Advancement 11" and "Advancement 13": only the live rows of the active
    canvases are queries; a live row of canvas c sees every position below
    prompt_len + canvas_len * (c + 1), whether that position is stored in the
    arena (k_arena[b] with absolute positions arena_pos[b]) or is itself a
    live row.  P0 = prompt_len and D = canvas_len.
    q_live [B, max_live, Hq, d]; k_live/v_live [B, max_live, Hkv, d];
    live_pos [B, max_live]; live_count [B].  window > 0 adds the band of a
    sliding-window layer (``sliding_window_mask``) to the block rule.
    Returns fp64 [B, max_live, Hq, d]; rows past live_count are NaN.
    """
    q_live, k_live, v_live = _f64(q_live), _f64(k_live), _f64(v_live)
    live_pos, live_count = _i64(live_pos), _i64(live_count)
    out = np.full(q_live.shape, np.nan, dtype=np.float64)
    for b in (range(q_live.shape[0]) if seqs is None else seqs):
        n = int(live_count[b])
        if n == 0:
            continue
        ka, va, pa = _f64(k_arena[b]), _f64(v_arena[b]), _i64(arena_pos[b])
        keys = np.concatenate([ka, k_live[b, :n]], axis=0)
        vals = np.concatenate([va, v_live[b, :n]], axis=0)
        k_pos = np.concatenate([pa, live_pos[b, :n]])
        mask = None
        if window > 0:
            mask = (block_causal_mask(live_pos[b, :n], k_pos, prompt_len, canvas_len)
                    & sliding_window_mask(live_pos[b, :n], k_pos, window))
        out[b, :n] = attention(q_live[b, :n], keys, vals, live_pos[b, :n], k_pos,
                               P0=prompt_len, D=canvas_len, scale=scale, nthreads=nthreads,
                               mask=mask)
    return out


def commit(pool, page_table, start_pos, blk, num_tokens: int, page_size: int):
    """KV commit: a bit copy of a finished block into its pages.

    "Inference for Interpretable Text-Diffusion Models", "KV Cache", step 3
    (a final pass writes the completed block into the cache) and "Paged
    Attention" (logical position p of sequence b lives in page
    page_table[b][p // page_size], slot p % page_size).
    pool [num_pages, Hkv, page_size, d] and blk [B, >=num_tokens, Hkv, d] are
    raw 16-bit words (np.uint16 / any integer view); returns the new pool.
    """
    pool = np.array(pool, copy=True)
    pt = _i64(page_table)
    sp = _i64(start_pos)
    blk = np.asarray(blk)
    B = blk.shape[0]
    for b in range(B):
        for t in range(num_tokens):
            p = int(sp[b]) + t
            page = int(pt[b, p // page_size])
            slot = p % page_size
            pool[page, :, slot, :] = blk[b, t, :, :]
    return pool


def tile_classes(q_pos, k_pos, P0: int, D: int, tile_q: int, tile_k: int) -> np.ndarray:
    """Classify each (query tile, key tile) of the dense mask.

    "Inference for Interpretable Text-Diffusion Models", "FlexAttention with
    Aligned Tiles": a tile is fully included ('F'), fully excluded ('S') or
    partially included ('P').  Tiles are consecutive runs of tile_q queries
    and tile_k keys in the given order (the last ones may be short).
    """
    mask = block_causal_mask(q_pos, k_pos, P0, D)
    Tq, Tk = mask.shape
    nq, nk = -(-Tq // tile_q), -(-Tk // tile_k)
    out = np.empty((nq, nk), dtype="<U1")
    for a in range(nq):
        for c in range(nk):
            t = mask[a * tile_q:(a + 1) * tile_q, c * tile_k:(c + 1) * tile_k]
            out[a, c] = "F" if t.all() else ("S" if not t.any() else "P")
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even), returned as fp64.

    Used only to report how many output elements differ at the bit level;
    the acceptance tolerance is checked against the unrounded fp64 value.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)


def qkv_post(qkv, positions, Hq: int, Hkv: int, q_norm_w=None, k_norm_w=None,
             eps: float = 1e-6, rope_theta: float = 0.0):
    """The step between the QKV projection and attention, in fp64.

    "Inference: Fewer, smaller forwards", "Advancement 16" (an optional fused
    QKV-post: RoPE, norms and the arena write) and "Advancement 10" (RoPE is
    baked into keys at the token's true absolute position).  qkv
    [..., Hq + 2 Hkv, d]: the projection's output, query heads first, then
    key heads, then value heads; positions [...] the absolute positions.
    Norms: each query and key head vector x is RMS-normalised with a weight
    w of length d shared by the heads, x * w / sqrt(mean(x^2) + eps) (no
    norm where the weight is None).  RoPE (rope_theta > 0): the pair
    (x_i, x_{i+d/2}), i < d/2, is rotated by the angle pos * theta^(-2i/d).
    Values pass through.  Returns fp64 (q [..., Hq, d], k [..., Hkv, d],
    v [..., Hkv, d]); rounding to bf16 is the caller's (``bf16_round``).
    """
    x = _f64(qkv)
    d = x.shape[-1]
    q = x[..., :Hq, :].copy()
    k = x[..., Hq:Hq + Hkv, :].copy()
    v = x[..., Hq + Hkv:Hq + 2 * Hkv, :].copy()

    def rms(a, w):
        if w is None:
            return a
        w = _f64(w)
        return a * w / np.sqrt(np.mean(a * a, axis=-1, keepdims=True) + eps)

    q, k = rms(q, q_norm_w), rms(k, k_norm_w)
    if rope_theta > 0:
        half = d // 2
        inv_freq = rope_theta ** (-2.0 * np.arange(half, dtype=np.float64) / d)
        ang = _i64(positions).astype(np.float64)[..., None] * inv_freq  # [..., d/2]
        c, s = np.cos(ang)[..., None, :], np.sin(ang)[..., None, :]

        def rot(a):
            a1, a2 = a[..., :half], a[..., half:]
            return np.concatenate([a1 * c - a2 * s, a2 * c + a1 * s], axis=-1)

        q, k = rot(q), rot(k)
    return q, k, v


def confidence(logits):
    """Top prediction and its probability for each row of logits.

    "Inference: Fewer, smaller forwards", "Advancement 2: tau_conf": on every
    forward the model gives a distribution over the vocabulary at each
    uncommitted position (the softmax of its logits), and the confidence is
    the probability of the argmax, the top prediction; "Advancement 16" lists
    the fused softmax-plus-argmax over the vocabulary that computes it.

    logits [rows, vocab], any float dtype (read exactly as fp64).  Returns
    (argmax int64 [rows], confidence fp64 [rows]).  Among equal maxima the
    lowest index is the argmax.  Since the argmax holds the largest logit m,
    its probability is exp(0) / sum_v exp(l_v - m) = 1 / sum_v exp(l_v - m).
    A row whose logits are all -inf has no distribution: argmax 0,
    confidence 0.
    """
    x = np.asarray(logits, dtype=np.float64)
    if x.ndim != 2:
        raise ValueError("logits must be [rows, vocab]")
    rows = x.shape[0]
    arg = np.zeros(rows, dtype=np.int64)
    conf = np.zeros(rows, dtype=np.float64)
    for r in range(rows):
        m = x[r].max() if x.shape[1] else -math.inf
        if m == -math.inf:
            continue
        arg[r] = int(np.argmax(x[r]))  # first occurrence of the maximum
        conf[r] = 1.0 / np.exp(x[r] - m).sum()
    return arg, conf
