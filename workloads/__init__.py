"""Seeded synthetic inputs for block-causal paged attention.

Used by both the tests (which hand the same tensors to the CUDA path and to
the fp64 oracle) and ``bench.py``.  This module holds no attention, mask or
commit arithmetic: it draws random numbers and lays them out in the storage
formats the library takes (token-major Q/K/V, a paged K/V pool with a page
table, an arena with stored positions).

Shapes follow the workloads the pages describe: 64-token diffusion blocks
written block by block into a cache with pages of 16 tokens ("Inference for
Interpretable Text-Diffusion Models", "Block-Causal Paged Attention"),
256-token canvases after a 1024-token prompt with a shrinking set of live rows
and an arena of promoted rows ("Inference: Fewer, smaller forwards",
"Advancement 1", "Advancement 9", "Advancement 11"), and generations up to
32768 tokens at concurrency up to 64.  Values are N(0, 1) rounded to bf16.

Every sequence draws from its own generator (seeded from the workload seed
and the sequence index), so any subset of sequences can be regenerated
bit-identically on its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN_BITS = 0x7FC0        # quiet NaN in bf16: fills pool slots nobody owns
BF16_CANARY_BITS = 0x3F81     # 1.0078125: a finite marker for commit tests


def _gen(seed: int, *tags: int) -> torch.Generator:
    h = (seed & 0xFFFFFFFF) * 1000003
    for t in tags:
        h = (h * 7919 + (t & 0xFFFFFFFF) + 17) % (1 << 62)
    g = torch.Generator()
    g.manual_seed(h)
    return g


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def fill_bits(shape, bits: int) -> torch.Tensor:
    signed = bits if bits < 0x8000 else bits - 0x10000
    return torch.full(shape, signed, dtype=torch.int16).view(torch.bfloat16)


# ---------------------------------------------------------------------------
# Prefix-length distributions
# ---------------------------------------------------------------------------

def prefix_uniform_blocks(B: int, lo: int, hi: int, step: int, seed: int) -> list[int]:
    """Uniform over {lo, lo+step, ..., hi}."""
    g = _gen(seed, 101)
    n = (hi - lo) // step + 1
    idx = torch.randint(0, n, (B,), generator=g)
    return [lo + step * int(i) for i in idx]


def prefix_loguniform_blocks(B: int, lo: int, hi: int, step: int, seed: int) -> list[int]:
    """step * round(exp(U[ln lo, ln hi]) / step), clamped to [lo, hi]."""
    g = _gen(seed, 102)
    u = torch.rand((B,), generator=g, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    out = []
    for val in x.tolist():
        p = step * int(round(val / step))
        out.append(min(max(p, lo), hi))
    return out


# ---------------------------------------------------------------------------
# Paged pool construction
# ---------------------------------------------------------------------------

@dataclass
class PagedPool:
    k_pool: torch.Tensor          # [num_pages, Hkv, page_size, d] bf16
    v_pool: torch.Tensor
    page_table: torch.Tensor      # int32 [B, max_pages_per_seq], unused entries -1
    num_pages: int
    max_pages_per_seq: int
    page_size: int


def build_paged_pool(capacity: list[int], Hkv: int, d: int, page_size: int, seed: int,
                     pool_factor: float = 2.0, num_pages: int | None = None,
                     fill_bits_value: int | None = BF16_NAN_BITS) -> PagedPool:
    """Pool with room for ``capacity[b]`` tokens per sequence, pages in random order.

    Physical page ids come from one seeded random permutation of the pool;
    sequence b takes the next ceil(capacity[b] / page_size) ids from it.
    Slots are filled with ``fill_bits_value`` (NaN by default, so that a read
    of a slot the caller never wrote shows up in the output), or N(0,1) if None.
    """
    need = [-(-c // page_size) for c in capacity]
    total = sum(need)
    if num_pages is None:
        num_pages = max(total, int(math.ceil(pool_factor * total)))
    if num_pages < total:
        raise ValueError("pool too small")
    g = _gen(seed, 201)
    perm = torch.randperm(num_pages, generator=g)
    max_pp = max(need) if need else 1
    pt = torch.full((len(capacity), max(max_pp, 1)), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    shape = (num_pages, Hkv, page_size, d)
    if fill_bits_value is None:
        k_pool = randn_bf16(shape, _gen(seed, 202))
        v_pool = randn_bf16(shape, _gen(seed, 203))
    else:
        k_pool = fill_bits(shape, fill_bits_value)
        v_pool = fill_bits(shape, fill_bits_value)
    return PagedPool(k_pool, v_pool, pt, num_pages, max(max_pp, 1), page_size)


def write_logical_into_pool(pool: PagedPool, b: int, k_log: torch.Tensor, v_log: torch.Tensor,
                            start: int = 0) -> None:
    """Lay logical rows [n, Hkv, d] of sequence b at positions start.. into the pool.

    Input preparation only (the caller of the library owns this layout); it
    is the storage convention, position p -> (page_table[b][p // S], p % S).
    """
    S = pool.page_size
    n = k_log.shape[0]
    if n == 0:
        return
    if start % S == 0 and n % S == 0:
        # whole pages: one indexed assignment
        pages = pool.page_table[b, start // S:(start + n) // S].long()
        shape = (n // S, S) + tuple(k_log.shape[1:])
        pool.k_pool[pages] = k_log.reshape(shape).transpose(1, 2)
        pool.v_pool[pages] = v_log.reshape(shape).transpose(1, 2)
        return
    for p0 in range(start - start % S, start + n, S):
        page = int(pool.page_table[b, p0 // S])
        lo, hi = max(p0, start), min(p0 + S, start + n)
        pool.k_pool[page, :, lo - p0:hi - p0, :] = k_log[lo - start:hi - start].transpose(0, 1)
        pool.v_pool[page, :, lo - p0:hi - p0, :] = v_log[lo - start:hi - start].transpose(0, 1)


# ---------------------------------------------------------------------------
# Decode step (one diffusion block per sequence, optionally commit)
# ---------------------------------------------------------------------------

@dataclass
class DecodeCase:
    B: int
    D: int
    Hq: int
    Hkv: int
    d: int
    prefix_len: list[int]
    q: torch.Tensor               # [B, D, Hq, d]
    k_blk: torch.Tensor           # [B, D, Hkv, d]
    v_blk: torch.Tensor
    k_prefix: list                # per b: [P_b, Hkv, d] logical prefix keys
    v_prefix: list
    pool: PagedPool
    seed: int
    meta: dict = field(default_factory=dict)


def sequence_prefix_kv(seed: int, b: int, P: int, Hkv: int, d: int):
    return (randn_bf16((P, Hkv, d), _gen(seed, 301, b)),
            randn_bf16((P, Hkv, d), _gen(seed, 302, b)))


def sequence_block(seed: int, b: int, D: int, Hq: int, Hkv: int, d: int):
    return (randn_bf16((D, Hq, d), _gen(seed, 311, b)),
            randn_bf16((D, Hkv, d), _gen(seed, 312, b)),
            randn_bf16((D, Hkv, d), _gen(seed, 313, b)))


def make_decode_case(prefix_len: list[int], D: int, Hq: int, Hkv: int, d: int,
                     page_size: int = 16, seed: int = 0, pool_factor: float = 2.0,
                     num_pages: int | None = None,
                     fill_bits_value: int | None = BF16_NAN_BITS,
                     keep_logical: bool = True) -> DecodeCase:
    B = len(prefix_len)
    cap = [P + D for P in prefix_len]          # room to commit the block
    pool = build_paged_pool(cap, Hkv, d, page_size, seed, pool_factor, num_pages,
                            fill_bits_value)
    q = torch.empty((B, D, Hq, d), dtype=torch.bfloat16)
    k_blk = torch.empty((B, D, Hkv, d), dtype=torch.bfloat16)
    v_blk = torch.empty((B, D, Hkv, d), dtype=torch.bfloat16)
    kp, vp = [], []
    for b, P in enumerate(prefix_len):
        qb, kb, vb = sequence_block(seed, b, D, Hq, Hkv, d)
        q[b], k_blk[b], v_blk[b] = qb, kb, vb
        k_log, v_log = sequence_prefix_kv(seed, b, P, Hkv, d)
        write_logical_into_pool(pool, b, k_log, v_log)
        if keep_logical:
            kp.append(k_log)
            vp.append(v_log)
    return DecodeCase(B, D, Hq, Hkv, d, list(prefix_len), q, k_blk, v_blk, kp, vp, pool, seed)


# ---------------------------------------------------------------------------
# Prefill (packed sequences, block-causal over the whole prompt)
# ---------------------------------------------------------------------------

@dataclass
class PrefillCase:
    seq_lens: list[int]
    D: int
    Hq: int
    Hkv: int
    d: int
    q: torch.Tensor               # [T_total, Hq, d]
    k: torch.Tensor               # [T_total, Hkv, d]
    v: torch.Tensor
    cu_seqlens: torch.Tensor      # int32 [B+1]
    pool: PagedPool
    seed: int


def make_prefill_case(seq_lens: list[int], D: int, Hq: int, Hkv: int, d: int,
                      page_size: int = 16, seed: int = 0, pool_factor: float = 2.0,
                      fill_bits_value: int | None = BF16_NAN_BITS) -> PrefillCase:
    B = len(seq_lens)
    T = sum(seq_lens)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int32), 0)
    q = torch.empty((T, Hq, d), dtype=torch.bfloat16)
    k = torch.empty((T, Hkv, d), dtype=torch.bfloat16)
    v = torch.empty((T, Hkv, d), dtype=torch.bfloat16)
    for b, L in enumerate(seq_lens):
        s = int(cu[b])
        q[s:s + L] = randn_bf16((L, Hq, d), _gen(seed, 401, b))
        k[s:s + L] = randn_bf16((L, Hkv, d), _gen(seed, 402, b))
        v[s:s + L] = randn_bf16((L, Hkv, d), _gen(seed, 403, b))
    pool = build_paged_pool(list(seq_lens), Hkv, d, page_size, seed, pool_factor, None,
                            fill_bits_value)
    return PrefillCase(list(seq_lens), D, Hq, Hkv, d, q, k, v, cu, pool, seed)


# ---------------------------------------------------------------------------
# Multi-canvas shrinking window with an arena of promoted rows
# ---------------------------------------------------------------------------

@dataclass
class MulticanvasCase:
    B: int
    prompt_len: int
    n_canvas: int
    canvas_len: int
    Hq: int
    Hkv: int
    d: int
    q_live: torch.Tensor          # [B, max_live, Hq, d]
    k_live: torch.Tensor          # [B, max_live, Hkv, d]
    v_live: torch.Tensor
    live_pos: torch.Tensor        # int32 [B, max_live] absolute positions
    live_count: torch.Tensor      # int32 [B]
    pool: PagedPool               # the arena, as pages
    kv_pos: torch.Tensor          # int32 [num_pages, page_size], -1 where empty
    arena_len: torch.Tensor       # int32 [B]
    arena_k: list                 # per b: [arena_len, Hkv, d] entries in storage order
    arena_v: list
    arena_pos: list               # per b: int64 [arena_len]
    commit_rows: torch.Tensor     # int32 [B, max_commit] indices into the live rows
    commit_count: torch.Tensor    # int32 [B]
    seed: int


def make_multicanvas_case(B: int, prompt_len: int, n_canvas: int, canvas_len: int,
                          Hq: int, Hkv: int, d: int, active_lo: float = 0.3,
                          active_hi: float = 1.0, commit_frac: float = 0.25,
                          page_size: int = 16, seed: int = 0, pool_factor: float = 1.0,
                          shuffle_live: bool = False,
                          fill_bits_value: int | None = BF16_NAN_BITS) -> MulticanvasCase:
    """Arena = the prompt in order, then the already promoted rows of every
    canvas in a seeded random order, each with its absolute position; live rows
    = the still active rows of each canvas (a fraction U[active_lo, active_hi]),
    listed in ascending position (or shuffled).  Every position below the end
    of the last canvas is stored exactly once, in the arena or as a live row.
    ``commit_rows`` = a seeded ``commit_frac`` of each canvas's live rows (at
    least one), to be appended to the arena after the step.
    """
    total = prompt_len + n_canvas * canvas_len
    cap = [total] * B
    pool = build_paged_pool(cap, Hkv, d, page_size, seed, pool_factor, None, fill_bits_value)
    kv_pos = torch.full((pool.num_pages, page_size), -1, dtype=torch.int32)
    lives, arenas, commits = [], [], []
    for b in range(B):
        g = _gen(seed, 501, b)
        live, promoted, com = [], [], []
        for c in range(n_canvas):
            base = prompt_len + c * canvas_len
            frac = active_lo + (active_hi - active_lo) * float(torch.rand((), generator=g))
            n_act = max(1, int(round(frac * canvas_len)))
            perm = torch.randperm(canvas_len, generator=g)
            act = sorted(int(x) + base for x in perm[:n_act])
            prom = [int(x) + base for x in perm[n_act:]]
            first = len(live)              # live index of this canvas's first row
            live.extend(act)
            promoted.extend(prom)
            n_com = max(1, int(round(commit_frac * n_act)))
            pick = torch.randperm(n_act, generator=g)[:n_com]
            com.extend(first + i for i in sorted(int(x) for x in pick))
        order = torch.randperm(len(promoted), generator=g)
        promoted = [promoted[int(i)] for i in order]
        if shuffle_live:
            lperm = torch.randperm(len(live), generator=g)
            inv = {int(old): new for new, old in enumerate(lperm)}
            live = [live[int(i)] for i in lperm]
            com = sorted(inv[i] for i in com)
        lives.append(live)
        arenas.append(list(range(prompt_len)) + promoted)
        commits.append(com)
    max_live = max(len(x) for x in lives)
    max_commit = max(len(x) for x in commits)
    q_live = torch.zeros((B, max_live, Hq, d), dtype=torch.bfloat16)
    k_live = torch.zeros((B, max_live, Hkv, d), dtype=torch.bfloat16)
    v_live = torch.zeros((B, max_live, Hkv, d), dtype=torch.bfloat16)
    live_pos = torch.full((B, max_live), -1, dtype=torch.int32)
    live_count = torch.zeros(B, dtype=torch.int32)
    arena_len = torch.zeros(B, dtype=torch.int32)
    commit_rows = torch.full((B, max_commit), -1, dtype=torch.int32)
    commit_count = torch.zeros(B, dtype=torch.int32)
    ak, av, ap = [], [], []
    for b in range(B):
        # one K/V vector per absolute position, shared by arena and live rows
        k_all = randn_bf16((total, Hkv, d), _gen(seed, 511, b))
        v_all = randn_bf16((total, Hkv, d), _gen(seed, 512, b))
        q_all = randn_bf16((total, Hq, d), _gen(seed, 513, b))
        live = torch.tensor(lives[b], dtype=torch.long)
        n = live.numel()
        q_live[b, :n] = q_all[live]
        k_live[b, :n] = k_all[live]
        v_live[b, :n] = v_all[live]
        live_pos[b, :n] = live.to(torch.int32)
        live_count[b] = n
        arena = torch.tensor(arenas[b], dtype=torch.long)
        ka, va = k_all[arena], v_all[arena]
        write_logical_into_pool(pool, b, ka, va)
        S = page_size
        for idx, p in enumerate(arenas[b]):
            kv_pos[int(pool.page_table[b, idx // S]), idx % S] = p
        arena_len[b] = arena.numel()
        ak.append(ka)
        av.append(va)
        ap.append(arena.clone())
        commit_rows[b, :len(commits[b])] = torch.tensor(commits[b], dtype=torch.int32)
        commit_count[b] = len(commits[b])
    return MulticanvasCase(B, prompt_len, n_canvas, canvas_len, Hq, Hkv, d, q_live, k_live,
                           v_live, live_pos, live_count, pool, kv_pos, arena_len, ak, av, ap,
                           commit_rows, commit_count, seed)


# ---------------------------------------------------------------------------
# The named workloads
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = 0, **kw) -> DecodeCase:
    """1 sequence, 2 q heads / 1 kv head, d=64, 16-token block after a
    48-token prefix (3 pages) in a pool of 8 pages in random order."""
    return make_decode_case([48], D=16, Hq=2, Hkv=1, d=64, page_size=16, seed=seed,
                            num_pages=8, **kw)


def block_decode(seed: int = 0, **kw) -> DecodeCase:
    """Batch 8, 32/8 heads, d=128, 64-token block, prefix uniform in
    {512, 576, ..., 4096}, pool of 2x need."""
    P = prefix_uniform_blocks(8, 512, 4096, 64, seed)
    return make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, page_size=16, seed=seed, **kw)


def serving_decode(seed: int = 0, D: int = 64, B: int = 64, **kw) -> DecodeCase:
    """Batch 64, 32/8 heads, d=128, prefix log-uniform in [128, 32768]
    rounded to 64-token blocks, block D in {32, 64}, pool of 2x need."""
    P = prefix_loguniform_blocks(B, 128, 32768, 64, seed)
    return make_decode_case(P, D=D, Hq=32, Hkv=8, d=128, page_size=16, seed=seed, **kw)


def prefill_4x8192(seed: int = 0, **kw) -> PrefillCase:
    return make_prefill_case([8192] * 4, D=64, Hq=32, Hkv=8, d=128, page_size=16, seed=seed,
                             **kw)


def multicanvas_b16(seed: int = 0, **kw) -> MulticanvasCase:
    return make_multicanvas_case(16, 1024, 3, 256, Hq=32, Hkv=8, d=128, seed=seed, **kw)


def confidence_logits(rows: int, vocab: int, seed: int = 0, dtype=None, device="cpu"):
    """Synthetic language-model logits [rows, vocab] for the confidence pass:
    N(0, 3) scores, and in every fourth row one token lifted by 6 to 14 (a
    confident position), so both flat and peaked distributions occur.
    Generated in fp32 from `seed` on `device` (a CPU draw and a device draw
    of the same seed differ), then cast (bf16 by default)."""
    import torch
    if dtype is None:
        dtype = torch.bfloat16
    g = torch.Generator(device=device).manual_seed(int(seed) * 7919 + 17)
    x = torch.randn((rows, vocab), generator=g, device=device) * 3.0
    if rows and vocab:
        peaked = torch.arange(0, rows, 4, device=device)
        tok = torch.randint(0, vocab, (len(peaked),), generator=g, device=device)
        lift = 6.0 + 8.0 * torch.rand((len(peaked),), generator=g, device=device)
        x[peaked, tok] += lift
    return x.to(dtype)


# ---------------------------------------------------------------------------
# QKV-post (the step between the QKV projection and attention)
# ---------------------------------------------------------------------------

@dataclass
class QkvPostCase:
    B: int
    n: int
    Hq: int
    Hkv: int
    d: int
    qkv: torch.Tensor             # [B, n, Hq + 2 Hkv, d] bf16
    positions: torch.Tensor       # int32 [B, n]
    q_norm_w: torch.Tensor        # bf16 [d]
    k_norm_w: torch.Tensor
    write_pos: torch.Tensor       # int32 [B, n]: cache position of each token
    pool: PagedPool
    seed: int


def make_qkv_post_case(B: int, n: int, Hq: int, Hkv: int, d: int, prefix_len=None,
                       page_size: int = 16, seed: int = 0, qkv_scale: float = 2.0,
                       pos_max: int = 32768) -> QkvPostCase:
    """Projection rows N(0, qkv_scale^2) in bf16, norm weights 1 + N(0, 0.1^2)
    (learned weights near one), and positions: the block after each prefix
    (P_b .. P_b+n-1, also the cache positions) when ``prefix_len`` is given,
    else distinct random positions below ``pos_max`` written to the first n
    cache slots (an arena)."""
    g = _gen(seed, 401)
    qkv = (torch.randn((B, n, Hq + 2 * Hkv, d), generator=g) * qkv_scale).to(torch.bfloat16)
    q_norm_w = (1.0 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    k_norm_w = (1.0 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    if prefix_len is not None:
        P = torch.tensor(prefix_len, dtype=torch.int64)
        positions = (P[:, None] + torch.arange(n)[None, :]).to(torch.int32)
        write_pos = positions.clone()
        cap = [int(p) + n for p in prefix_len]
    else:
        positions = torch.stack([torch.randperm(pos_max, generator=g)[:n] for _ in range(B)])
        positions = positions.to(torch.int32)
        write_pos = torch.arange(n, dtype=torch.int32)[None, :].repeat(B, 1)
        cap = [n] * B
    pool = build_paged_pool(cap, Hkv, d, page_size, seed, fill_bits_value=None)
    return QkvPostCase(B, n, Hq, Hkv, d, qkv, positions, q_norm_w, k_norm_w, write_pos, pool, seed)
