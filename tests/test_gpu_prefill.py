"""GPU parity of bca_prefill (block-causal attention + page write)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_cases import PrefillRun, assert_close

pytestmark = pytest.mark.gpu


def _ref(case, q_rows=None):
    return oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, case.D, q_rows=q_rows)


@pytest.mark.parametrize("lens,D,Hq,Hkv,d", [
    ([300, 512, 64, 1000], 64, 8, 2, 128),   # ragged lengths, partial diagonal tiles
    ([257, 128, 5], 16, 8, 2, 64),           # D = 16, head_dim 64, a 5-token prompt
    ([640, 130], 1, 4, 4, 128),              # block size 1 = causal attention, G = 1
    ([384], 384, 6, 2, 128),                 # one block = bidirectional, G = 3
    ([0, 200, 0, 64], 64, 8, 2, 128),        # zero-length sequences among others
])
def test_prefill_small(cuda_lib, lens, D, Hq, Hkv, d):
    case = workloads.make_prefill_case(lens, D=D, Hq=Hq, Hkv=Hkv, d=d, seed=21)
    r = PrefillRun(case)
    out = r.run()
    assert r.status() == 0
    assert_close(out, _ref(case), what=f"prefill {lens} D={D}")
    # the page write: every token at its logical position, bit-exact
    S = case.pool.page_size
    for name, pool_dev, pool_src, src in (("k", r.k_pool, case.pool.k_pool, case.k),
                                          ("v", r.v_pool, case.pool.v_pool, case.v)):
        want = pool_src.view(torch.int16).numpy().copy()
        cu = case.cu_seqlens.tolist()
        for b, L in enumerate(lens):
            blk = src[cu[b]:cu[b + 1]].view(torch.int16).numpy()[None]
            want = oracle.commit(want, case.pool.page_table[b:b + 1], [0], blk, L, S)
        assert np.array_equal(pool_dev.cpu().view(torch.int16).numpy(), want), name


def test_prefill_4x8192_sampled_rows_and_tile_counts(cuda_lib):
    """4 x 8192 tokens, D = 64, 32/8 heads: the whole prefill on the GPU, the
    oracle on sampled query rows (first block, middle, last block) of every
    sequence; the tile classifier's counts equal the dense-mask classes."""
    import block_causal_paged_gb300 as bca
    case = workloads.prefill_4x8192(seed=0)
    r = PrefillRun(case, write_pages=False)
    out = r.run()
    assert r.status() == 0
    rows = np.concatenate([np.arange(0, 64), np.arange(4000, 4064), np.arange(8128, 8192)])
    ref = _ref(case, q_rows={b: rows for b in range(4)})
    cu = case.cu_seqlens.tolist()
    for b in range(4):
        assert_close(out[cu[b] + rows], ref[cu[b] + rows], what=f"seq {b}")
    full, partial, skipped = bca.read_tile_counters(r.ws)
    pos = np.arange(8192)
    cls = oracle.tile_classes(pos, pos, 0, 64, 128, 128)  # 128-query x 128-key tiles
    per = 4 * 8 * 2                                        # sequences x kv heads x head pairs
    assert full == per * int((cls == "F").sum())
    assert partial == per * int((cls == "P").sum())
    assert skipped == per * int((cls == "S").sum())


def test_prefill_full_sequence_every_row(cuda_lib):
    """One whole 8192-token sequence of the 4 x 8192 workload (seed 1), every
    query row of every head against the oracle."""
    case = workloads.prefill_4x8192(seed=1)
    r = PrefillRun(case, write_pages=False)
    out = r.run()
    assert r.status() == 0
    b = 2
    ref = _ref(case, q_rows={b: np.arange(8192)})
    cu = case.cu_seqlens.tolist()
    assert_close(out[cu[b]:cu[b + 1]], ref[cu[b]:cu[b + 1]], what=f"seq {b}, all rows")


def test_appending_a_block_leaves_completed_blocks_unchanged(cuda_lib):
    """A completed block's outputs cannot change when later blocks are added
    ("Inference for Interpretable Text-Diffusion Models", "Background"): the
    prefill of T tokens and of the same tokens plus one more block of D give
    bit-identical rows for the first T tokens (the same tiles are computed
    for them; the added keys are never visible to them)."""
    D, T = 64, 1024
    big = workloads.make_prefill_case([T + D], D=D, Hq=16, Hkv=4, d=128, seed=41)
    small = workloads.make_prefill_case([T], D=D, Hq=16, Hkv=4, d=128, seed=41)
    small.q.copy_(big.q[:T])
    small.k.copy_(big.k[:T])
    small.v.copy_(big.v[:T])
    a = PrefillRun(small, write_pages=False).run().cpu()
    bb = PrefillRun(big, write_pages=False).run().cpu()
    assert torch.equal(a.view(torch.int16), bb[:T].view(torch.int16))
    assert_close(a, _ref(small), what="prefill of T tokens")


def test_prefill_within_block_permutation_equivariance(cuda_lib):
    """Permuting the tokens inside each block of a prompt (queries, keys and
    values together) permutes the prefill outputs the same way."""
    D, T = 64, 640
    case = workloads.make_prefill_case([T], D=D, Hq=8, Hkv=2, d=128, seed=43)
    base = PrefillRun(case, write_pages=False).run().cpu().clone()
    g = torch.Generator().manual_seed(43)
    perm = torch.cat([j * D + torch.randperm(D, generator=g) for j in range(T // D)])
    pc = workloads.make_prefill_case([T], D=D, Hq=8, Hkv=2, d=128, seed=43)
    pc.q.copy_(case.q[perm])
    pc.k.copy_(case.k[perm])
    pc.v.copy_(case.v[perm])
    got = PrefillRun(pc, write_pages=False).run().cpu()
    assert_close(got, base[perm].double().numpy(), what="permuted vs unpermuted")
    assert_close(got, _ref(pc), what="permuted vs oracle")


def test_decode_block_equals_prefill_rows(cuda_lib):
    """decode(block j | prefix) on the GPU equals the GPU prefill rows of block j
    within the tolerance (both against the same oracle values)."""
    from _gpu_cases import DecodeRun
    D, T = 64, 1024
    pc = workloads.make_prefill_case([T], D=D, Hq=8, Hkv=2, d=128, seed=31)
    pre = PrefillRun(pc).run().cpu()
    j = 9
    s = j * D
    dc = workloads.make_decode_case([s], D=D, Hq=8, Hkv=2, d=128, seed=31)
    dc.q[0] = pc.q[s:s + D]
    dc.k_blk[0] = pc.k[s:s + D]
    dc.v_blk[0] = pc.v[s:s + D]
    dc.k_prefix[0] = pc.k[:s]
    dc.v_prefix[0] = pc.v[:s]
    workloads.write_logical_into_pool(dc.pool, 0, pc.k[:s], pc.v[:s])
    dec = DecodeRun(dc).run().cpu()
    ref = oracle.decode(dc.q, dc.k_blk, dc.v_blk, dc.k_prefix, dc.v_prefix)
    assert_close(dec[0], ref[0], what="decode")
    assert_close(pre[s:s + D], ref[0], what="prefill rows")
