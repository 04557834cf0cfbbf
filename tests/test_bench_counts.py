"""The algorithmic work that bench.py's roofline divides by, counted
independently: flops from the (query, key) pairs the oracle's block rule
makes visible, bytes from the sizes of a generated step's tensors."""
import math

import numpy as np
import pytest

import bench
import oracle
import workloads

CASES = [
    ([48, 0, 160], 16, 4, 2, 8, 16),
    ([64, 640, 128], 64, 32, 8, 128, 16),
    ([96, 32], 32, 6, 3, 64, 32),
]


@pytest.mark.parametrize("P,D,Hq,Hkv,d,S", CASES)
def test_decode_flops_are_the_visible_pairs(P, D, Hq, Hkv, d, S):
    """4 d flops per visible (query, key) pair and query head: Q K^T and P V,
    a multiply and an add each per element of d."""
    pairs = 0
    for Pb in P:
        pos = np.arange(Pb + D)
        pairs += int(oracle.block_causal_mask(pos[Pb:], pos, Pb, D).sum())
    assert bench.algorithmic(P, D, Hq, Hkv, d, S)["flops"] == 4 * d * Hq * pairs


@pytest.mark.parametrize("P,D,Hq,Hkv,d,S", CASES)
def test_decode_bytes_are_the_tensor_sizes(P, D, Hq, Hkv, d, S):
    """Every input once (the prefix K/V a sequence attends, Q, the block's
    K/V, the page-table entries it uses, its prefix length), the output; the
    step adds the commit's page writes."""
    c = workloads.make_decode_case(P, D=D, Hq=Hq, Hkv=Hkv, d=d, page_size=S, seed=0)
    nbytes = lambda t: t.numel() * t.element_size()
    prefix = sum(nbytes(k) + nbytes(v) for k, v in zip(c.k_prefix, c.v_prefix))
    blk = nbytes(c.k_blk) + nbytes(c.v_blk)
    pages = 4 * sum(math.ceil(Pb / S) for Pb in P)
    lens = 4 * len(P)
    attn = prefix + nbytes(c.q) + blk + nbytes(c.q) + pages + lens  # output shaped as q
    alg = bench.algorithmic(P, D, Hq, Hkv, d, S)
    assert alg["attn_bytes"] == attn
    assert alg["step_bytes"] == attn + blk
    assert alg["sum_prefix"] == sum(P)
