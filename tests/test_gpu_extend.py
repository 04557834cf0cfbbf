"""GPU parity of bca_extend (short causal extend over the paged cache) against
the fp64 oracle, and its commit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_cases import DecodeRun, assert_close

pytestmark = pytest.mark.gpu


def _ref(case, seqs=None):
    return oracle.extend(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix, seqs=seqs)


@pytest.mark.parametrize("n", [1, 3, 5, 9])
def test_short_extend_ragged_prefixes(cuda_lib, n):
    """2N-1 <= 9 new tokens after prefixes of any length (none a multiple of
    the extend), including an empty one and ragged last tiles."""
    P = [0, 1, 37, 128, 129, 300, 1001, 2047]
    case = workloads.make_decode_case(P, D=n, Hq=32, Hkv=8, d=128, seed=n)
    r = DecodeRun(case)
    out = r.run(extend=True)
    assert r.status() == 0
    assert_close(out, _ref(case), what=f"extend n={n}")


def test_extend_head_dim_64_and_group_2(cuda_lib):
    case = workloads.make_decode_case([5, 64, 333, 700], D=7, Hq=8, Hkv=4, d=64, seed=3)
    r = DecodeRun(case)
    assert_close(r.run(extend=True), _ref(case), what="extend d=64")


@pytest.mark.parametrize("n", [64, 200])
def test_long_extend_spans_row_blocks_and_tiles(cuda_lib, n):
    """Extends longer than one M-tile of tokens (32 at 32/8 heads) and than
    one key tile: several row blocks, causal partial tiles inside the block."""
    case = workloads.make_decode_case([77, 512, 1500], D=n, Hq=32, Hkv=8, d=128, seed=n)
    r = DecodeRun(case)
    assert_close(r.run(extend=True), _ref(case), what=f"extend n={n}")


def test_one_token_extend_equals_one_token_decode(cuda_lib):
    """With one new token the causal rule and the block rule coincide: the
    two entry points give the same bits."""
    case = workloads.make_decode_case([3, 64, 999, 4096], D=1, Hq=32, Hkv=8, d=128, seed=5)
    r = DecodeRun(case)
    a = r.run(extend=True).clone()
    b = r.run(extend=False).clone()
    assert torch.equal(a, b)


def test_serving_extend_b64_n9(cuda_lib):
    """Batch 64, 9 new tokens (N = 5), prefixes log-uniform in [128, 32768]
    at token granularity: the bench workload; every sequence against the
    oracle, every row."""
    P = workloads.prefix_loguniform_blocks(64, 128, 32768, 1, seed=0)
    case = workloads.make_decode_case(P, D=9, Hq=32, Hkv=8, d=128, seed=0)
    r = DecodeRun(case)
    out = r.run(extend=True)
    assert r.status() == 0
    ref = _ref(case)
    for b in range(len(P)):
        assert_close(out[b], ref[b], what=f"serving extend seq {b} P={P[b]}")


def test_extend_commit_writes_unaligned_slots(cuda_lib):
    """commit = 1 copies the new rows into positions P_b .. P_b+n-1, which
    here start mid-page and cross page boundaries."""
    P = [5, 14, 31, 100]
    n = 9
    case = workloads.make_decode_case(P, D=n, Hq=8, Hkv=2, d=64, seed=7)
    r = DecodeRun(case)
    out = r.run(commit=True, extend=True)
    assert r.status() == 0
    assert_close(out, _ref(case), what="extend with commit")
    S = case.pool.page_size
    for name, pool, blk in (("k", r.k_pool, case.k_blk), ("v", r.v_pool, case.v_blk)):
        src = (case.pool.k_pool if name == "k" else case.pool.v_pool).view(torch.int16).numpy()
        want = oracle.commit(src, case.pool.page_table, case.prefix_len,
                             blk.view(torch.int16).numpy(), n, S)
        assert np.array_equal(pool.cpu().view(torch.int16).numpy(), want), name


def test_extend_bad_prefix_is_reported(cuda_lib):
    import block_causal_paged_gb300 as bca
    case = workloads.make_decode_case([10, 20], D=3, Hq=8, Hkv=2, d=64, seed=8)
    r = DecodeRun(case)
    r.prefix_len[1] = -4
    r.run(extend=True)
    assert r.status() == bca.ERR_DEVICE_BAD_LENGTH
