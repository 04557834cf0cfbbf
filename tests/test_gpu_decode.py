"""GPU parity of bca_decode (and its commit) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import block_causal_paged_gb300 as bca
import oracle
import workloads
from _gpu_cases import DecodeRun, assert_close

pytestmark = pytest.mark.gpu


def _ref(case, seqs=None):
    return oracle.decode(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix, seqs=seqs)


def test_tiny_decode_and_commit(cuda_lib):
    """One sequence, 2/1 heads, d=64, D=16 after 48 prefix tokens in a pool of
    8 shuffled pages; then the block is committed to the 4th logical page."""
    case = workloads.tiny_decode(seed=0)
    r = DecodeRun(case)
    out = r.run(commit=True)
    assert r.status() == 0
    assert_close(out, _ref(case), what="tiny")
    S = case.pool.page_size
    for name, pool, blk in (("k", r.k_pool, case.k_blk), ("v", r.v_pool, case.v_blk)):
        src = (case.pool.k_pool if name == "k" else case.pool.v_pool).view(torch.int16).numpy()
        want = oracle.commit(src, case.pool.page_table, case.prefix_len,
                             blk.view(torch.int16).numpy(), case.D, S)
        assert np.array_equal(pool.cpu().view(torch.int16).numpy(), want), name


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_decode_batch8(cuda_lib, seed):
    """Batch 8, 32/8 heads, d=128, D=64, prefix uniform in {512..4096}."""
    case = workloads.block_decode(seed=seed)
    r = DecodeRun(case)
    out = r.run(commit=False)
    assert r.status() == 0
    assert_close(out, _ref(case), what=f"block decode seed {seed}")


def test_page_permutation_is_bit_identical(cuda_lib):
    """Scrambling the physical page layout leaves the output bits unchanged."""
    P = [960, 2048, 64, 3072]
    a = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=7)
    b = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=7, pool_factor=3.0)
    assert not torch.equal(a.pool.page_table, b.pool.page_table)
    out_a = DecodeRun(a).run().cpu()
    out_b = DecodeRun(b).run().cpu()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


@pytest.mark.parametrize("P,D,Hq,Hkv,d", [
    ([0, 64, 640], 64, 8, 2, 128),        # empty prefix, one prefix tile
    ([37, 5, 1000], 1, 4, 1, 64),          # block size 1: ordinary causal decode
    ([17 * 3, 0, 17 * 40], 17, 6, 2, 128),  # ragged block (not a multiple of 16)
    ([200, 1000], 100, 4, 4, 64),           # G = 1, block of 100 over two M-tiles
    ([96, 2976], 96, 12, 4, 128),           # G = 3 (rows 126 of 128), 2 row blocks
    ([4096, 128], 32, 32, 8, 128),         # D = 32: one M-tile per KV head
])
def test_generic_shapes(cuda_lib, P, D, Hq, Hkv, d):
    case = workloads.make_decode_case(P, D=D, Hq=Hq, Hkv=Hkv, d=d, seed=11)
    r = DecodeRun(case)
    out = r.run()
    assert r.status() == 0
    assert_close(out, _ref(case), what=f"P={P} D={D} {Hq}/{Hkv} d={d}")


def test_block_size_one_is_causal_decode(cuda_lib):
    """D = 1 reduces to single-token causal decode: compare with SDPA on the GPU
    in fp32 as an independent second reference."""
    P = [31, 300]
    case = workloads.make_decode_case(P, D=1, Hq=8, Hkv=2, d=128, seed=3)
    out = DecodeRun(case).run().cpu().double()
    for b in range(2):
        k = torch.cat([case.k_prefix[b], case.k_blk[b]]).double()
        v = torch.cat([case.v_prefix[b], case.v_blk[b]]).double()
        q = case.q[b].double()
        kk = k.repeat_interleave(4, 1).transpose(0, 1)
        vv = v.repeat_interleave(4, 1).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(q.transpose(0, 1), kk, vv)
        err = (out[b] - ref.transpose(0, 1)).abs()
        assert err.max() < 2e-2 and err.mean() < 2e-3


def test_split_kv_matches_unsplit(cuda_lib):
    """The split-KV path (partials + combine) and a workspace too small to
    split give the same result within the tolerance."""
    P = [32768, 128, 9000 // 64 * 64]
    case = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=5)
    r = DecodeRun(case)
    ref = _ref(case)
    a = r.run().clone()
    assert_close(a, ref, what="split")
    import block_causal_paged_gb300 as bca
    n = bca.workspace_size(r.d, bca.OP_DECODE_MIN)   # no room for split-KV partials
    assert 0 < n < bca.workspace_size(r.d, bca.OP_DECODE)
    small = torch.empty(n, dtype=torch.uint8, device="cuda")
    bca.workspace_init(small)
    b = r.run(ws=small).clone()
    assert bca.read_device_status(small) == 0
    assert_close(b, ref, what="unsplit")


def test_batch96_planned_by_plan_kernel(cuda_lib):
    """Batches above 64 are planned by the separate plan kernel (smaller ones
    inside the attention kernel): same results, including split prefixes."""
    rng = np.random.default_rng(12)
    P = (rng.integers(0, 40, 96) * 64).tolist()
    P[5] = 24576                                    # one long prefix: split into chunks
    case = workloads.make_decode_case(P, D=64, Hq=16, Hkv=4, d=128, seed=12)
    r = DecodeRun(case)
    out = r.run(commit=True)
    assert r.status() == 0
    seqs = [0, 5, 37, 95]
    ref = _ref(case, seqs=seqs)
    for b in seqs:
        assert_close(out[b], ref[b], what=f"batch 96 seq {b}")
    S = case.pool.page_size
    src = case.pool.k_pool.view(torch.int16).numpy()
    want = oracle.commit(src, case.pool.page_table, case.prefix_len,
                         case.k_blk.view(torch.int16).numpy(), case.D, S)
    assert np.array_equal(r.k_pool.cpu().view(torch.int16).numpy(), want)


def test_serving_batch64_commit_bit_exact(cuda_lib):
    """The step with commit on, at the benchmarked size: every page of the pool
    equals the oracle's commit (blocks written at P .. P+D-1, everything else
    untouched), and the attention output is unaffected by the commit."""
    case = workloads.serving_decode(seed=3, D=64)
    r = DecodeRun(case)
    out = r.run(commit=True).clone()
    assert r.status() == 0
    S = case.pool.page_size
    for name, pool, blk in (("k", r.k_pool, case.k_blk), ("v", r.v_pool, case.v_blk)):
        src = (case.pool.k_pool if name == "k" else case.pool.v_pool).view(torch.int16).numpy()
        want = oracle.commit(src, case.pool.page_table, case.prefix_len,
                             blk.view(torch.int16).numpy(), case.D, S)
        assert np.array_equal(pool.cpu().view(torch.int16).numpy(), want), name
    # every sequence of the step, one comparison over the whole output
    assert_close(out, _ref(case), what="serving with commit, all 64 sequences")


@pytest.mark.parametrize("D", [64, 32])
def test_serving_batch64_every_sequence(cuda_lib, D):
    """Batch 64, prefix log-uniform in [128, 32768]: the full step on the GPU
    and the oracle on every one of the 64 sequences (the benchmarked step)."""
    case = workloads.serving_decode(seed=0, D=D)
    r = DecodeRun(case)
    out = r.run()
    assert r.status() == 0
    ref = _ref(case)
    P = np.array(case.prefix_len)
    for b in range(case.B):
        assert_close(out[b], ref[b], what=f"serving D={D} seq {b} P={P[b]}")
    assert_close(out, ref, what=f"serving D={D}, whole step")


def test_within_block_permutation_equivariance(cuda_lib):
    """Permuting the rows of a block (its queries and its own keys/values
    together) permutes the decode outputs the same way: there is no
    positional operation in the kernel, Q and K arrive rotated ("Inference:
    Fewer, smaller forwards", "Advancement 10").  Checked on the GPU against
    the unpermuted GPU result and against the oracle."""
    P = [0, 512, 1984, 4096, 64 * 33]
    case = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=17)
    base = DecodeRun(case).run().cpu().clone()
    g = torch.Generator().manual_seed(17)
    perm = torch.stack([torch.randperm(64, generator=g) for _ in P])
    pc = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=17)
    for b in range(len(P)):
        pc.q[b] = case.q[b][perm[b]]
        pc.k_blk[b] = case.k_blk[b][perm[b]]
        pc.v_blk[b] = case.v_blk[b][perm[b]]
    got = DecodeRun(pc).run().cpu()
    want = torch.stack([base[b][perm[b]] for b in range(len(P))])
    assert_close(got, want.double().numpy(), what="permuted vs unpermuted")
    assert_close(got, _ref(pc), what="permuted vs oracle")


def test_device_error_bad_page_is_reported(cuda_lib):
    import block_causal_paged_gb300 as bca
    case = workloads.make_decode_case([256, 512], D=64, Hq=8, Hkv=2, d=128, seed=2)
    r = DecodeRun(case)
    r.page_table[1, 3] = case.pool.num_pages + 5   # outside the pool
    r.run()
    assert r.status() == bca.ERR_DEVICE_PAGE_OOB
    assert torch.isfinite(r.out.float()).all()


def test_device_error_bad_prefix_is_reported(cuda_lib):
    import block_causal_paged_gb300 as bca
    case = workloads.make_decode_case([256, 512], D=64, Hq=8, Hkv=2, d=128, seed=2)
    r = DecodeRun(case)
    r.prefix_len[0] = 100                           # not a multiple of D
    r.run()
    assert r.status() == bca.ERR_DEVICE_BAD_LENGTH


def test_tile_counters_decode(cuda_lib):
    import block_causal_paged_gb300 as bca
    case = workloads.make_decode_case([640, 64, 0], D=64, Hq=32, Hkv=8, d=128, seed=1)
    r = DecodeRun(case)
    r.run()
    full, partial, skipped = bca.read_tile_counters(r.ws)
    # tiles of 128 keys per KV head: 640 prefix keys = 5 full tiles; 64 prefix
    # keys = 1 tile with 64 valid keys; each 64-key own block = 1 tile with 64
    # valid keys (masked past the end); nothing is skipped in a decode step
    assert (full, partial, skipped) == (8 * 5, 8 * (1 + 1 + 1 + 1), 0)


def test_decode_on_every_visible_device(cuda_lib):
    """One process, one decode step on each visible device (the kernels'
    launch settings are per device)."""
    n = torch.cuda.device_count()
    if n < 2:
        pytest.skip("one device visible")
    case = workloads.make_decode_case([256, 1024, 4096], D=64, Hq=8, Hkv=2, d=128, seed=23)
    ref = _ref(case)
    for dev in range(n):
        with torch.cuda.device(dev):
            r = DecodeRun(case, dev=f"cuda:{dev}")
            out = r.run()
            assert r.status() == 0
            assert_close(out, ref, what=f"device {dev}")


def test_debug_checks_on_device_tables(cuda_lib, monkeypatch):
    """BCA_DEBUG=1 with device-resident lengths and page table: a valid
    decode runs and matches the oracle; a used page-table entry outside the
    pool is refused on the host before any launch (the output buffer keeps
    its contents), where without the switch the device would skip it."""
    monkeypatch.setenv("BCA_DEBUG", "1")
    case = workloads.make_decode_case([128, 4096, 64 * 7], D=64, Hq=8, Hkv=2, d=128, seed=12)
    r = DecodeRun(case)
    out = r.run(commit=True).clone()
    assert r.status() == 0
    assert_close(out, _ref(case), what="decode under BCA_DEBUG=1")
    r.out.fill_(7.0)
    r.page_table[1, 5] = case.pool.num_pages
    with pytest.raises(bca.BcaError) as e:
        r.run()
    assert e.value.code == bca.ERR_PAGE_RANGE
    assert bool((r.out == 7.0).all())
