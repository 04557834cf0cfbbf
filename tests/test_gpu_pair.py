"""The CTA-pair attention kernel (decode blocks of >= 2 M-tiles, prefill;
head_dim 128) against the fp64 oracle and against the single-CTA kernel on
the same inputs (BCA_PAIR_KERNEL=0 routes every shape to the latter)."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_cases import DecodeRun, PrefillRun, assert_close

pytestmark = pytest.mark.gpu


class single_cta_kernel:
    """Context manager: run the library with the pair kernel disabled."""

    def __enter__(self):
        self.old = os.environ.get("BCA_PAIR_KERNEL")
        os.environ["BCA_PAIR_KERNEL"] = "0"

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop("BCA_PAIR_KERNEL", None)
        else:
            os.environ["BCA_PAIR_KERNEL"] = self.old


def _decode_ref(case, seqs=None):
    return oracle.decode(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix, seqs=seqs)


@pytest.mark.parametrize("P,D,Hq,Hkv", [
    ([128, 512], 64, 32, 8),                  # the serving shape, two short prefixes
    ([0, 64, 4096, 960], 64, 32, 8),          # empty prefix; a 64-key last prefix tile
    ([96 * 3, 96 * 40], 96, 32, 8),           # second row block with one M-tile only
    ([48 * 7, 48 * 100, 0], 48, 32, 8),       # second M-tile of 16 tokens
    ([64 * 11, 64 * 300], 64, 64, 8),         # G = 8: two row blocks per KV head
    ([32 * 5, 32 * 77], 32, 16, 8),           # G = 2, D = 32: one M-tile, single-CTA kernel
    ([2048, 30080], 128, 32, 8),              # D = 128: two row blocks, a full own tile
])
def test_pair_decode_matches_oracle_and_single_cta(cuda_lib, P, D, Hq, Hkv):
    case = workloads.make_decode_case(P, D=D, Hq=Hq, Hkv=Hkv, d=128, seed=51)
    r = DecodeRun(case)
    got = r.run().clone()
    assert r.status() == 0
    ref = _decode_ref(case)
    assert_close(got, ref, what=f"pair decode P={P} D={D} {Hq}/{Hkv}")
    with single_cta_kernel():
        one = r.run().clone()
    assert r.status() == 0
    assert_close(one, ref, what="single-CTA decode")
    diff = (got.double() - one.double()).abs()
    assert float(diff.max()) <= 2e-2 and float(diff.mean()) <= 2e-3


def test_pair_decode_serving_with_commit_and_splits(cuda_lib):
    """Batch 64 serving step with commit: pair and single-CTA kernels agree,
    the commit is bit-exact, the tile counters are unchanged."""
    import block_causal_paged_gb300 as bca
    case = workloads.serving_decode(seed=5, D=64, keep_logical=False)
    r = DecodeRun(case)
    bca.workspace_init(r.ws)
    got = r.run(commit=True).clone()
    assert r.status() == 0
    counts_pair = bca.read_tile_counters(r.ws)
    kp_pair = r.k_pool.clone()
    r2 = DecodeRun(case)
    with single_cta_kernel():
        bca.workspace_init(r2.ws)
        one = r2.run(commit=True).clone()
    assert r2.status() == 0
    assert counts_pair == bca.read_tile_counters(r2.ws)
    assert torch.equal(kp_pair.view(torch.int16), r2.k_pool.view(torch.int16))
    diff = (got.double() - one.double()).abs()
    assert float(diff.max()) <= 2e-2 and float(diff.mean()) <= 2e-3


def test_pair_decode_repeated_launches_are_stable(cuda_lib):
    """Twenty launches in a row on one workspace (work counter reset by the
    last CTA, mailbox and barrier phases restart per launch): identical bits."""
    case = workloads.make_decode_case([4096, 128, 20480, 640], D=64, Hq=32, Hkv=8, d=128,
                                      seed=52, keep_logical=False)
    r = DecodeRun(case)
    first = r.run().clone()
    for _ in range(19):
        r.run()
    assert r.status() == 0
    assert torch.equal(first.view(torch.int16), r.out.view(torch.int16))


@pytest.mark.parametrize("lens,D,Hq,Hkv", [
    ([300, 512, 64, 1000], 64, 8, 2),       # ragged lengths, partial diagonal tiles
    ([1024, 129], 16, 32, 8),               # D = 16
    ([384, 77], 384, 6, 2),                 # G = 3: the last head pair has one head
    ([2048], 128, 16, 8),                   # G = 2
])
def test_pair_prefill_matches_oracle_and_single_cta(cuda_lib, lens, D, Hq, Hkv):
    case = workloads.make_prefill_case(lens, D=D, Hq=Hq, Hkv=Hkv, d=128, seed=53)
    r = PrefillRun(case, write_pages=False)
    got = r.run().clone()
    assert r.status() == 0
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, case.D)
    assert_close(got, ref, what=f"pair prefill {lens} D={D}")
    with single_cta_kernel():
        one = r.run().clone()
    assert r.status() == 0
    diff = (got.double() - one.double()).abs()
    assert float(diff.max()) <= 2e-2 and float(diff.mean()) <= 2e-3


@pytest.mark.parametrize("single", [False, True])
def test_decode_with_growing_scores_rescales(cuda_lib, single):
    """Keys scaled by 1 + 3t in prefix tile t: each new tile raises the row
    maxima by far more than 2^8 (in exp2 units), so the online softmax
    rescales O at most tiles (the rare path of both kernels), including
    across split-KV chunks; outputs against the oracle."""
    P = [2048, 4096, 640]
    case = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=57)
    for b, Pb in enumerate(P):
        f = (1.0 + 3.0 * (torch.arange(Pb) // 128)).to(torch.float32)[:, None, None]
        case.k_prefix[b] = (case.k_prefix[b].float() * f).to(torch.bfloat16)
        workloads.write_logical_into_pool(case.pool, b, case.k_prefix[b], case.v_prefix[b])
    r = DecodeRun(case)
    if single:
        with single_cta_kernel():
            got = r.run().clone()
    else:
        got = r.run().clone()
    assert r.status() == 0
    assert_close(got, _decode_ref(case), what=f"growing scores, single={single}")


def _mc_ref(c, window=0):
    return oracle.multicanvas(c.q_live, c.k_live, c.v_live, c.live_pos, c.live_count, c.arena_k,
                              c.arena_v, c.arena_pos, c.prompt_len, c.canvas_len, window=window)


@pytest.mark.parametrize("args,window,shuffle", [
    ((4, 1024, 3, 256, 32, 8, 128), 0, False),    # the 3-canvas step (prompt 1024)
    ((3, 300, 4, 96, 16, 4, 128), 0, True),       # ragged arena and prompt, shuffled live rows
    ((4, 1024, 5, 256, 32, 8, 128), 1024, False),  # 5 canvases under a 1024-token window
    ((2, 100, 3, 64, 32, 8, 128), 50, True),       # a narrow band, shuffled live rows
])
def test_pair_multicanvas_matches_oracle_and_single_cta(cuda_lib, args, window, shuffle):
    """The multicanvas step on CTA pairs: key masks from stored positions
    (arena kv_pos, live_pos), the band, ragged arena chunks whose unused pool
    slots hold NaN; live rows against the oracle and the single-CTA kernel."""
    from _gpu_cases import MulticanvasRun
    c = workloads.make_multicanvas_case(*args, seed=61, shuffle_live=shuffle)
    m = torch.from_numpy(np.arange(c.q_live.shape[1])[None, :] < c.live_count.numpy()[:, None])
    r = MulticanvasRun(c, promote=False)
    got = r.run(window=window).cpu().clone()
    assert r.status() == 0
    ref = _mc_ref(c, window)
    assert_close(got[m], ref[m.numpy()], what=f"pair multicanvas {args} window {window}")
    with single_cta_kernel():
        one = MulticanvasRun(c, promote=False).run(window=window).cpu()
    diff = (got[m].double() - one[m].double()).abs()
    assert float(diff.max()) <= 2e-2 and float(diff.mean()) <= 2e-3


@pytest.mark.parametrize("P,D", [([5, 77, 1000, 33], 48), ([129, 3000], 72)])
def test_pair_decode_ragged_chunks(cuda_lib, P, D):
    """Blocks and prefixes that are not whole 16-key chunks on CTA pairs (the
    extend's causal mask, and a block decode after prefixes that are multiples
    of D but not of 16): the ragged V rows, NaN in the pool, are zeroed."""
    case = workloads.make_decode_case(P, D=D, Hq=32, Hkv=8, d=128, seed=63)
    r = DecodeRun(case)
    got = r.run(extend=True).clone()
    assert r.status() == 0
    ref = oracle.extend(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix)
    assert_close(got, ref, what=f"pair extend P={P} D={D}")
    Pd = [p_ // D * D for p_ in P]
    cd = workloads.make_decode_case(Pd, D=D, Hq=32, Hkv=8, d=128, seed=64)
    rd = DecodeRun(cd)
    gd = rd.run().clone()
    assert rd.status() == 0
    assert_close(gd, _decode_ref(cd), what=f"pair decode P={Pd} D={D}")


def test_pair_output_only_16_byte_aligned(cuda_lib):
    """The pair kernel stores each row's output 32 bytes at a time when the
    output is 32-byte aligned, 16 bytes at a time otherwise: an output buffer
    offset by 16 bytes gets the same bits as an aligned one."""
    case = workloads.make_decode_case([1024, 64 * 9, 4096], D=64, Hq=32, Hkv=8, d=128, seed=21)
    r = DecodeRun(case)
    ref = r.run().clone()
    assert r.status() == 0
    assert r.out.data_ptr() % 32 == 0
    flat = torch.empty(r.out.numel() + 8, dtype=r.out.dtype, device=r.out.device)
    r.out = flat[8:].view(r.out.shape)
    assert r.out.data_ptr() % 32 == 16
    got = r.run()
    assert r.status() == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert_close(got, _decode_ref(case), what="pair decode, 16-byte aligned output")
