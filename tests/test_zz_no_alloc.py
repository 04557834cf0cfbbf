"""bca_decode_static_scratch: the decode step for callers that cannot allocate.

Some callers of this library are not allowed to allocate device memory on the
decode path (an engine that owns all device memory and gives its plugins no
allocator, a serving loop where an allocation could stall the device or fail
under fragmentation).  For them the library offers a decode entry point whose
scratch lives in a fixed array inside the library.  These tests call it
through the C ABI:

- twice in a row, on different inputs with long prefixes (so split-KV
  partials in the scratch array are used and the second call runs on the
  array's leftover contents), each output checked against the fp64 oracle
  within the tolerance of the other GPU tests and against the ordinary
  workspace entry point;
- with the commit on, the pools afterwards bit-exact against the oracle's
  commit;
- on long prefixes whose full plan needs more split-KV slots than the fixed
  array holds: the device status stays 0 (the kernel reports
  BCA_ERR_WORKSPACE when a plan does not fit the scratch), so a smaller plan
  with fewer splits was taken, and the output still matches;
- on the benchmarked batch (64 sequences, D = 64).

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu_cases import MAX_ABS, MEAN_ABS, DecodeRun, assert_close

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20   # size of the library's fixed scratch array


def _static_decode(bca, r, status, commit=0):
    out = torch.empty_like(r.q)
    stream = torch.cuda.current_stream().cuda_stream
    rc = bca.load().bca_decode_static_scratch(
        ctypes.byref(r.d), r.q.data_ptr(), r.k_blk.data_ptr(), r.v_blk.data_ptr(),
        r.k_pool.data_ptr(), r.v_pool.data_ptr(), r.page_table.data_ptr(),
        r.prefix_len.data_ptr(), out.data_ptr(), commit, status.data_ptr(), stream)
    assert rc == bca.OK, bca.status_string(rc)
    torch.cuda.synchronize()
    return out


def _oracle(case, seqs=None):
    return oracle.decode(case.q, case.k_blk, case.v_blk, case.k_prefix, case.v_prefix, seqs=seqs)


def test_static_scratch_decode_matches_oracle_twice(cuda_lib):
    bca = cuda_lib
    for seed, P in ((3, [32768, 8192, 512, 128, 4096]), (4, [128, 20480, 64 * 9, 32768])):
        case = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=seed)
        r = DecodeRun(case)
        ref = r.run().clone()
        assert r.status() == 0
        status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
        got = _static_decode(bca, r, status)
        assert int(status.item()) == 0
        assert_close(got, _oracle(case), what=f"static scratch vs oracle, seed {seed}")
        diff = (got.double() - ref.double()).abs().cpu().numpy()
        assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())


def test_static_scratch_commit_is_bit_exact(cuda_lib):
    bca = cuda_lib
    P = [64 * 5, 0, 4096, 30016]
    case = workloads.make_decode_case(P, D=64, Hq=16, Hkv=4, d=128, seed=6)
    r = DecodeRun(case)
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    got = _static_decode(bca, r, status, commit=1)
    assert int(status.item()) == 0
    assert_close(got, _oracle(case), what="static scratch with commit vs oracle")
    S = case.pool.page_size
    for name, pool, blk in (("k", r.k_pool, case.k_blk), ("v", r.v_pool, case.v_blk)):
        src = (case.pool.k_pool if name == "k" else case.pool.v_pool).view(torch.int16).numpy()
        want = oracle.commit(src, case.pool.page_table, case.prefix_len,
                             blk.view(torch.int16).numpy(), case.D, S)
        assert np.array_equal(pool.cpu().view(torch.int16).numpy(), want), name


def _full_plan_slots(r):
    """Split-KV slots of the plan made with the full workspace (the header's
    n_split_slots field, at byte 40)."""
    return int(r.ws[40:44].view(torch.int32).item())


def _static_slot_capacity(bca, r):
    per_slot = 16 + 256 * 2 * 4 + 256 * r.case.d * 4   # table entry, (max, sum), O
    return (STATIC_BYTES - bca.workspace_size(r.d, bca.OP_DECODE_MIN) - 512) // per_slot


def test_static_scratch_takes_a_smaller_plan_when_splits_do_not_fit(cuda_lib):
    """Eight 32768-token prefixes: the plan made with a full workspace splits
    every prefix into more chunks than the fixed array has split-KV slots
    for.  The call through the fixed array still succeeds (device status 0;
    the kernel reports BCA_ERR_WORKSPACE when a plan does not fit the
    scratch), so it planned fewer splits, and its output matches."""
    bca = cuda_lib
    case = workloads.make_decode_case([32768] * 8, D=64, Hq=32, Hkv=8, d=128, seed=8)
    r = DecodeRun(case)
    ref = r.run().clone()
    assert r.status() == 0
    assert _full_plan_slots(r) > _static_slot_capacity(bca, r) > 0
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    got = _static_decode(bca, r, status)
    assert int(status.item()) == 0
    diff = (got.double() - ref.double()).abs().cpu().numpy()
    assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())
    seqs = [0, 5]
    ref_o = _oracle(case, seqs=seqs)
    for b in seqs:
        assert_close(got[b], ref_o[b], what=f"static scratch, 32768-token prefix, seq {b}")


def test_static_scratch_serving_batch(cuda_lib):
    """The benchmarked batch (64 sequences, D = 64, prefixes log-uniform in
    [128, 32768]) through the fixed array."""
    bca = cuda_lib
    case = workloads.serving_decode(seed=2, D=64)
    r = DecodeRun(case)
    ref = r.run().clone()
    assert r.status() == 0
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    got = _static_decode(bca, r, status)
    assert int(status.item()) == 0
    diff = (got.double() - ref.double()).abs().cpu().numpy()
    assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())
    Pv = np.array(case.prefix_len)
    seqs = sorted({int(Pv.argmax()), int(Pv.argmin()), 7, 33})
    ref64 = _oracle(case, seqs=seqs)
    for b in seqs:
        assert_close(got[b], ref64[b], what=f"static scratch serving seq {b}")


def test_static_scratch_rejects_oversized_requests(cuda_lib):
    bca = cuda_lib
    # a batch whose minimum scratch (per-sequence table + work list) exceeds 16 MiB
    d = bca.dims(200000, 64, 32, 8, 128, 16, 1 << 16, 4)
    assert bca.workspace_size(d, bca.OP_DECODE_MIN) > STATIC_BYTES
    rc = bca.load().bca_decode_static_scratch(ctypes.byref(d), 16, 16, 16, 16, 16, 16, 16, 16, 0,
                                              None, None)
    assert rc == bca.ERR_WORKSPACE
