"""bca_decode_static_scratch: the decode step for callers that cannot allocate.

Some callers of this library are not allowed to allocate device memory on the
decode path (an engine that owns all device memory and gives its plugins no
allocator, a serving loop where an allocation could stall the device or fail
under fragmentation).  For them the library offers a decode entry point whose
scratch lives in a fixed array inside the library.  This test calls it through
the C ABI twice in a row, on different inputs with long prefixes (so split-KV
partials in the scratch array are used and the second call runs on the
array's leftover contents), and checks each output against the ordinary
workspace entry point within the tolerance the other GPU tests use.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from _gpu_cases import MAX_ABS, MEAN_ABS, DecodeRun

pytestmark = pytest.mark.gpu


def _static_decode(bca, r, status):
    out = torch.empty_like(r.q)
    stream = torch.cuda.current_stream().cuda_stream
    rc = bca.load().bca_decode_static_scratch(
        ctypes.byref(r.d), r.q.data_ptr(), r.k_blk.data_ptr(), r.v_blk.data_ptr(),
        r.k_pool.data_ptr(), r.v_pool.data_ptr(), r.page_table.data_ptr(),
        r.prefix_len.data_ptr(), out.data_ptr(), 0, status.data_ptr(), stream)
    assert rc == bca.OK, bca.status_string(rc)
    torch.cuda.synchronize()
    return out


def test_static_scratch_decode_matches_workspace_decode(cuda_lib):
    bca = cuda_lib
    for seed, P in ((3, [32768, 8192, 512, 128, 4096]), (4, [128, 20480, 64 * 9, 32768])):
        case = workloads.make_decode_case(P, D=64, Hq=32, Hkv=8, d=128, seed=seed,
                                          keep_logical=False)
        r = DecodeRun(case)
        ref = r.run().clone()
        assert r.status() == 0
        status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
        got = _static_decode(bca, r, status)
        assert int(status.item()) == 0
        diff = (got.double() - ref.double()).abs().cpu().numpy()
        assert np.isfinite(got.float().cpu().numpy()).all()
        assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())


def test_static_scratch_rejects_oversized_requests(cuda_lib):
    bca = cuda_lib
    # a batch whose minimum scratch (per-sequence table + work list) exceeds 16 MiB
    d = bca.dims(200000, 64, 32, 8, 128, 16, 1 << 16, 4)
    assert bca.workspace_size(d, bca.OP_DECODE_MIN) > (16 << 20)
    rc = bca.load().bca_decode_static_scratch(ctypes.byref(d), 16, 16, 16, 16, 16, 16, 16, 16, 0,
                                              None, None)
    assert rc == bca.ERR_WORKSPACE
