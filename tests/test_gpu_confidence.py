"""GPU parity of bca_confidence (softmax-plus-argmax over the vocabulary)
against the fp64 oracle.

Tolerance: the kernel sums exp(l - max) in fp32 (per thread, then a tree
over 256 threads) with ex2.approx (relative error ~2^-22 per term); over a
vocabulary of 2^18 the sum's relative error stays far below 1e-4, so
conf is checked with rtol 1e-4.  The argmax is an exact comparison of the
input values on both sides and must match exactly."""
import numpy as np
import pytest
import torch

import block_causal_paged_gb300 as bca
import oracle
import workloads

pytestmark = pytest.mark.gpu
RTOL = 1e-4


def _run(logits, vocab=None):
    rows = logits.shape[0]
    arg = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    conf = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
    bca.bca_confidence(logits, arg, conf, vocab=vocab)
    torch.cuda.synchronize()
    return arg.cpu().numpy(), conf.cpu().numpy()


def _check(logits_cpu, arg, conf, what):
    want_arg, want_conf = oracle.confidence(logits_cpu.float().numpy())
    assert np.array_equal(arg, want_arg), f"{what}: argmax"
    assert np.allclose(conf, want_conf, rtol=RTOL, atol=1e-7), \
        f"{what}: conf max rel err {np.max(np.abs(conf - want_conf) / np.maximum(want_conf, 1e-30)):.2e}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("vocab", [1, 7, 8, 9, 1000, 4097, 32003])
def test_shapes(cuda_lib, dtype, vocab):
    x = workloads.confidence_logits(5, vocab, seed=vocab, dtype=dtype)
    arg, conf = _run(x.cuda())
    _check(x, arg, conf, f"{dtype} V={vocab}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ties_go_to_the_lowest_index(cuda_lib, dtype):
    V = 20000
    x = torch.full((6, V), -3.0, dtype=dtype)
    spots = [(0, [5, 9000]), (1, [19999, 12]), (2, [2048, 2049, 2056]), (3, [8, 8 * 256 + 8]),
             (4, [7, 15, 23, 31]), (5, [18000, 17999])]
    for r, cols in spots:
        for c in cols:
            x[r, c] = 4.0
    arg, conf = _run(x.cuda())
    _check(x, arg, conf, "ties")
    assert list(arg) == [5, 12, 2048, 8, 7, 17999]


def test_minus_inf(cuda_lib):
    V = 3000
    x = workloads.confidence_logits(3, V, seed=4, dtype=torch.float32)
    x[0, ::2] = -float("inf")                      # masked half of the vocabulary
    x[1, :] = -float("inf")                        # no distribution: (0, 0)
    x[2, :2999] = -float("inf")                    # only the last token left: (2999, 1)
    arg, conf = _run(x.cuda())
    _check(x, arg, conf, "-inf")
    assert arg[1] == 0 and conf[1] == 0.0 and arg[2] == 2999 and conf[2] == 1.0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_padded_row_stride(cuda_lib, dtype):
    vocab, ld = 5000, 5120
    full = workloads.confidence_logits(4, ld, seed=9, dtype=dtype)
    full[:, vocab:] = 1e4                          # padding past the vocabulary must be ignored
    arg, conf = _run(full.cuda(), vocab=vocab)
    _check(full[:, :vocab], arg, conf, "padded")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_unaligned_row_starts(cuda_lib, dtype):
    """Rows of a column-sliced view start at every offset modulo 16 bytes."""
    full = workloads.confidence_logits(9, 2051, seed=13, dtype=dtype).cuda()
    view = full[:, 3:]                               # vocab 2048, row stride 2051
    arg, conf = _run(view)
    _check(view.cpu(), arg, conf, "unaligned rows")


def test_vocab_262144(cuda_lib):
    x = workloads.confidence_logits(64, 262144, seed=1)
    arg, conf = _run(x.cuda())
    _check(x, arg, conf, "V=262144")


def test_step_size_sampled_rows(cuda_lib):
    """The benchmarked size: 4096 rows (64 sequences x 64 block positions) of
    262144 bf16 logits (2 GiB), checked on sampled rows."""
    rows, V = 4096, 262144
    x = workloads.confidence_logits(rows, V, seed=2, device="cuda")
    arg, conf = _run(x)
    sample = np.random.default_rng(0).choice(rows, 24, replace=False)
    sample.sort()
    xs = x[torch.as_tensor(sample, device="cuda")].cpu()
    _check(xs, arg[sample], conf[sample], "4096 x 262144 sample")


def test_zero_rows_is_a_no_op(cuda_lib):
    x = torch.zeros((0, 100), dtype=torch.bfloat16, device="cuda")
    _run(x)
