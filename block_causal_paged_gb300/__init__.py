"""Python binding of libbca.so, block-causal paged attention on GB300 (sm_103a).

Argument marshalling only: every function below forwards raw device pointers
and sizes to the C ABI declared in include/bca.h, on the current PyTorch CUDA
stream unless a stream is given.  PyTorch is used for device memory and
streams; all computation happens in the library's CUDA kernels.  There is no
fallback: if the library is missing or the device is not an sm_103 GPU, the
calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libbca.so")

ABI_VERSION = 1
OK = 0
ERR_INVALID_ARG = -1
ERR_NULL = -2
ERR_ALIGN = -3
ERR_WORKSPACE = -4
ERR_CAPACITY = -5
ERR_CUDA = -6
ERR_UNSUPPORTED = -7
ERR_PAGE_SHARED = -8
ERR_PAGE_RANGE = -9
ERR_DEVICE_PAGE_OOB = -16
ERR_DEVICE_BAD_LENGTH = -17
ERR_DEVICE_TIMEOUT = -18

OP_DECODE, OP_PREFILL, OP_MULTICANVAS, OP_COMMIT, OP_DECODE_MIN = 1, 2, 3, 4, 5

# Every C entry point of include/bca.h, with its ctypes signature.
_vp, _i32, _i64, _sz, _f = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class Dims(ctypes.Structure):
    """struct bca_dims."""
    _fields_ = [("version", _i32), ("batch", _i32), ("block_size", _i32),
                ("num_q_heads", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
                ("page_size", _i32), ("num_pages", _i32), ("max_pages_per_seq", _i32),
                ("softmax_scale", _f)]


class KernelTimes(ctypes.Structure):
    """struct bca_kernel_times."""
    _fields_ = [("launches", _i32 * 7), ("total_ms", ctypes.c_double * 7)]


KERNEL_NAMES = ("attention", "combine", "commit", "promote", "plan", "confidence", "qkv_post")

_DP = ctypes.POINTER(Dims)
SIGNATURES = {
    "bca_version": ([], ctypes.c_int),
    "bca_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "bca_workspace_size": ([_DP, ctypes.c_int], _sz),
    "bca_workspace_init": ([_vp, _sz, _vp], ctypes.c_int),
    "bca_read_device_status": ([_vp, _vp], ctypes.c_int),
    "bca_read_tile_counters": ([_vp, ctypes.POINTER(_i64), _vp], ctypes.c_int),
    "bca_decode": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _sz, _vp],
                   ctypes.c_int),
    "bca_extend": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _sz, _vp],
                   ctypes.c_int),
    "bca_qkv_post": ([_DP, _vp, _vp, _vp, _vp, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                      _vp, _sz, _vp], ctypes.c_int),
    "bca_commit_kv": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp], ctypes.c_int),
    "bca_prefill": ([_DP, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
                    ctypes.c_int),
    "bca_multicanvas": ([_DP, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                         _vp, _vp, _vp, _i32, _vp, _vp, _sz, _vp], ctypes.c_int),
    "bca_multicanvas_window": ([_DP, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp,
                                _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _sz, _vp], ctypes.c_int),
    "bca_validate_page_table": ([_DP, _vp, _vp, ctypes.POINTER(_i32), ctypes.POINTER(_i32)],
                                ctypes.c_int),
    "bca_decode_static_scratch": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                   _vp, _vp], ctypes.c_int),
    "bca_confidence": ([_i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp], ctypes.c_int),
    "bca_profile_start": ([_i32], ctypes.c_int),
    "bca_profile_stop": ([ctypes.POINTER(KernelTimes)], ctypes.c_int),
}

_lib = None


class BcaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def load(path: str | None = None):
    """Load libbca.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} not found: build it with block_causal_paged_gb300/build.py "
            "(or __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().bca_status_string(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != OK:
        raise BcaError(rc, where)


def dims(batch: int, block_size: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
         page_size: int = 16, num_pages: int = 1, max_pages_per_seq: int = 1,
         softmax_scale: float = 0.0) -> Dims:
    return Dims(ABI_VERSION, batch, block_size, num_q_heads, num_kv_heads, head_dim, page_size,
                num_pages, max_pages_per_seq, softmax_scale)


def workspace_size(d: Dims, op: int) -> int:
    return int(load().bca_workspace_size(ctypes.byref(d), op))


def new_workspace(d: Dims, op: int, device="cuda", stream=None):
    """Allocate (torch) and initialise a workspace for `op`."""
    import torch
    n = workspace_size(d, op)
    if n == 0:
        raise BcaError(ERR_INVALID_ARG, "workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(load().bca_workspace_init(ws.data_ptr(), n, _stream(stream)), "bca_workspace_init")
    return ws


def workspace_init(ws, stream=None):
    _check(load().bca_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "bca_workspace_init")


def read_device_status(ws, stream=None) -> int:
    return int(load().bca_read_device_status(_ptr(ws), _stream(stream)))


def read_tile_counters(ws, stream=None) -> tuple[int, int, int]:
    arr = (_i64 * 3)()
    _check(load().bca_read_tile_counters(_ptr(ws), arr, _stream(stream)), "bca_read_tile_counters")
    return int(arr[0]), int(arr[1]), int(arr[2])


def bca_decode(d: Dims, q, k_blk, v_blk, k_pool, v_pool, page_table, prefix_len, out,
               commit: bool, workspace, stream=None) -> None:
    rc = load().bca_decode(ctypes.byref(d), _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(k_pool),
                           _ptr(v_pool), _ptr(page_table), _ptr(prefix_len), _ptr(out),
                           1 if commit else 0, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "bca_decode")


def bca_extend(d: Dims, q, k_new, v_new, k_pool, v_pool, page_table, prefix_len, out,
               commit: bool, workspace, stream=None) -> None:
    """Short causal extend: d.block_size new tokens per sequence (see include/bca.h)."""
    rc = load().bca_extend(ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                           _ptr(v_pool), _ptr(page_table), _ptr(prefix_len), _ptr(out),
                           1 if commit else 0, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "bca_extend")


def bca_qkv_post(d: Dims, qkv, positions, q_out, k_out, v_out, workspace, q_norm_w=None,
                 k_norm_w=None, eps: float = 1e-6, rope_theta: float = 0.0, write_pos=None,
                 k_pool=None, v_pool=None, page_table=None, kv_pos=None, stream=None) -> None:
    """Norms + RoPE of the QKV projection's output, optional cache write (see include/bca.h)."""
    rc = load().bca_qkv_post(ctypes.byref(d), _ptr(qkv), _ptr(positions), _ptr(q_norm_w),
                             _ptr(k_norm_w), float(eps), float(rope_theta), _ptr(q_out),
                             _ptr(k_out), _ptr(v_out), _ptr(write_pos), _ptr(k_pool),
                             _ptr(v_pool), _ptr(page_table), _ptr(kv_pos), _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(rc, "bca_qkv_post")


def bca_decode_static_scratch(d: Dims, q, k_blk, v_blk, k_pool, v_pool, page_table, prefix_len,
                              out, commit: bool, device_status=None, stream=None) -> None:
    """bca_decode with the library's own fixed scratch array (no workspace).

    For callers that cannot allocate device memory on this path; see
    include/bca.h for the size limit and the sharing rules."""
    rc = load().bca_decode_static_scratch(ctypes.byref(d), _ptr(q), _ptr(k_blk), _ptr(v_blk),
                                          _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                          _ptr(prefix_len), _ptr(out), 1 if commit else 0,
                                          _ptr(device_status), _stream(stream))
    _check(rc, "bca_decode_static_scratch")


def bca_commit_kv(d: Dims, k_blk, v_blk, k_pool, v_pool, page_table, start_pos, num_tokens: int,
                  workspace, stream=None) -> None:
    rc = load().bca_commit_kv(ctypes.byref(d), _ptr(k_blk), _ptr(v_blk), _ptr(k_pool),
                              _ptr(v_pool), _ptr(page_table), _ptr(start_pos), int(num_tokens),
                              _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "bca_commit_kv")


DTYPE_BF16, DTYPE_F32 = 0, 1


def bca_confidence(logits, argmax, conf, vocab: int | None = None, stream=None) -> None:
    """Top prediction and its probability per row of `logits` ([rows, ld] bf16
    or fp32 device tensor; the first `vocab` columns are the vocabulary)."""
    import torch
    rows, ld = logits.shape
    dtype = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}.get(logits.dtype)
    if dtype is None:
        raise BcaError(ERR_INVALID_ARG, "bca_confidence: logits must be bf16 or fp32")
    rc = load().bca_confidence(int(rows), int(ld if vocab is None else vocab), int(logits.stride(0)),
                               dtype, _ptr(logits), _ptr(argmax), _ptr(conf), _stream(stream))
    _check(rc, "bca_confidence")


def bca_prefill(d: Dims, q, k, v, cu_seqlens, total_tokens: int, max_seqlen: int, k_pool, v_pool,
                page_table, out, workspace, stream=None) -> None:
    rc = load().bca_prefill(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens),
                            int(total_tokens), int(max_seqlen), _ptr(k_pool), _ptr(v_pool),
                            _ptr(page_table), _ptr(out), _ptr(workspace), workspace.numel(),
                            _stream(stream))
    _check(rc, "bca_prefill")


def bca_multicanvas(d: Dims, q_live, k_live, v_live, live_pos, live_count, max_live: int,
                    prompt_len: int, n_canvas: int, k_pool, v_pool, page_table, kv_pos,
                    arena_len, commit_rows, commit_count, max_commit: int, out, workspace,
                    stream=None, window: int = 0) -> None:
    """window > 0 calls bca_multicanvas_window (sliding-window layer)."""
    if window:
        rc = load().bca_multicanvas_window(
            ctypes.byref(d), _ptr(q_live), _ptr(k_live), _ptr(v_live), _ptr(live_pos),
            _ptr(live_count), int(max_live), int(prompt_len), int(n_canvas), int(window),
            _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(kv_pos), _ptr(arena_len),
            _ptr(commit_rows), _ptr(commit_count), int(max_commit), _ptr(out), _ptr(workspace),
            workspace.numel(), _stream(stream))
        _check(rc, "bca_multicanvas_window")
        return
    rc = load().bca_multicanvas(ctypes.byref(d), _ptr(q_live), _ptr(k_live), _ptr(v_live),
                                _ptr(live_pos), _ptr(live_count), int(max_live), int(prompt_len),
                                int(n_canvas), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                _ptr(kv_pos), _ptr(arena_len), _ptr(commit_rows),
                                _ptr(commit_count), int(max_commit), _ptr(out), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "bca_multicanvas")


def bca_validate_page_table(d: Dims, page_table_host, used_tokens_host) -> tuple[int, int, int]:
    """Host-side check; arguments are CPU int32 tensors.  Returns (status, seq, entry)."""
    bs, be = _i32(-1), _i32(-1)
    rc = load().bca_validate_page_table(ctypes.byref(d), _ptr(page_table_host),
                                        _ptr(used_tokens_host), ctypes.byref(bs), ctypes.byref(be))
    return int(rc), int(bs.value), int(be.value)


def profile_start(max_launches: int = 4096) -> None:
    _check(load().bca_profile_start(int(max_launches)), "bca_profile_start")


def profile_stop() -> dict:
    """{kernel name: (launches, total device ms)} since profile_start."""
    t = KernelTimes()
    _check(load().bca_profile_stop(ctypes.byref(t)), "bca_profile_stop")
    return {n: (int(t.launches[i]), float(t.total_ms[i])) for i, n in enumerate(KERNEL_NAMES)}


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
