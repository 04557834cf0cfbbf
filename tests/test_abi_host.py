"""The C-ABI library builds, loads and exports every symbol include/bca.h
declares; host-side checks reject bad arguments before any launch.  CPU only:
no call here reaches a kernel."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bca():
    from block_causal_paged_gb300 import build
    build.build()
    import block_causal_paged_gb300 as m
    m.load()
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "bca.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bca_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound(bca):
    names = _declared_functions()
    assert "bca_decode" in names and "bca_multicanvas" in names
    lib = ctypes.CDLL(bca.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(bca.SIGNATURES), "binding and header disagree"


def test_version_and_status_strings(bca):
    assert bca.load().bca_version() == bca.ABI_VERSION
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -16, -17, -18):
        s = bca.status_string(code)
        assert s and s != "unknown status"


def _d(bca, **kw):
    base = dict(batch=2, block_size=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
                page_size=16, num_pages=64, max_pages_per_seq=16)
    base.update(kw)
    return bca.dims(**base)


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(num_q_heads=30), dict(page_size=8),
                                 dict(page_size=24), dict(page_size=272), dict(block_size=0),
                                 dict(num_pages=0), dict(softmax_scale=-1.0)])
def test_invalid_dims_rejected_without_launch(bca, bad):
    d = _d(bca, **bad)
    assert bca.workspace_size(d, bca.OP_DECODE) == 0
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    rc = bca.load().bca_decode(ctypes.byref(d), p, p, p, p, p, p, p, p, 0, p, 1 << 20, None)
    assert rc == bca.ERR_INVALID_ARG


@pytest.mark.parametrize("S", [16, 32, 64, 128, 256])
def test_page_sizes_accepted(bca, S):
    """Any multiple of 16 from 16 to 256 tokens per page."""
    assert bca.workspace_size(_d(bca, page_size=S), bca.OP_DECODE) > 0


def test_wrong_abi_version_rejected(bca):
    d = _d(bca)
    d.version = 99
    assert bca.workspace_size(d, bca.OP_DECODE) == 0


def test_null_and_alignment_checks(bca):
    d = _d(bca)
    lib = bca.load()
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    rc = lib.bca_decode(ctypes.byref(d), a, a, a, a, a, a, a, None, 0, a, 1 << 20, None)
    assert rc == bca.ERR_NULL
    rc = lib.bca_decode(ctypes.byref(d), a + 2, a, a, a, a, a, a, a, 0, a, 1 << 20, None)
    assert rc == bca.ERR_ALIGN
    rc = lib.bca_decode(ctypes.byref(d), a, a, a, a, a, a, a, a, 2, a, 1 << 20, None)
    assert rc == bca.ERR_INVALID_ARG


def test_capacity_and_workspace_checks(bca):
    lib = bca.load()
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    d = _d(bca, block_size=512, max_pages_per_seq=16)   # 512 > 16 pages * 16
    rc = lib.bca_decode(ctypes.byref(d), a, a, a, a, a, a, a, a, 0, a, 1 << 20, None)
    assert rc == bca.ERR_CAPACITY
    d = _d(bca)
    rc = lib.bca_decode(ctypes.byref(d), a, a, a, a, a, a, a, a, 0, a, 16, None)
    assert rc == bca.ERR_WORKSPACE
    rc = lib.bca_commit_kv(ctypes.byref(d), a, a, a, a, a, a, 65, a, 256, None)
    assert rc == bca.ERR_INVALID_ARG            # more rows than the block holds


def test_zero_batch_is_a_no_op(bca):
    d = _d(bca, batch=0)
    rc = bca.load().bca_decode(ctypes.byref(d), None, None, None, None, None, None, None, None,
                               0, None, 0, None)
    assert rc == bca.OK


def test_workspace_size_grows_with_batch(bca):
    s1 = bca.workspace_size(_d(bca, batch=8), bca.OP_DECODE)
    s2 = bca.workspace_size(_d(bca, batch=64), bca.OP_DECODE)
    assert 0 < s1 < s2
    assert bca.workspace_size(_d(bca), bca.OP_PREFILL) == 256


def test_multicanvas_workspace_holds_arena_tile_summaries(bca):
    # header + 8 bytes per sequence and 128 entries of page-table capacity
    d = _d(bca, batch=3, max_pages_per_seq=20)          # 20 pages of 16 = 320 entries -> 3 tiles
    n = bca.workspace_size(d, bca.OP_MULTICANVAS)
    assert n == 256 + (3 * 3 * 8 + 255) // 256 * 256
    lib = bca.load()
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    rc = lib.bca_multicanvas(ctypes.byref(d), a, a, a, a, a, 32, 64, 2, a, a, a, a, a, None, None,
                             0, a, a, n - 1, None)
    assert rc == bca.ERR_WORKSPACE


def test_validate_page_table(bca):
    d = _d(bca, batch=2, num_pages=8, max_pages_per_seq=4)
    pt = torch.tensor([[0, 1, 2, -1], [3, 4, -1, -1]], dtype=torch.int32)
    used = torch.tensor([40, 20], dtype=torch.int32)
    assert bca.bca_validate_page_table(d, pt, used)[0] == bca.OK
    pt2 = pt.clone()
    pt2[1, 1] = 2                                           # shared with sequence 0
    assert bca.bca_validate_page_table(d, pt2, used) == (bca.ERR_PAGE_SHARED, 1, 1)
    pt3 = pt.clone()
    pt3[0, 2] = 8                                           # outside the pool
    assert bca.bca_validate_page_table(d, pt3, used) == (bca.ERR_PAGE_RANGE, 0, 2)
    used2 = torch.tensor([40, 100], dtype=torch.int32)      # beyond 4 pages of 16
    assert bca.bca_validate_page_table(d, pt, used2)[0] == bca.ERR_CAPACITY


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "block_causal_paged_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_kernels_never_trap():
    """No device code traps or asserts: a failure detected on the device is a
    status word the host reads (bca_read_device_status), never a fault."""
    import re
    csrc = os.path.join(ROOT, "block_causal_paged_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        code = re.sub(r"//[^\n]*", "", open(os.path.join(csrc, f)).read())
        assert "__trap" not in code and "brkpt" not in code, f
        assert not re.search(r"(?<!static_)assert\s*\(", code), f


def test_confidence_argument_errors(bca):
    """Host checks of bca_confidence that need no GPU."""
    import ctypes
    lib = bca.load()
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    f = lib.bca_confidence
    assert f(4, 0, 8, 0, base, base, base, None) == bca.ERR_INVALID_ARG      # empty vocabulary
    assert f(4, 8, 7, 0, base, base, base, None) == bca.ERR_INVALID_ARG      # ld < vocab
    assert f(4, 8, 8, 3, base, base, base, None) == bca.ERR_INVALID_ARG      # unknown dtype
    assert f(-1, 8, 8, 0, base, base, base, None) == bca.ERR_INVALID_ARG     # negative rows
    assert f(0, 8, 8, 0, None, None, None, None) == bca.OK                   # no rows: no-op
    assert f(4, 8, 8, 0, None, base, base, None) == bca.ERR_NULL
    assert f(4, 8, 8, 0, base + 1, base, base, None) == bca.ERR_ALIGN        # bf16 logits at an odd byte
    assert f(4, 8, 8, 1, base + 2, base, base, None) == bca.ERR_ALIGN        # fp32 logits at 2 bytes
    assert f(4, 8, 8, 0, base, base + 2, base, None) == bca.ERR_ALIGN        # int32 argmax misaligned


def test_extend_and_qkv_post_argument_errors(bca):
    """Host checks of bca_extend and bca_qkv_post that need no GPU."""
    lib = bca.load()
    buf = (ctypes.c_uint8 * 4096)()
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    d = _d(bca, block_size=9)
    assert lib.bca_extend(ctypes.byref(d), a, a, a, a, a, a, a, a, 2, a, 1 << 20, None) == \
        bca.ERR_INVALID_ARG                                   # commit flag not 0/1
    assert lib.bca_extend(ctypes.byref(d), a, a, a, a, a, a, None, a, 0, a, 1 << 20, None) == \
        bca.ERR_NULL
    f = lib.bca_qkv_post
    ok = (a, a, None, None, 1e-6, 0.0, a, a, a, None, None, None, None, None, a, 256, None)
    assert f(ctypes.byref(d), *ok[:4], -1.0, *ok[5:]) == bca.ERR_INVALID_ARG   # eps < 0
    assert f(ctypes.byref(d), *ok[:5], -2.0, *ok[6:]) == bca.ERR_INVALID_ARG   # theta < 0
    assert f(ctypes.byref(d), a, None, None, None, 1e-6, 1e4, a, a, a, None, None, None, None,
             None, a, 256, None) == bca.ERR_NULL                               # RoPE needs positions
    assert f(ctypes.byref(d), a, a, None, None, 1e-6, 0.0, a, a, a, a, None, None, None, None,
             a, 256, None) == bca.ERR_NULL                                     # write without pools
    assert f(ctypes.byref(d), a, a, None, None, 1e-6, 0.0, a, a, a, None, None, None, None, a,
             a, 256, None) == bca.ERR_INVALID_ARG                              # kv_pos without write
    assert f(ctypes.byref(d), a + 2, *ok[1:]) == bca.ERR_ALIGN
    assert f(ctypes.byref(d), *ok[:14], a, 16, None) == bca.ERR_WORKSPACE
    z = _d(bca, batch=0)
    assert f(ctypes.byref(z), *ok) == bca.OK                                   # empty batch: no-op
