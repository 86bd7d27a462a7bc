"""Host-side checks of the C ABI: the library loads without a GPU, exports
every function include/tw.h declares, and refuses bad arguments with the
documented status before any CUDA call.  Only fake (never dereferenced)
addresses are passed, and every call here returns before touching CUDA."""
import ctypes
import os
import re

import pytest

from reduce_residual_rmsnorm_tw_gb300 import build as twbuild
from reduce_residual_rmsnorm_tw_gb300 import tw

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "tw.h")

OK, INVALID, ALIGN, ALIAS, CUDA, UNSUP = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def lib():
    twbuild.build()
    return tw.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tw_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8, names
    for name in names:
        assert hasattr(lib, name), f"libtw.so does not export {name}"


def test_version_and_error_string(lib):
    assert tw.tw_version() == 10100
    assert isinstance(tw.tw_last_error_string(), str)


BASE = 0x7f0000000000  # fake, 16-byte aligned device addresses (never used)
MB = 1 << 20


def call(lib, n_parts=2, n_out=1, T=4, H=64, eps=1e-6, t0=0, t1=None,
         max_sms=8, dtype=0, path=0, partials=None, out=None, residual=None,
         weight=None, residual_out=None):
    t1 = T if t1 is None else t1
    partials = partials if partials is not None else [BASE + i * MB for i in range(n_parts)]
    out = out if out is not None else [BASE + (32 + k) * MB for k in range(n_out)]
    residual = BASE + 64 * MB if residual is None else residual
    weight = BASE + 65 * MB if weight is None else weight
    residual_out = BASE + 66 * MB if residual_out is None else residual_out
    p_arr = (ctypes.c_void_p * max(1, len(partials)))(*partials)
    o_arr = (ctypes.c_void_p * max(1, len(out)))(*out)
    return lib.tw_fused_reduce_add_rmsnorm_ex(
        p_arr, n_parts, residual, weight, o_arr, n_out, residual_out, T, H,
        eps, t0, t1, max_sms, None, dtype, path, None)


@pytest.mark.parametrize("kwargs,status", [
    ({"n_parts": 0}, INVALID),
    ({"n_parts": 17}, INVALID),
    ({"n_out": 0}, INVALID),
    ({"n_out": 9}, INVALID),
    ({"T": -1, "t1": 0}, INVALID),
    ({"H": 0}, INVALID),
    ({"t0": 3, "t1": 2}, INVALID),
    ({"t1": 5}, INVALID),
    ({"t0": -1}, INVALID),
    ({"eps": -1e-6}, INVALID),
    ({"eps": float("inf")}, INVALID),
    ({"eps": float("nan")}, INVALID),
    ({"max_sms": 0}, INVALID),
    ({"dtype": 2}, INVALID),
    ({"path": 7}, INVALID),
    ({"H": 12}, ALIGN),                       # 24 bytes per row
    ({"H": 6, "dtype": 1}, ALIGN),            # 24 bytes per row
    ({"residual": BASE + 64 * MB + 8}, ALIGN),
    ({"partials": [BASE, BASE + MB + 4]}, ALIGN),
    ({"T": 1 << 47, "t1": 1}, INVALID),       # buffers of 2^54 bytes: over 2^48
    ({"H": 16392}, UNSUP),                    # above the bf16 limit
    ({"H": 8196, "dtype": 1}, UNSUP),         # above the fp32 limit
    ({"residual_out": BASE + 64 * MB + 16}, ALIAS),   # overlaps residual, not equal
    ({"out": [BASE]}, ALIAS),                          # output == partials[0]
    ({"out": [BASE + 65 * MB - 64]}, ALIAS),           # overlaps weight
    ({"n_out": 2, "out": [BASE + 32 * MB, BASE + 32 * MB + 256]}, ALIAS),
    ({"out": [BASE + 66 * MB]}, ALIAS),                # out == residual_out
    ({"out": [BASE + 64 * MB]}, ALIAS),                # out == residual
])
def test_bad_arguments_are_refused(lib, kwargs, status):
    assert call(lib, **kwargs) == status
    assert tw.tw_last_error_string() != ""


def test_null_pointers_are_refused(lib):
    assert call(lib, partials=[BASE, 0]) == INVALID
    assert call(lib, out=[0]) == INVALID
    assert call(lib, residual=0) == INVALID
    p_arr = (ctypes.c_void_p * 1)(BASE)
    assert lib.tw_fused_reduce_add_rmsnorm_ex(
        None, 1, BASE + 64 * MB, BASE + 65 * MB, p_arr, 1, BASE + 66 * MB, 4, 64,
        1e-6, 0, 4, 8, None, 0, 0, None) == INVALID


def test_empty_range_is_a_no_op(lib):
    # t0 == t1 returns TW_OK before any CUDA call, even without a GPU.
    assert call(lib, t0=2, t1=2) == OK
    assert call(lib, T=0, t0=0, t1=0) == OK


def test_in_place_residual_is_allowed_by_the_checks(lib):
    # residual_out == residual passes the alias rule; with an empty range no
    # kernel is launched.
    assert call(lib, residual_out=BASE + 64 * MB, t0=1, t1=1) == OK


def test_split_launch_argument_checks(lib):
    p_arr = (ctypes.c_void_p * 2)(BASE, BASE + MB)
    o_arr = (ctypes.c_void_p * 1)(BASE + 32 * MB)
    args = [p_arr, 2, BASE + 64 * MB, BASE + 65 * MB, o_arr, 1, BASE + 66 * MB]
    assert lib.tw_split_launch(*args, 8, 64, 1e-6, 9, 8, None, None, 0) == INVALID
    assert lib.tw_split_launch(*args, 8, 12, 1e-6, 4, 8, None, None, 0) == ALIGN
    assert lib.tw_split_launch(*args, 0, 64, 1e-6, -1, 8, None, None, 0) == OK


def test_binding_marshalling_checks():
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        tw.tw_fused_reduce_add_rmsnorm([x], x, torch.zeros(63, dtype=torch.bfloat16),
                                       [x.clone()], x.clone(), 1e-6)
    with pytest.raises(ValueError):
        tw.tw_fused_reduce_add_rmsnorm([x.float()], x, torch.zeros(64, dtype=torch.bfloat16),
                                       [x.clone()], x.clone(), 1e-6)
    with pytest.raises(ValueError):
        tw.tw_fused_reduce_add_rmsnorm_f32([x], x, torch.zeros(64, dtype=torch.bfloat16),
                                           [x.clone()], x.clone(), 1e-6)
    # Well-formed CPU tensors: refused for a device entry point before any
    # CUDA call, and unpinned ones for a host entry point.
    w = torch.zeros(64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA device"):
        tw.tw_fused_reduce_add_rmsnorm([x], x, w, [x.clone()], x.clone(), 1e-6)
    with pytest.raises(ValueError, match="pinned"):
        tw.tw_fused_reduce_add_rmsnorm_host_noalloc([x], x, w, [x.clone()], x.clone(), 1e-6)


def test_colsplit_slice_alignment(lib):
    p_arr = (ctypes.c_void_p * 3)(BASE, BASE + MB, BASE + 2 * MB)
    o_arr = (ctypes.c_void_p * 1)(BASE + 32 * MB)
    # H = 4096 bf16 over 3 ranks: slice bounds 1365 and 2730 columns are not
    # 16-byte aligned; over 2 ranks they are (checked with an empty range).
    args = [BASE + 64 * MB, BASE + 65 * MB, o_arr, 1, BASE + 66 * MB, 4, 4096, 1e-6]
    assert lib.tw_fused_reduce_add_rmsnorm_colsplit(p_arr, 3, *args, 0, 4, 8, None, 0) == ALIGN
    assert lib.tw_fused_reduce_add_rmsnorm_colsplit(p_arr, 2, *args, 2, 2, 8, None, 0) == OK
    assert lib.tw_fused_reduce_add_rmsnorm_colsplit(p_arr, 2, *args, 0, 4, 8, None, 7) == INVALID


def test_host_entry_workspace_and_argument_checks(lib):
    need = tw.tw_host_workspace_bytes(8, 1, 8192, 128, torch_bf16())
    row = 8192 * 2
    chunk = 128 * row
    assert need == row + 2 * (8 + 1 + 1 + 1) * chunk
    p_arr = (ctypes.c_void_p * 2)(BASE, BASE + MB)
    o_arr = (ctypes.c_void_p * 1)(BASE + 32 * MB)
    args = [p_arr, 2, BASE + 64 * MB, BASE + 65 * MB, o_arr, 1, BASE + 66 * MB, 4, 64, 1e-6]
    ws = BASE + 128 * MB
    big = 1 << 30
    f = lib.tw_fused_reduce_add_rmsnorm_host
    assert f(*args, 0, 4, 8, ws, big, -1, None, 0) == INVALID       # chunk_tokens < 0
    # chunk_tokens 0 reads the tensors in place (no workspace): with no GPU
    # the call stops at its first CUDA call, with one at the check that the
    # fake addresses are mapped host memory.
    assert f(*args, 0, 4, 8, None, 0, 0, None, 0) in (CUDA, INVALID)
    assert f(*args, 2, 2, 8, None, 0, 0, None, 0) == OK             # empty range: no-op
    assert f(*args, 0, 4, 8, None, big, 2, None, 0) == INVALID      # no workspace
    assert f(*args, 0, 4, 8, ws + 16, big, 2, None, 0) == ALIGN     # workspace alignment
    assert f(*args, 0, 4, 8, ws, 100, 2, None, 0) == INVALID        # workspace too small
    assert f(*args, 2, 2, 8, ws, big, 2, None, 0) == OK             # empty range: no-op


def torch_bf16():
    import torch
    return torch.bfloat16


def test_flags_argument_checks(lib):
    p_arr = (ctypes.c_void_p * 2)(BASE, BASE + MB)
    o_arr = (ctypes.c_void_p * 1)(BASE + 32 * MB)
    args = [p_arr, 2, BASE + 64 * MB, BASE + 65 * MB, o_arr, 1, BASE + 66 * MB, 4, 64, 1e-6,
            0, 4, 8, None, 0]
    f = lib.tw_fused_reduce_add_rmsnorm_flags  # signature set by the binding
    assert f(*args, None, 1, 1) == INVALID                    # no flag array
    assert f(*args, BASE + 2, 1, 1) == ALIGN                  # misaligned flags
    assert f(*args, BASE + 128 * MB, 0, 1) == INVALID         # block_tokens 0


GB = 1 << 30


def noalloc(lib, H, dtype, n_parts, n_out, T, chunk_tokens, t0=0, t1=None):
    """Call the no-allocation host entry point with fake, non-overlapping
    addresses 1 GiB apart (every buffer here is smaller)."""
    t1 = T if t1 is None else t1
    p_arr = (ctypes.c_void_p * n_parts)(*[BASE + i * GB for i in range(n_parts)])
    o_arr = (ctypes.c_void_p * n_out)(*[BASE + (20 + k) * GB for k in range(n_out)])
    return lib.tw_fused_reduce_add_rmsnorm_host_noalloc(
        p_arr, n_parts, BASE + 30 * GB, BASE + 31 * GB, o_arr, n_out, BASE + 32 * GB,
        T, H, 1e-6, t0, t1, 8, chunk_tokens, None, dtype)


# Rows of 8 to 16 KB, including rows whose staging size is not a whole number
# of 256-byte units (H = 136, 152, 200 bf16), and rows of at most 128 bytes,
# where one more token can leave the rounded staging size unchanged.
NOALLOC_SHAPES = [(8, 0, 8, 2, 5000), (64, 0, 8, 2, 300), (136, 0, 8, 2, 7000),
                  (152, 0, 1, 1, 20000), (200, 0, 8, 1, 1000), (8192, 0, 8, 2, 70),
                  (4, 1, 4, 4, 100), (32, 1, 2, 1, 40000), (5120, 1, 4, 4, 8192)]


@pytest.mark.parametrize("H,dtype,n_parts,n_out,T", NOALLOC_SHAPES)
def test_noalloc_default_chunk_is_never_refused(lib, H, dtype, n_parts, n_out, T):
    # chunk_tokens = 0 must size a chunk that fits the array: the call gets
    # past the sizing to its first CUDA call (no device here: TW_ERR_CUDA; on
    # a GPU machine the fake addresses are refused as not page-locked).
    rc = noalloc(lib, H, dtype, n_parts, n_out, T, 0)
    assert rc in (CUDA, INVALID), (rc, tw.tw_last_error_string())
    assert "staging" not in tw.tw_last_error_string()


@pytest.mark.parametrize("H,dtype,n_parts,n_out,T", NOALLOC_SHAPES)
def test_noalloc_default_chunk_is_the_largest_that_fits(lib, H, dtype, n_parts, n_out, T):
    # Closed form of the largest chunk: the workspace is the weight row plus
    # 2 * (n_parts + n_out + 2) chunk buffers, each rounded up to 256 bytes,
    # so k tokens fit 16 MiB iff k * row <= the per-buffer share rounded down
    # to 256 bytes.
    limit = 16 << 20
    row = H * (2 if dtype == 0 else 4)
    weight = -(-row // 256) * 256
    share = (limit - weight) // (2 * (n_parts + n_out + 2)) // 256 * 256
    k = min(T, share // row)
    tdt = torch_bf16() if dtype == 0 else torch_f32()
    assert tw.tw_host_workspace_bytes(n_parts, n_out, H, k, tdt) <= limit
    if k < T:
        assert tw.tw_host_workspace_bytes(n_parts, n_out, H, k + 1, tdt) > limit
    # An explicit chunk of exactly k tokens is accepted, k + 1 refused.
    assert noalloc(lib, H, dtype, n_parts, n_out, T, k) in (CUDA, INVALID)
    assert "staging" not in tw.tw_last_error_string()
    if k < T:
        assert noalloc(lib, H, dtype, n_parts, n_out, T, k + 1) == UNSUP
        assert "staging" in tw.tw_last_error_string()


def test_noalloc_huge_and_oversized_chunks(lib):
    # A chunk longer than the range is cut to the range: fits, no overflow.
    assert noalloc(lib, 8192, 0, 8, 2, 4, 1 << 50) in (CUDA, INVALID)
    assert noalloc(lib, 8192, 0, 8, 2, 4, (1 << 63) - 1) in (CUDA, INVALID)
    assert "staging" not in tw.tw_last_error_string()
    # 4096-token chunks of 16 KB rows need far more than 16 MiB.
    assert noalloc(lib, 8192, 0, 8, 1, 8192, 4096) == UNSUP
    # Argument rules come first; an empty range is a no-op with no CUDA call.
    assert noalloc(lib, 8192, 0, 0, 1, 8, 0) == INVALID
    assert noalloc(lib, 12, 0, 2, 1, 8, 0) == ALIGN
    assert noalloc(lib, 8192, 0, 8, 1, 8, 0, t0=3, t1=3) == OK


def test_workspace_query_refuses_overflowing_chunks(lib):
    import ctypes as c
    out = c.c_size_t()
    assert lib.tw_host_workspace_bytes(8, 1, 8192, 1 << 50, 0, c.byref(out)) == INVALID
    assert lib.tw_host_workspace_bytes(8, 1, 8192, (1 << 63) - 1, 0, c.byref(out)) == INVALID
    assert lib.tw_host_workspace_bytes(8, 1, 8192, 1 << 20, 0, c.byref(out)) == OK
    assert out.value == 2 * 11 * (1 << 20) * 16384 + 16384
    # The host entry point cuts a huge chunk to its range before sizing the
    # workspace (on a machine without a GPU the call then fails at its first
    # CUDA call; with one, at the page-locked check of the fake addresses).
    p_arr = (ctypes.c_void_p * 2)(BASE, BASE + GB)
    o_arr = (ctypes.c_void_p * 1)(BASE + 20 * GB)
    args = [p_arr, 2, BASE + 30 * GB, BASE + 31 * GB, o_arr, 1, BASE + 32 * GB, 4, 8192, 1e-6]
    need4 = tw.tw_host_workspace_bytes(2, 1, 8192, 4, torch_bf16())
    f = lib.tw_fused_reduce_add_rmsnorm_host
    assert f(*args, 0, 4, 8, BASE + 40 * GB, need4, 1 << 50, None, 0) in (CUDA, INVALID)
    assert "workspace" not in tw.tw_last_error_string()
    assert f(*args, 0, 4, 8, BASE + 40 * GB, need4 - 256, 1 << 50, None, 0) == INVALID
    assert "workspace" in tw.tw_last_error_string()


def torch_f32():
    import torch
    return torch.float32


def test_set_ready_argument_checks(lib):
    f = lib.tw_set_ready
    assert f(None, 0, 1, 1, None) == INVALID
    assert f(BASE + 2, 0, 1, 1, None) == ALIGN
    assert f(BASE, -1, 1, 1, None) == INVALID
    assert f(BASE, 0, -1, 1, None) == INVALID
    assert f(BASE, 0, 0, 1, None) == OK              # nothing to raise: no launch
