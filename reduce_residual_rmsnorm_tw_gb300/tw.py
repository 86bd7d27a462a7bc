"""Thin ctypes binding of libtw.so (argument marshalling only).

Every function keeps the name of the C entry point it calls.  Tensors are
torch tensors used only as device memory: the binding reads their pointers,
shapes and dtypes, the library checks the rules of ``include/tw.h`` and runs
every step of the computation in its CUDA kernels.  There is no fallback: if
``libtw.so`` is missing the first call raises.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtw.so")

TW_BF16, TW_F32 = 0, 1
PATHS = {"auto": 0, "rows": 1, "warp": 2, "cluster": 3}
MAX_PARTS, MAX_OUTS = 16, 8
STATUS_NAMES = {0: "TW_OK", -1: "TW_ERR_INVALID_ARG", -2: "TW_ERR_ALIGNMENT",
                -3: "TW_ERR_ALIAS", -4: "TW_ERR_CUDA", -5: "TW_ERR_UNSUPPORTED"}
_DTYPES = {torch.bfloat16: TW_BF16, torch.float32: TW_F32}
_ALL_SMS = 1 << 30  # clamped to the device's SM count by the library


class TwError(RuntimeError):
    """A libtw.so call returned a status other than TW_OK."""

    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load():
    """Load libtw.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    pp = ctypes.POINTER(ctypes.c_void_p)
    common = [pp, ctypes.c_int, vp, vp, pp, ctypes.c_int, vp, i64, i64,
              ctypes.c_float, i64, i64, ctypes.c_int, vp]
    for name, extra in (("tw_fused_reduce_add_rmsnorm_bf16", []),
                        ("tw_fused_reduce_add_rmsnorm_f32", []),
                        ("tw_fused_reduce_add_rmsnorm", [ctypes.c_int]),
                        ("tw_fused_reduce_add_rmsnorm_colsplit", [ctypes.c_int]),
                        ("tw_fused_reduce_add_rmsnorm_ex",
                         [ctypes.c_int, ctypes.c_int, vp])):
        fn = getattr(lib, name)
        fn.argtypes = common + extra
        fn.restype = ctypes.c_int
    lib.tw_fused_reduce_add_rmsnorm_flags.argtypes = common + [
        ctypes.c_int, vp, i64, ctypes.c_uint32]
    lib.tw_fused_reduce_add_rmsnorm_flags.restype = ctypes.c_int
    lib.tw_set_ready.argtypes = [vp, i64, i64, ctypes.c_uint32, vp]
    lib.tw_set_ready.restype = ctypes.c_int
    lib.tw_split_launch.argtypes = [pp, ctypes.c_int, vp, vp, pp, ctypes.c_int,
                                    vp, i64, i64, ctypes.c_float, i64,
                                    ctypes.c_int, vp, vp, ctypes.c_int]
    lib.tw_split_launch.restype = ctypes.c_int
    lib.tw_fused_reduce_add_rmsnorm_host.argtypes = [
        pp, ctypes.c_int, vp, vp, pp, ctypes.c_int, vp, i64, i64, ctypes.c_float,
        i64, i64, ctypes.c_int, vp, ctypes.c_size_t, i64, vp, ctypes.c_int]
    lib.tw_fused_reduce_add_rmsnorm_host.restype = ctypes.c_int
    lib.tw_fused_reduce_add_rmsnorm_host_noalloc.argtypes = [
        pp, ctypes.c_int, vp, vp, pp, ctypes.c_int, vp, i64, i64, ctypes.c_float,
        i64, i64, ctypes.c_int, i64, vp, ctypes.c_int]
    lib.tw_fused_reduce_add_rmsnorm_host_noalloc.restype = ctypes.c_int
    lib.tw_host_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64,
                                            ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    lib.tw_host_workspace_bytes.restype = ctypes.c_int
    lib.tw_device_status.argtypes = [ctypes.c_int]
    lib.tw_device_status.restype = ctypes.c_int
    lib.tw_last_error_string.argtypes = []
    lib.tw_last_error_string.restype = ctypes.c_char_p
    lib.tw_version.argtypes = []
    lib.tw_version.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc):
    if rc != 0:
        raise TwError(rc, load().tw_last_error_string().decode())


def _stream_handle(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _marshal(partials, residual, weight, out, residual_out, on_device=True):
    """Pointer arrays and (T, H, dtype) from tensors; shapes must agree.  The
    device entry points take tensors on the current CUDA device; the host
    entry points (on_device=False) take pinned CPU tensors."""
    partials, out = list(partials), list(out)
    if not partials or not out:
        raise ValueError("need at least one partial and one destination")
    if residual.dim() != 2:
        raise ValueError("residual must be [T, H]")
    T, H = residual.shape
    dtype = residual.dtype
    if dtype not in _DTYPES:
        raise ValueError(f"dtype {dtype} not supported (bfloat16 or float32)")
    for name, ts in (("partials", partials), ("out", out),
                     ("residual_out", [residual_out])):
        for t in ts:
            if t.shape != (T, H) or t.dtype != dtype or not t.is_contiguous():
                raise ValueError(f"{name}: every tensor must be a contiguous "
                                 f"[{T}, {H}] {dtype} tensor")
    if (weight.shape != (H,) or weight.dtype != dtype
            or not weight.is_contiguous()):
        raise ValueError(f"weight must be a contiguous [{H}] {dtype} tensor")
    every = partials + out + [residual, weight, residual_out]
    if on_device:
        if any(not t.is_cuda for t in every):
            raise ValueError("every tensor must be on the current CUDA device")
        dev = torch.cuda.current_device()
        if any(t.device.index != dev for t in every):
            raise ValueError(f"every tensor must be on the current CUDA device (cuda:{dev})")
    elif any(t.is_cuda or not t.is_pinned() for t in every):
        raise ValueError("every tensor must be a pinned (page-locked) CPU tensor")
    p_arr = (ctypes.c_void_p * len(partials))(*[t.data_ptr() for t in partials])
    o_arr = (ctypes.c_void_p * len(out))(*[t.data_ptr() for t in out])
    return p_arr, len(partials), o_arr, len(out), T, H, _DTYPES[dtype]


def tw_fused_reduce_add_rmsnorm_ex(partials, residual, weight, out,
                                   residual_out, eps, t0=0, t1=None,
                                   max_sms=None, stream=None, path="auto",
                                   smid_log=None):
    """Fused reduce + residual add + RMSNorm on rows [t0, t1), kernel chosen
    by ``path`` ("auto", "rows", "warp" or "cluster").  ``smid_log`` is an optional int32
    device tensor with at least max_sms entries."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out)
    rc = load().tw_fused_reduce_add_rmsnorm_ex(
        p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
        residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
        _ALL_SMS if max_sms is None else max_sms, _stream_handle(stream), dt,
        PATHS[path], None if smid_log is None else smid_log.data_ptr())
    _check(rc)


def tw_fused_reduce_add_rmsnorm(partials, residual, weight, out, residual_out,
                                eps, t0=0, t1=None, max_sms=None, stream=None):
    """Fused reduce + residual add + RMSNorm on rows [t0, t1) (kernel chosen
    by the library)."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out)
    rc = load().tw_fused_reduce_add_rmsnorm(
        p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
        residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
        _ALL_SMS if max_sms is None else max_sms, _stream_handle(stream), dt)
    _check(rc)


def tw_fused_reduce_add_rmsnorm_colsplit(partials, residual, weight, out,
                                         residual_out, eps, t0=0, t1=None,
                                         max_sms=None, stream=None):
    """The fused step for zero-padded column-split partials: partial r is
    nonzero only in columns [r*H//N, (r+1)*H//N), and only those are read."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out)
    rc = load().tw_fused_reduce_add_rmsnorm_colsplit(
        p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
        residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
        _ALL_SMS if max_sms is None else max_sms, _stream_handle(stream), dt)
    _check(rc)


def tw_fused_reduce_add_rmsnorm_flags(partials, residual, weight, out,
                                      residual_out, eps, ready, block_tokens,
                                      epoch, t0=0, t1=None, max_sms=None,
                                      stream=None):
    """The fused step gated by readiness flags: token t is read only once
    ``ready[t // block_tokens]`` (an int32 CUDA tensor) has reached ``epoch``."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out)
    if ready.dtype != torch.int32 or not ready.is_cuda:
        raise ValueError("ready must be an int32 CUDA tensor")
    rc = load().tw_fused_reduce_add_rmsnorm_flags(
        p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
        residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
        _ALL_SMS if max_sms is None else max_sms, _stream_handle(stream), dt,
        ready.data_ptr(), block_tokens, epoch & 0xFFFFFFFF)
    _check(rc)


def tw_set_ready(ready, epoch, first_block=0, n_blocks=None, stream=None):
    """Raise ``ready[first_block:first_block + n_blocks]`` (an int32 CUDA
    tensor) to ``epoch`` with release stores, after the work queued earlier
    on ``stream``: the producer side of tw_fused_reduce_add_rmsnorm_flags."""
    if ready.dtype != torch.int32 or not ready.is_cuda or not ready.is_contiguous():
        raise ValueError("ready must be a contiguous int32 CUDA tensor")
    if n_blocks is None:
        n_blocks = ready.numel() - first_block
    if first_block < 0 or n_blocks < 0 or first_block + n_blocks > ready.numel():
        raise ValueError("flag range outside the ready tensor")
    _check(load().tw_set_ready(ready.data_ptr(), first_block, n_blocks, epoch & 0xFFFFFFFF,
                               _stream_handle(stream)))


def _typed(name, dtype):
    def call(partials, residual, weight, out, residual_out, eps, t0=0, t1=None,
             max_sms=None, stream=None):
        if residual.dtype != dtype:
            raise ValueError(f"{name} takes {dtype} tensors")
        p_arr, n, o_arr, n_out, T, H, _ = _marshal(partials, residual, weight,
                                                   out, residual_out)
        rc = getattr(load(), name)(
            p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
            residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
            _ALL_SMS if max_sms is None else max_sms, _stream_handle(stream))
        _check(rc)
    call.__name__ = name
    call.__doc__ = f"The fused step on {dtype} tensors (C entry point {name})."
    return call


tw_fused_reduce_add_rmsnorm_bf16 = _typed("tw_fused_reduce_add_rmsnorm_bf16",
                                          torch.bfloat16)
tw_fused_reduce_add_rmsnorm_f32 = _typed("tw_fused_reduce_add_rmsnorm_f32",
                                         torch.float32)


def tw_split_launch(partials, residual, weight, out, residual_out, eps,
                    t_split=-1, max_sms=None, s0=None, s1=None):
    """Two-chunk token split: rows [0, t_split) on s0, [t_split, T) on s1.
    Synchronising s0 covers both chunks."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out)
    if s1 is None:
        raise ValueError("tw_split_launch needs a second stream s1")
    rc = load().tw_split_launch(
        p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
        residual_out.data_ptr(), T, H, eps, t_split,
        _ALL_SMS if max_sms is None else max_sms, _stream_handle(s0),
        _stream_handle(s1), dt)
    _check(rc)


def tw_host_workspace_bytes(n_parts, n_out, H, chunk_tokens, dtype):
    """Device workspace bytes of tw_fused_reduce_add_rmsnorm_host."""
    out = ctypes.c_size_t()
    _check(load().tw_host_workspace_bytes(n_parts, n_out, H, chunk_tokens,
                                          _DTYPES[dtype], ctypes.byref(out)))
    return out.value


def tw_fused_reduce_add_rmsnorm_host(partials, residual, weight, out,
                                     residual_out, eps, workspace, chunk_tokens,
                                     t0=0, t1=None, max_sms=None, stream=None):
    """The fused step on pinned HOST tensors.  ``chunk_tokens`` >= 1: pipelined
    in chunks of that many tokens through the device ``workspace`` (a uint8
    CUDA tensor of at least tw_host_workspace_bytes bytes).  ``chunk_tokens``
    == 0: one kernel reads the host tensors in place (``workspace`` may be
    None)."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out, on_device=False)
    if workspace is not None and not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    rc = load().tw_fused_reduce_add_rmsnorm_host(
        p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
        residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
        _ALL_SMS if max_sms is None else max_sms,
        None if workspace is None else workspace.data_ptr(),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        chunk_tokens, _stream_handle(stream), dt)
    _check(rc)


def tw_fused_reduce_add_rmsnorm_host_noalloc(partials, residual, weight, out,
                                             residual_out, eps, chunk_tokens=0,
                                             t0=0, t1=None, max_sms=None,
                                             stream=None):
    """The host-buffer step for callers that cannot allocate device memory:
    pinned host tensors only; the library stages the chunks in its own
    fixed device array (chunk_tokens <= 0: the largest chunk that fits)."""
    p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                out, residual_out, on_device=False)
    rc = load().tw_fused_reduce_add_rmsnorm_host_noalloc(p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr, n_out,
            residual_out.data_ptr(), T, H, eps, t0, T if t1 is None else t1,
            _ALL_SMS if max_sms is None else max_sms, chunk_tokens,
            _stream_handle(stream), dt)
    _check(rc)


def tw_device_status(clear=False):
    """Device status word: nonzero if a kernel gave up on a bounded wait."""
    rc = load().tw_device_status(1 if clear else 0)
    if rc < 0:
        raise TwError(-4, load().tw_last_error_string().decode())
    return rc


def tw_last_error_string():
    return load().tw_last_error_string().decode()


def tw_version():
    return load().tw_version()


class Prepared:
    """A tw_fused_reduce_add_rmsnorm_ex call with its arguments marshalled
    once, for launch loops where per-call Python work would outlast the
    kernel.  The tensors must stay alive and unchanged in shape."""

    def __init__(self, partials, residual, weight, out, residual_out, eps, t0=0,
                 t1=None, max_sms=None, path="auto", ready=None, block_tokens=0, epoch=0):
        p_arr, n, o_arr, n_out, T, H, dt = _marshal(partials, residual, weight,
                                                    out, residual_out)
        self._keep = (p_arr, o_arr, list(partials), residual, weight, list(out),
                      residual_out)
        self._args = [p_arr, n, residual.data_ptr(), weight.data_ptr(), o_arr,
                      n_out, residual_out.data_ptr(), T, H, eps, t0,
                      T if t1 is None else t1,
                      _ALL_SMS if max_sms is None else max_sms]
        if ready is not None:
            # tw_fused_reduce_add_rmsnorm_flags: gated by readiness flags.
            if ready.dtype != torch.int32 or not ready.is_cuda:
                raise ValueError("ready must be an int32 CUDA tensor")
            self._keep += (ready,)
            self._fn = load().tw_fused_reduce_add_rmsnorm_flags
            self._tail = [dt, ready.data_ptr(), block_tokens, epoch & 0xFFFFFFFF]
        elif path == "colsplit":
            # tw_fused_reduce_add_rmsnorm_colsplit: zero-padded column split.
            self._fn = load().tw_fused_reduce_add_rmsnorm_colsplit
            self._tail = [dt]
        else:
            self._fn = load().tw_fused_reduce_add_rmsnorm_ex
            self._tail = [dt, PATHS[path], None]

    def __call__(self, stream_handle):
        """Launch on the raw cudaStream_t handle (an int)."""
        rc = self._fn(*self._args, stream_handle, *self._tail)
        if rc != 0:
            _check(rc)


def prepare(partials, residual, weight, out, residual_out, eps, t0=0, t1=None,
            max_sms=None, path="auto", ready=None, block_tokens=0, epoch=0):
    """Marshal a fused call once; returns a :class:`Prepared` callable.
    ``path`` is a kernel name of tw_fused_reduce_add_rmsnorm_ex, or "colsplit"
    for tw_fused_reduce_add_rmsnorm_colsplit; with ``ready`` the call is
    tw_fused_reduce_add_rmsnorm_flags."""
    return Prepared(partials, residual, weight, out, residual_out, eps, t0, t1,
                    max_sms, path, ready, block_tokens, epoch)
