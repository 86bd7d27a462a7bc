"""fp64 CPU oracle for TokenWeave's reduce + residual add + RMSNorm.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg import this module; the product path never does,
and this module imports nothing from the product package.

The arithmetic lives in ``tw_oracle.c`` (plain C, fp64); this wrapper only
marshals numpy arrays.  Inputs are widened to fp64 by the caller (bf16 and fp32
values widen exactly).

Pages followed ("TokenWeave 策略详解：以大模型推理为例"):
  * §1 背景: output = RMSNorm(residual + allreduce_output) * weight.
  * §2 核心思想 / §3.2-3.4: the reordered ReduceScatter -> residual add ->
    RMSNorm -> AllGather, split on token boundaries.
"""
import ctypes

import numpy as np

from . import build as _build


class Oracle:
    """ctypes handle on one build of the oracle's shared object."""

    def __init__(self, lib_path):
        lib = ctypes.CDLL(lib_path)
        pp = ctypes.POINTER(ctypes.c_void_p)
        sig = [pp, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, pp,
               ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
               ctypes.c_double, ctypes.c_int64, ctypes.c_int64]
        for name in ("tw_oracle_traditional", "tw_oracle_reordered"):
            fn = getattr(lib, name)
            fn.argtypes = sig
            fn.restype = ctypes.c_int
        lib.tw_oracle_token_slice.argtypes = [
            ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
        lib.tw_oracle_token_slice.restype = ctypes.c_int
        lib.tw_oracle_threads.argtypes = []
        lib.tw_oracle_threads.restype = ctypes.c_int
        lib.tw_oracle_set_threads.argtypes = [ctypes.c_int]
        lib.tw_oracle_set_threads.restype = None
        self.lib = lib
        self.path = lib_path

    def _run(self, name, partials, residual, weight, eps, n_out, t0, t1, fill):
        partials = [_f64(p) for p in partials]
        residual = _f64(residual)
        weight = _f64(weight)
        if residual.ndim != 2:
            raise ValueError("residual must be [T, H]")
        T, H = residual.shape
        if any(p.shape != (T, H) for p in partials) or weight.shape != (H,):
            raise ValueError("partials must be [T, H] each and weight [H]")
        t1 = T if t1 is None else t1
        outs = [np.full((T, H), fill, dtype=np.float64) for _ in range(n_out)]
        res_out = np.full((T, H), fill, dtype=np.float64)
        p_arr = (ctypes.c_void_p * max(1, len(partials)))(
            *[p.ctypes.data for p in partials])
        o_arr = (ctypes.c_void_p * max(1, n_out))(*[o.ctypes.data for o in outs])
        rc = getattr(self.lib, name)(
            p_arr, len(partials), residual.ctypes.data, weight.ctypes.data,
            o_arr, n_out, res_out.ctypes.data, T, H, float(eps), t0, t1)
        if rc != 0:
            raise ValueError(f"{name}: invalid arguments")
        return outs, res_out

    def traditional(self, partials, residual, weight, eps, n_out=1, t0=0,
                    t1=None, fill=np.nan):
        """AllReduce(sum) -> residual add -> RMSNorm on every simulated rank.

        Returns ``(outs, residual_out)``: ``n_out`` fp64 [T, H] destinations
        and the fp64 residual output.  Rows outside ``[t0, t1)`` hold ``fill``.
        """
        return self._run("tw_oracle_traditional", partials, residual, weight,
                         eps, n_out, t0, t1, fill)

    def reordered(self, partials, residual, weight, eps, n_out=1, t0=0,
                  t1=None, fill=np.nan):
        """ReduceScatter (token slices) -> residual add -> RMSNorm -> AllGather.

        Same return convention as :meth:`traditional`.
        """
        return self._run("tw_oracle_reordered", partials, residual, weight,
                         eps, n_out, t0, t1, fill)

    def token_slice(self, n_tokens, n_ranks, r):
        """Token slice ``(first, last)`` that rank ``r`` of ``n_ranks`` owns."""
        a, b = ctypes.c_int64(), ctypes.c_int64()
        if self.lib.tw_oracle_token_slice(n_tokens, n_ranks, r,
                                          ctypes.byref(a), ctypes.byref(b)) != 0:
            raise ValueError("bad token_slice arguments")
        return a.value, b.value

    def threads(self):
        """Threads the oracle's token loops run on."""
        return self.lib.tw_oracle_threads()

    def set_threads(self, n):
        """Run later calls on `n` threads."""
        self.lib.tw_oracle_set_threads(int(n))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


_default = None


def default():
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def traditional(*args, **kwargs):
    return default().traditional(*args, **kwargs)


def reordered(*args, **kwargs):
    return default().reordered(*args, **kwargs)


def token_slice(n_tokens, n_ranks, r):
    return default().token_slice(n_tokens, n_ranks, r)


def threads():
    return default().threads()


def set_threads(n):
    return default().set_threads(n)
