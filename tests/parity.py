"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it element by element with the fp64 oracle on the same seeded inputs.

Tolerances (an element passes if |gpu - ref| <= max(atol, rtol * |ref|)):
  bf16: rtol 8e-3, atol 1e-2;   fp32: rtol 1e-5, atol 1e-5.
They apply to every gather destination and to residual_out; the
destinations must also be bit-identical to one another, and rows outside
[t0, t1) must keep their sentinel bytes.
"""
import numpy as np
import torch

import oracle
from reduce_residual_rmsnorm_tw_gb300 import inputs, tw

TOL = {"bf16": (8e-3, 1e-2), "f32": (1e-5, 1e-5)}
SENTINEL = -12288.0  # exact in bf16 and fp32; never a plausible output


def check_close(got, ref, dtype, what):
    """Element-wise tolerance check of a device tensor against fp64 values."""
    rtol, atol = TOL[dtype]
    g = inputs.to_f64(got)
    err = np.abs(g - ref)
    bound = np.maximum(atol, rtol * np.abs(ref))
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        worst = np.unravel_index(np.nanargmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside tolerance; first {i}: "
            f"gpu {g[i]!r} ref {ref[i]!r}; worst {worst}: gpu {g[worst]!r} ref {ref[worst]!r}")


def alloc_outputs(wl, device="cuda"):
    out = [torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype, device=device)
           for _ in range(wl.n_out)]
    res_out = torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype, device=device)
    return out, res_out


def check_untouched(t, t0, t1, what):
    outside = torch.cat([t[:t0], t[t1:]]).float()
    assert bool((outside == SENTINEL).all()), f"{what}: rows outside [{t0}, {t1}) written"


def run_gpu(d, wl, out, res_out, t0, t1, path="auto", max_sms=None, split=None,
            stream=None, colsplit=False):
    if colsplit:
        tw.tw_fused_reduce_add_rmsnorm_colsplit(d["partials"], d["residual"], d["weight"], out,
                                                res_out, wl.eps, t0, t1, max_sms=max_sms,
                                                stream=stream)
    elif split is None:
        tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out,
                                          res_out, wl.eps, t0, t1, max_sms=max_sms,
                                          path=path, stream=stream)
    else:
        s1 = torch.cuda.Stream()
        tw.tw_split_launch(d["partials"], d["residual"], d["weight"], out, res_out,
                           wl.eps, t_split=split, max_sms=max_sms, s0=stream, s1=s1)


def check_workload(wl, path="auto", t0=0, t1=None, in_place=False, max_sms=None,
                   split=None, order="reordered", colsplit=False):
    """Full element-wise parity of one workload (inputs drawn on the CPU)."""
    t1 = wl.T if t1 is None else t1
    host = inputs.make_inputs(wl, device="cpu")
    d = {"partials": [p.cuda() for p in host["partials"]],
         "residual": host["residual"].cuda(), "weight": host["weight"].cuda()}
    out, res_out = alloc_outputs(wl)
    if in_place:
        res_out = d["residual"]  # residual_out == residual
    run_gpu(d, wl, out, res_out, t0, t1, path=path, max_sms=max_sms, split=split,
            colsplit=colsplit)
    torch.cuda.synchronize()

    fn = oracle.reordered if order == "reordered" else oracle.traditional
    ref_out, ref_res = fn([inputs.to_f64(p) for p in host["partials"]],
                          inputs.to_f64(host["residual"]), inputs.to_f64(host["weight"]),
                          wl.eps, n_out=wl.n_out, t0=t0, t1=t1)
    for k in range(wl.n_out):
        check_close(out[k][t0:t1], ref_out[k][t0:t1], wl.dtype, f"{wl.name} out[{k}]")
        assert torch.equal(out[k], out[0]), f"{wl.name}: out[{k}] differs from out[0]"
        check_untouched(out[k], t0, t1, f"{wl.name} out[{k}]")
    check_close(res_out[t0:t1], ref_res[t0:t1], wl.dtype, f"{wl.name} residual_out")
    if in_place:
        # Rows outside the range keep the input residual.
        keep = torch.cat([res_out[:t0], res_out[t1:]])
        want = torch.cat([host["residual"][:t0], host["residual"][t1:]]).cuda()
        assert torch.equal(keep, want)
    else:
        check_untouched(res_out, t0, t1, f"{wl.name} residual_out")
    return out, res_out


def check_sampled(wl, d, out, res_out, tokens):
    """Parity on sampled tokens of a full-size run: the oracle recomputes only
    the sampled rows (gathered from the device inputs)."""
    idx = torch.as_tensor(sorted(set(int(t) for t in tokens)), device="cuda")
    parts = [inputs.to_f64(p.index_select(0, idx)) for p in d["partials"]]
    ref_out, ref_res = oracle.reordered(parts, inputs.to_f64(d["residual"].index_select(0, idx)),
                                        inputs.to_f64(d["weight"]), wl.eps, n_out=wl.n_out)
    for k in range(wl.n_out):
        check_close(out[k].index_select(0, idx), ref_out[k], wl.dtype,
                    f"{wl.name} out[{k}] sampled")
    check_close(res_out.index_select(0, idx), ref_res, wl.dtype,
                f"{wl.name} residual_out sampled")


def sample_tokens(T, n, seed, must=()):
    rng = np.random.default_rng(seed)
    picks = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    picks.update(t for t in must if 0 <= t < T)
    return sorted(picks)


def check_chunked(wl, d, out, res_out, t0=0, t1=None, chunk=1024):
    """Element-wise parity of a full-size run on EVERY row of [t0, t1): the
    inputs (drawn on the device) are copied to the host `chunk` tokens at a
    time and the oracle computes each chunk, so host memory stays small.
    Destinations must also be bit-identical to out[0]."""
    t1 = wl.T if t1 is None else t1
    w = inputs.to_f64(d["weight"])
    for c0 in range(t0, t1, chunk):
        c1 = min(c0 + chunk, t1)
        parts = [inputs.to_f64(p[c0:c1]) for p in d["partials"]]
        ref_out, ref_res = oracle.reordered(parts, inputs.to_f64(d["residual"][c0:c1]), w,
                                            wl.eps, n_out=wl.n_out)
        del parts
        for k in range(wl.n_out):
            check_close(out[k][c0:c1], ref_out[k], wl.dtype, f"{wl.name} out[{k}] rows {c0}-{c1}")
            if k:
                assert torch.equal(out[k][c0:c1], out[0][c0:c1]), \
                    f"{wl.name}: out[{k}] differs from out[0] in rows {c0}-{c1}"
        check_close(res_out[c0:c1], ref_res, wl.dtype, f"{wl.name} residual_out rows {c0}-{c1}")

