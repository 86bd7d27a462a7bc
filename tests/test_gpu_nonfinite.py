"""IEEE special values go through the fused step with no special case, in
the kernels' fp32 as in the oracle's fp64.  A NaN in one partial element
makes that token's x NaN there and its rms NaN, so every output of the token
is NaN and residual_out is NaN at that element only.  An infinite element
makes x infinite there and the rms infinite, so y is NaN at that element and
zero elsewhere in the row.  No other token is affected."""
import numpy as np
import pytest
import torch

import oracle
from reduce_residual_rmsnorm_tw_gb300 import inputs
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import TOL, alloc_outputs, run_gpu

pytestmark = pytest.mark.gpu

CASE = Workload("nonfinite_n3_t6_h64_bf16", 3, 6, 64, "bf16", 1e-6, 2, 71)


def same_specials_and_close(got, ref, dtype, what):
    g = inputs.to_f64(got)
    assert np.array_equal(np.isnan(g), np.isnan(ref)), f"{what}: NaN positions differ"
    assert np.array_equal(np.isposinf(g), np.isposinf(ref)), f"{what}: +inf positions differ"
    assert np.array_equal(np.isneginf(g), np.isneginf(ref)), f"{what}: -inf positions differ"
    fin = np.isfinite(ref)
    rtol, atol = TOL[dtype]
    assert np.all(np.abs(g[fin] - ref[fin]) <= np.maximum(atol, rtol * np.abs(ref[fin]))), what


@pytest.mark.parametrize("path", ["rows", "warp", "cluster"])
def test_nan_and_inf_propagate_like_the_oracle(path):
    host = inputs.make_inputs(CASE)
    host["partials"][1][2, 5] = float("nan")
    host["partials"][0][4, 10] = float("inf")
    d = {"partials": [p.cuda() for p in host["partials"]], "residual": host["residual"].cuda(),
         "weight": host["weight"].cuda()}
    out, res_out = alloc_outputs(CASE)
    run_gpu(d, CASE, out, res_out, 0, CASE.T, path=path)
    torch.cuda.synchronize()
    ref_out, ref_res = oracle.reordered([inputs.to_f64(p) for p in host["partials"]],
                                        inputs.to_f64(host["residual"]),
                                        inputs.to_f64(host["weight"]), CASE.eps,
                                        n_out=CASE.n_out)
    # The pattern the pages' arithmetic implies, checked on the oracle first.
    assert np.isnan(ref_out[0][2]).all() and np.isnan(ref_res[2, 5])
    assert np.isnan(ref_out[0][4, 10]) and np.isposinf(ref_res[4, 10])
    assert (ref_out[0][4, np.arange(CASE.H) != 10] == 0).all()
    assert np.isfinite(np.delete(ref_out[0], [2, 4], axis=0)).all()
    for k in range(CASE.n_out):
        same_specials_and_close(out[k], ref_out[k], CASE.dtype, f"{path} out[{k}]")
    same_specials_and_close(res_out, ref_res, CASE.dtype, f"{path} residual_out")
