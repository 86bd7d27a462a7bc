"""Properties of the CUDA path that hold at any size: for a fixed kernel the
result does not depend on the SM budget, on how the token range is split
into launches, or on the two-stream split; and a launch with budget k runs on
at most k SMs."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from tests.parity import alloc_outputs

pytestmark = pytest.mark.gpu


def _run(wl, d, path="rows", max_sms=None, ranges=None, split=None):
    out, res_out = alloc_outputs(wl)
    if split is not None:
        s1 = torch.cuda.Stream()
        tw.tw_split_launch(d["partials"], d["residual"], d["weight"], out, res_out, wl.eps,
                           t_split=split, max_sms=max_sms, s1=s1)
    else:
        for t0, t1 in ranges or [(0, wl.T)]:
            tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out,
                                              res_out, wl.eps, t0, t1, max_sms=max_sms,
                                              path=path)
    torch.cuda.synchronize()
    return out, res_out


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a[0] + [a[1]], b[0] + [b[1]]))


@pytest.mark.parametrize("path", ["rows", "warp", "cluster"])
def test_bit_identical_across_budgets_and_splits(path):
    wl = inputs.WORKLOADS["tp8_t1024_h8192_bf16"].with_tokens(300)
    d = inputs.make_inputs(wl, device="cuda")
    ref = _run(wl, d, path)
    # The cluster kernel splits a token over min(8, budget) CTAs, so its
    # reduction order is fixed only for budgets of 8 SMs or more.
    for sms in ((8, 9, 16, 148) if path == "cluster" else (1, 3, 16, 148)):
        assert _same(ref, _run(wl, d, path, max_sms=sms)), sms
    assert _same(ref, _run(wl, d, path, ranges=[(0, 7), (7, 150), (150, 151), (151, 300)]))


def test_split_launch_equals_single_launch():
    wl = inputs.WORKLOADS["colsplit_tp4_t8192_h5120_f32_out4"].with_tokens(500)
    d = inputs.make_inputs(wl, device="cuda")
    ref = _run(wl, d, "rows")
    for t_split, sms in ((-1, None), (0, 4), (123, 2), (500, 148)):
        assert _same(ref, _run(wl, d, split=t_split, max_sms=sms)), (t_split, sms)


@pytest.mark.parametrize("path", ["rows", "warp", "cluster"])
@pytest.mark.parametrize("budget", [2, 8, 16])
def test_sm_budget_holds(path, budget):
    wl = inputs.WORKLOADS["tp8_t1024_h8192_bf16"].with_tokens(256)
    d = inputs.make_inputs(wl, device="cuda")
    out, res_out = alloc_outputs(wl)
    log = torch.full((budget,), -1, dtype=torch.int32, device="cuda")
    tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out, res_out,
                                      wl.eps, max_sms=budget, path=path, smid_log=log)
    torch.cuda.synchronize()
    ids = log.cpu().tolist()
    assert all(i >= 0 for i in ids), ids          # every CTA launched and logged
    assert len(ids) == budget                      # grid == budget (tokens >> budget)
    # Each CTA asks for more than half an SM's shared memory, so no two CTAs
    # of the launch share an SM: exactly `budget` distinct SMs.
    assert len(set(ids)) == budget
