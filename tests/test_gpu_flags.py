"""Readiness flags: the fused step waits (bounded) for each token block's
flag.  Flags raised before the launch give the normal result; a flag that
nothing raises makes the wait run out: the kernel returns, reports status 4,
writes no row of the blocked token, and the device stays usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import SENTINEL, alloc_outputs, check_close, check_workload

pytestmark = pytest.mark.gpu

WL = Workload("flags_tp8_t40_h8192_bf16", 8, 40, 8192, "bf16", 1e-5, 2, 31)


def _device_inputs():
    host = inputs.make_inputs(WL)
    return host, {"partials": [p.cuda() for p in host["partials"]],
                  "residual": host["residual"].cuda(), "weight": host["weight"].cuda()}


@pytest.mark.parametrize("block_tokens,epoch,value", [(1, 7, 7), (8, 7, 9), (64, 0xFFFFFFFF, 0)])
def test_flags_ready_matches_rows_path(block_tokens, epoch, value):
    host, d = _device_inputs()
    # value >= epoch as a wrap-safe signed difference (0 - 0xFFFFFFFF == 1).
    ready = torch.full((-(-WL.T // block_tokens),), value, dtype=torch.int32, device="cuda")
    out, res_out = alloc_outputs(WL)
    tw.tw_fused_reduce_add_rmsnorm_flags(d["partials"], d["residual"], d["weight"], out,
                                         res_out, WL.eps, ready, block_tokens, epoch)
    ref_out, ref_res = check_workload(WL, path="rows")
    torch.cuda.synchronize()
    for a, b in zip(out + [res_out], ref_out + [ref_res]):
        assert torch.equal(a, b)
    assert tw.tw_device_status() == 0


def test_flag_never_raised_times_out_and_reports():
    tw.tw_device_status(clear=True)
    host, d = _device_inputs()
    blocked = 13
    ready = torch.full((WL.T,), 3, dtype=torch.int32, device="cuda")
    ready[blocked] = 2                      # nothing ever raises this one to 3
    out, res_out = alloc_outputs(WL)
    torch.cuda.synchronize()
    t_start = time.monotonic()
    tw.tw_fused_reduce_add_rmsnorm_flags(d["partials"], d["residual"], d["weight"], out,
                                         res_out, WL.eps, ready, 1, 3, max_sms=4)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t_start
    assert elapsed < 10.0, elapsed           # bounded wait (about one second)
    assert tw.tw_device_status() & 4
    # The blocked token's rows are untouched; every row that was written is right.
    assert bool((res_out[blocked].float() == SENTINEL).all())
    assert bool((out[0][blocked].float() == SENTINEL).all())
    ref_out, ref_res = oracle.reordered([inputs.to_f64(p) for p in host["partials"]],
                                        inputs.to_f64(host["residual"]),
                                        inputs.to_f64(host["weight"]), WL.eps, n_out=WL.n_out)
    written = [t for t in range(WL.T) if not bool((res_out[t].float() == SENTINEL).all())]
    assert blocked not in written and len(written) >= WL.T - WL.T // 4
    idx = np.array(written)
    check_close(res_out[written], ref_res[idx], WL.dtype, "residual_out (written rows)")
    check_close(out[0][written], ref_out[0][idx], WL.dtype, "out[0] (written rows)")
    tw.tw_device_status(clear=True)
    assert tw.tw_device_status() == 0
    # The context is still usable.
    check_workload(WL, path="rows")
    assert tw.tw_device_status() == 0
