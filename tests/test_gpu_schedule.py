"""The rows kernel's unit schedule.  A long launch on many SMs (at least 64
CTAs and 16 units per CTA) lets its CTAs claim units from a work counter of
its own (faster SMs take more); other launches, and every launch captured
into a CUDA graph, keep the fixed schedule (CTA b takes units b, b + grid,
...).  Either way every token is processed exactly once
and its result does not depend on which CTA processed it: both are checked
bit for bit against each other and against the oracle (the fixed launches
here take the two-pipeline variant, which a budget or a unit that fits half
the ring selects, while claimed units always run one pipeline, so the
comparison also holds the two variants to the same bits), with many launches
in flight at once on several streams (each needs a counter of its own) and
with more launches in a row than the library holds counters."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import alloc_outputs, check_workload

pytestmark = pytest.mark.gpu

# 3000 tokens of 16 KB rows: 19.7 units per CTA on 152 SMs, 30 on 100.
WL = Workload("sched_tp2_t3000_h8192_bf16", 2, 3000, 8192, "bf16", 1e-5, 1, 81)
# 13001 tokens of 4 KB rows: units of 2 tokens, 42.8 per CTA on 152 SMs.
SMALL = Workload("sched_tp3_t13001_h2048_bf16", 3, 13001, 2048, "bf16", 1e-6, 2, 82)
# 8 slices of 1100 tokens, each launched on 64 SMs (17.2 units per CTA).
CONC = Workload("sched_tp2_t8800_h8192_bf16", 2, 8800, 8192, "bf16", 1e-6, 1, 83)


def _launch(w, d, out, res_out, t0, t1, sms, stream):
    tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out, res_out,
                                      w.eps, t0, t1, max_sms=sms, path="rows", stream=stream)


@pytest.mark.parametrize("w,sms", [(WL, None), (WL, 100), (WL, 5), (SMALL, None), (SMALL, 3)],
                         ids=["tp2_all", "tp2_sms100", "tp2_sms5", "tp3_all", "tp3_sms3"])
def test_claimed_units_equal_fixed_schedule_bitwise(w, sms):
    d = inputs.make_inputs(w, device="cuda")
    out_a, res_a = alloc_outputs(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    _launch(w, d, out_a, res_a, 0, w.T, sms, s)            # claimed units
    torch.cuda.synchronize()
    out_b, res_b = alloc_outputs(w)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):                     # fixed schedule
        _launch(w, d, out_b, res_b, 0, w.T, sms, torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(out_a + [res_a], out_b + [res_b]):
        assert torch.equal(a, b)
    assert tw.tw_device_status() == 0


@pytest.mark.parametrize("w,sms", [(WL, None), (SMALL, 64)], ids=["tp2_all", "tp3_sms64"])
def test_claimed_units_match_oracle(w, sms):
    check_workload(w, path="rows", max_sms=sms)
    check_workload(w, path="rows", max_sms=sms, t0=17, t1=w.T - 5)


def test_many_launches_in_flight_on_several_streams():
    # 8 streams, each running 12 launches over its own 1100-token slice on 64
    # SMs: several launches run at once, each with its own counter, 96 in all
    # (more than the library's 64 counters, so counters are handed out again).
    w = CONC
    d = inputs.make_inputs(w, device="cuda")
    ref_out, ref_res = alloc_outputs(w)
    _launch(w, d, ref_out, ref_res, 0, w.T, None, None)
    torch.cuda.synchronize()
    out, res_out = alloc_outputs(w)
    streams = [torch.cuda.Stream() for _ in range(8)]
    bounds = [w.T * i // 8 for i in range(9)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rep in range(12):
        for i, s in enumerate(streams):
            _launch(w, d, out, res_out, bounds[i], bounds[i + 1], 64, s)
    torch.cuda.synchronize()
    for a, b in zip(out + [res_out], ref_out + [ref_res]):
        assert torch.equal(a, b)
    assert tw.tw_device_status() == 0


def test_back_to_back_launches_reuse_counters():
    # 200 launches in a row on one stream (whole-GPU launches overlap their
    # start with the previous one's drain), alternating two ranges.
    w = WL
    d = inputs.make_inputs(w, device="cuda")
    ref_out, ref_res = alloc_outputs(w)
    _launch(w, d, ref_out, ref_res, 0, w.T, None, None)
    torch.cuda.synchronize()
    out, res_out = alloc_outputs(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    for rep in range(200):
        lo, hi = ((0, 2600), (2600, w.T))[rep % 2]
        _launch(w, d, out, res_out, lo, hi, None, s)
    torch.cuda.synchronize()
    for a, b in zip(out + [res_out], ref_out + [ref_res]):
        assert torch.equal(a, b)
    assert tw.tw_device_status() == 0
