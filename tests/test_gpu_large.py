"""Maximum sizes: input rows that sit beyond 4 GB from the start of their
buffer (N = 2, T = 300 000, H = 8192 bf16: 4.9 GB per tensor, ~25 GB in all).
Every kernel is run on tokens whose byte offsets need more than 32 bits and
checked against the oracle on sampled tokens; rows next to a sub-range must
keep their sentinel."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import SENTINEL, alloc_outputs, check_sampled, sample_tokens

pytestmark = pytest.mark.gpu

WL = Workload("large_tp2_t300000_h8192_bf16", 2, 300_000, 8192, "bf16", 1e-6, 1, 61)
FIRST_FAR = (1 << 32) // (WL.H * 2)   # first token whose row starts at 4 GB


@pytest.fixture(scope="module")
def data():
    free, _ = torch.cuda.mem_get_info()
    if free < 40e9:
        pytest.skip(f"needs ~40 GB of free device memory, {free / 1e9:.0f} GB free")
    d = inputs.make_inputs(WL, device="cuda")
    out, res_out = alloc_outputs(WL)
    torch.cuda.synchronize()
    yield d, out, res_out
    del d, out, res_out
    torch.cuda.empty_cache()


def test_full_range_beyond_4gb(data):
    d, out, res_out = data
    tw.tw_fused_reduce_add_rmsnorm(d["partials"], d["residual"], d["weight"], out, res_out,
                                   WL.eps)
    torch.cuda.synchronize()
    toks = sample_tokens(WL.T, 48, seed=5,
                         must=(0, FIRST_FAR - 1, FIRST_FAR, FIRST_FAR + 1, WL.T - 1))
    check_sampled(WL, d, out, res_out, toks)
    assert tw.tw_device_status() == 0


@pytest.mark.parametrize("path,t0,t1,max_sms", [
    ("rows", 270_000, 270_600, 2),       # a small budget: many tokens per CTA
    ("warp", WL.T - 40, WL.T - 3, None),
    ("cluster", WL.T - 7, WL.T - 1, None),
])
def test_sub_ranges_beyond_4gb(data, path, t0, t1, max_sms):
    d, out, res_out = data
    for t in out + [res_out]:
        t[t0 - 1:t1 + 1].fill_(SENTINEL)
    tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out, res_out,
                                      WL.eps, t0, t1, max_sms=max_sms, path=path)
    torch.cuda.synchronize()
    picks = sample_tokens(t1 - t0, 24, seed=6, must=(0, t1 - t0 - 1))
    check_sampled(WL, d, out, res_out, [t0 + i for i in picks])
    for t in out + [res_out]:
        assert bool((t[t0 - 1].float() == SENTINEL).all()), "row before the range written"
        assert bool((t[t1].float() == SENTINEL).all()), "row after the range written"
    assert tw.tw_device_status() == 0
