"""The fused step beside compute ("Der intelligente Split", "Der Fused
Kernel"): results while a bf16 GEMM runs on another stream, and the two-chunk
layer step whose fused steps read the rows the GEMM writes (ordered by
events).  Every output row is compared with the oracle, fed the GEMM's actual
output."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, layer_step, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import alloc_outputs, check_chunked, check_untouched

pytestmark = pytest.mark.gpu

WL = Workload("overlap_tp8_t2048_h8192_bf16", 8, 2048, 8192, "bf16", 1e-5, 1, 61,
              partial_std=(1.0 / 8.0) ** 0.5)


def _gemm_operands(K=4096, seed=62):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(WL.T, K, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    wmat = (torch.randn(K, WL.H, generator=g, device="cuda", dtype=torch.float32) *
            (1.0 / K) ** 0.5).to(torch.bfloat16)
    return x, wmat


@pytest.mark.parametrize("budget", [8, 16])
def test_two_chunk_layer_step_matches_oracle(budget):
    d = inputs.make_inputs(WL, device="cuda")
    out, res_out = alloc_outputs(WL)
    x, wmat = _gemm_operands()
    g, f = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    g.wait_stream(torch.cuda.current_stream())
    f.wait_stream(torch.cuda.current_stream())
    layer_step.two_chunk_layer_step(x, wmat, d["partials"], d["residual"], d["weight"], out,
                                    res_out, WL.eps, budget, g, f)
    torch.cuda.synchronize()
    # Partial 0 now holds the GEMM's output, which is what the oracle reads.
    ref0 = torch.matmul(x.float(), wmat.float())
    assert torch.allclose(d["partials"][0].float(), ref0, rtol=2e-2, atol=2e-2)
    check_chunked(WL, d, out, res_out)
    assert tw.tw_device_status() == 0


def test_fused_beside_a_running_gemm_matches_oracle():
    # The fused kernel on 8 SMs on a high-priority stream while GEMMs keep the
    # rest of the GPU busy; a second range follows on the same stream.
    d = inputs.make_inputs(WL, device="cuda")
    out, res_out = alloc_outputs(WL)
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    b = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    c = torch.empty(8192, 8192, device="cuda", dtype=torch.bfloat16)
    g, f = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    g.wait_stream(torch.cuda.current_stream())
    f.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(g):
        for _ in range(4):
            torch.matmul(a, b, out=c)
    tw.tw_fused_reduce_add_rmsnorm(d["partials"], d["residual"], d["weight"], out, res_out,
                                   WL.eps, 0, 1500, max_sms=8, stream=f)
    tw.tw_fused_reduce_add_rmsnorm(d["partials"], d["residual"], d["weight"], out, res_out,
                                   WL.eps, 1500, 2000, max_sms=8, stream=f)
    torch.cuda.synchronize()
    check_chunked(WL, d, out, res_out, 0, 2000)
    check_untouched(out[0], 0, 2000, "out[0]")
    check_untouched(res_out, 0, 2000, "residual_out")
    assert tw.tw_device_status() == 0
