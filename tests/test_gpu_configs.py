"""The five benchmark workloads at full size, in the launch configuration the
benchmark times, against the oracle element by element on every row: the
N=2 and N=8 x 1024-token cases and the decode sweep from host-drawn inputs;
the 16384-token split and the fp32 column-split case from device-drawn
inputs, compared in chunks of 1024 tokens (the oracle recomputes each chunk
from the device inputs copied to the host), plus sampled rows at the chunk
and split boundaries as an extra check."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from tests.parity import (alloc_outputs, check_chunked, check_sampled, check_workload,
                          sample_tokens)

pytestmark = pytest.mark.gpu
W = inputs.WORKLOADS


def test_tp2_t2048_h4096_bf16_full():
    check_workload(W["tp2_t2048_h4096_bf16"])


def test_tp8_t1024_h8192_bf16_full():
    check_workload(W["tp8_t1024_h8192_bf16"])


@pytest.mark.parametrize("max_sms", [2, 8, 148])
def test_tp8_t1024_h8192_bf16_sm_budgets(max_sms):
    check_workload(W["tp8_t1024_h8192_bf16"], max_sms=max_sms)


@pytest.mark.parametrize("T", inputs.DECODE_TOKENS)
@pytest.mark.parametrize("path", ["warp", "cluster", "rows", "auto"])
def test_decode_sweep_full(T, path):
    check_workload(W["decode_tp8_h8192_bf16"].with_tokens(T), path=path)


@pytest.mark.parametrize("max_sms", [2, 8, 148])
def test_split_t16384_every_row(max_sms):
    wl = W["split_tp8_t16384_h8192_bf16"]
    d = inputs.make_inputs(wl, device="cuda")
    out, res_out = alloc_outputs(wl)
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    # Side streams are non-blocking: order s0 after the input draw and the
    # sentinel fill on the current stream (the library orders s1 after s0).
    s0.wait_stream(torch.cuda.current_stream())
    tw.tw_split_launch(d["partials"], d["residual"], d["weight"], out, res_out, wl.eps,
                       t_split=-1, max_sms=max_sms, s0=s0, s1=s1)
    s0.synchronize()
    check_chunked(wl, d, out, res_out)
    toks = sample_tokens(wl.T, 32, seed=3, must=(0, 1, 8191, 8192, 8193, wl.T - 1))
    check_sampled(wl, d, out, res_out, toks)


@pytest.mark.parametrize("colsplit", [False, True])
def test_colsplit_t8192_h5120_f32_every_row(colsplit):
    wl = W["colsplit_tp4_t8192_h5120_f32_out4"]
    d = inputs.make_inputs(wl, device="cuda")
    out, res_out = alloc_outputs(wl)
    fn = (tw.tw_fused_reduce_add_rmsnorm_colsplit if colsplit
          else tw.tw_fused_reduce_add_rmsnorm)
    fn(d["partials"], d["residual"], d["weight"], out, res_out, wl.eps)
    torch.cuda.synchronize()
    check_chunked(wl, d, out, res_out)
    toks = sample_tokens(wl.T, 32, seed=4, must=(0, 1023, 1024, wl.T - 1))
    check_sampled(wl, d, out, res_out, toks)
