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


LIVE = Workload("flags_live_tp8_t512_h8192_bf16", 8, 512, 8192, "bf16", 1e-5, 1, 33)


@pytest.mark.parametrize("block_tokens", [16, 64])
def test_flags_live_producer(block_tokens):
    """A producer on a second stream writes the partial and residual rows of
    one token block at a time (copies), raises the block's flag with
    tw_set_ready (release stores after those copies), then pauses before the
    next block; the consumer, held to 8 SMs, was launched first and reads each
    block only once its flag is up.  The rows it reads hold NaN until the
    producer writes them, so a read before the flag would show."""
    tw.tw_device_status(clear=True)
    host = inputs.make_inputs(LIVE)
    src = [p.cuda() for p in host["partials"]] + [host["residual"].cuda()]
    weight = host["weight"].cuda()
    dst = [torch.full_like(t, float("nan")) for t in src]
    n_blocks = -(-LIVE.T // block_tokens)
    epoch = 5
    ready = torch.full((n_blocks,), epoch - 1, dtype=torch.int32, device="cuda")
    out, res_out = alloc_outputs(LIVE)
    consumer, producer = torch.cuda.Stream(), torch.cuda.Stream()
    # Every kernel the producer uses runs once before the consumer starts
    # waiting: a kernel's first launch may load it, and a load can wait for
    # the running consumer (lazy module loading).
    with torch.cuda.stream(producer):
        torch.cuda._sleep(10)
        dst[0][:1].copy_(src[0][:1])
        tw.tw_set_ready(ready, epoch - 1, first_block=0, n_blocks=1, stream=producer)
    torch.cuda.synchronize()
    consumer.wait_stream(torch.cuda.current_stream())
    producer.wait_stream(torch.cuda.current_stream())
    ev = {k: torch.cuda.Event(enable_timing=True)
          for k in ("launch", "done", "first_flag", "late_flag")}
    ev["launch"].record(consumer)
    tw.tw_fused_reduce_add_rmsnorm_flags(dst[:-1], dst[-1], weight, out, res_out, LIVE.eps,
                                         ready, block_tokens, epoch, max_sms=8,
                                         stream=consumer)
    ev["done"].record(consumer)
    with torch.cuda.stream(producer):
        torch.cuda._sleep(200_000)          # the consumer is waiting before the first flag
        for b in range(n_blocks):
            rows = slice(b * block_tokens, min((b + 1) * block_tokens, LIVE.T))
            for d_t, s_t in zip(dst, src):
                d_t[rows].copy_(s_t[rows])
            tw.tw_set_ready(ready, epoch, first_block=b, n_blocks=1, stream=producer)
            if b == 0:
                ev["first_flag"].record(producer)
            if b == n_blocks - 2:
                ev["late_flag"].record(producer)
            if b + 1 < n_blocks:
                torch.cuda._sleep(20_000)   # a gap before the next block
    torch.cuda.synchronize()
    assert tw.tw_device_status() == 0
    # The consumer's stream reached its launch before the first flag rose, and
    # the consumer finished after the last block but one was raised (the last
    # block follows a gap of 20 000 cycles and its copies).
    assert ev["launch"].elapsed_time(ev["first_flag"]) > 0
    assert ev["late_flag"].elapsed_time(ev["done"]) > 0
    # Bit-identical to the rows path on the same inputs (itself checked
    # against the oracle here).
    ref_out, ref_res = check_workload(LIVE, path="rows")
    torch.cuda.synchronize()
    for a, b in zip(out + [res_out], ref_out + [ref_res]):
        assert torch.equal(a, b)
