"""The host-buffer entry point: pinned host tensors, either read in place by
one kernel (chunk_tokens 0) or pipelined in chunks through a device
workspace.  Checked against the oracle element by element, and bit for bit
against the device entry point on the same kernel."""
import ctypes
from dataclasses import replace

import pytest
import torch

import oracle
from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import SENTINEL, check_close

pytestmark = pytest.mark.gpu


def workspace(wl, chunk):
    """The device workspace of a staged call (chunk >= 1); none for chunk 0,
    which reads the host tensors in place."""
    if chunk == 0:
        return None
    nbytes = tw.tw_host_workspace_bytes(wl.n_parts, wl.n_out, wl.H, chunk, wl.torch_dtype)
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda")


def host_run(wl, chunk, t0=0, t1=None, max_sms=None):
    t1 = wl.T if t1 is None else t1
    d = inputs.make_inputs(wl)
    pin = {"partials": [p.pin_memory() for p in d["partials"]],
           "residual": d["residual"].pin_memory(), "weight": d["weight"].pin_memory()}
    out = [torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype).pin_memory()
           for _ in range(wl.n_out)]
    res_out = torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype).pin_memory()
    tw.tw_fused_reduce_add_rmsnorm_host(pin["partials"], pin["residual"], pin["weight"], out,
                                        res_out, wl.eps, workspace(wl, chunk), chunk, t0, t1,
                                        max_sms=max_sms)
    torch.cuda.synchronize()
    return d, out, res_out


CASES = [
    Workload("host_tp8_t70_h8192_bf16", 8, 70, 8192, "bf16", 1e-5, 1, 21),
    Workload("host_tp4_t45_h5120_f32_out4", 4, 45, 5120, "f32", 1e-6, 4, 22,
             column_split=True),
]


@pytest.mark.parametrize("chunk,max_sms", [(1, None), (7, None), (33, None), (64, None),
                                           (1000, None), (0, None), (0, 8)])
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_host_parity(wl, chunk, max_sms):
    # chunk 0: one kernel reads the host tensors in place.
    t0, t1 = 2, wl.T - 3
    d, out, res_out = host_run(wl, chunk, t0, t1, max_sms)
    ref_out, ref_res = oracle.reordered([inputs.to_f64(p) for p in d["partials"]],
                                        inputs.to_f64(d["residual"]), inputs.to_f64(d["weight"]),
                                        wl.eps, n_out=wl.n_out, t0=t0, t1=t1)
    for k in range(wl.n_out):
        check_close(out[k][t0:t1], ref_out[k][t0:t1], wl.dtype, f"{wl.name} out[{k}]")
        assert bool((torch.cat([out[k][:t0], out[k][t1:]]).float() == SENTINEL).all())
    check_close(res_out[t0:t1], ref_res[t0:t1], wl.dtype, f"{wl.name} residual_out")
    assert bool((torch.cat([res_out[:t0], res_out[t1:]]).float() == SENTINEL).all())


def test_host_matches_device_path_bitwise():
    # The staged pipeline launches the automatic kernel choice once per chunk:
    # the same launches over the same ranges of device copies give the same
    # bits (chunks of 100 and 200 tokens, so either kernel may be chosen).
    for T, chunk in ((200, 100), (400, 200)):
        wl = CASES[0].with_tokens(T)
        d, out, res_out = host_run(wl, chunk)
        dev_out = [torch.empty(wl.T, wl.H, dtype=wl.torch_dtype, device="cuda")]
        dev_res = torch.empty(wl.T, wl.H, dtype=wl.torch_dtype, device="cuda")
        parts = [p.cuda() for p in d["partials"]]
        res, w = d["residual"].cuda(), d["weight"].cuda()
        for t0 in range(0, T, chunk):
            tw.tw_fused_reduce_add_rmsnorm_ex(parts, res, w, dev_out, dev_res, wl.eps, t0,
                                              t0 + chunk, path="auto")
        torch.cuda.synchronize()
        assert torch.equal(out[0], dev_out[0].cpu()) and torch.equal(res_out, dev_res.cpu())


def test_host_in_place_matches_device_cluster_path_bitwise():
    # Reading the host tensors in place runs the cluster kernel over the
    # mapped memory: the same bits as that kernel on device copies.
    wl = CASES[0].with_tokens(300)
    d, out, res_out = host_run(wl, 0)
    dev_out = [torch.empty(wl.T, wl.H, dtype=wl.torch_dtype, device="cuda")]
    dev_res = torch.empty(wl.T, wl.H, dtype=wl.torch_dtype, device="cuda")
    tw.tw_fused_reduce_add_rmsnorm_ex([p.cuda() for p in d["partials"]], d["residual"].cuda(),
                                      d["weight"].cuda(), dev_out, dev_res, wl.eps,
                                      path="cluster")
    torch.cuda.synchronize()
    assert torch.equal(out[0], dev_out[0].cpu()) and torch.equal(res_out, dev_res.cpu())
    assert tw.tw_device_status() == 0


def test_host_rejects_pageable_memory():
    wl = CASES[0].with_tokens(4)
    d = inputs.make_inputs(wl)
    out = [torch.empty(4, wl.H, dtype=wl.torch_dtype)]
    res_out = torch.empty_like(out[0])
    nbytes = tw.tw_host_workspace_bytes(8, 1, wl.H, 4, wl.torch_dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    # The binding refuses pageable tensors before the call ...
    with pytest.raises(ValueError, match="pinned"):
        tw.tw_fused_reduce_add_rmsnorm_host(d["partials"], d["residual"], d["weight"], out,
                                            res_out, wl.eps, ws, 4)
    # ... and so does the C entry point when called with their addresses.
    ptrs = lambda ts: (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])  # noqa: E731
    rc = tw.load().tw_fused_reduce_add_rmsnorm_host(
        ptrs(d["partials"]), 8, d["residual"].data_ptr(), d["weight"].data_ptr(), ptrs(out), 1,
        res_out.data_ptr(), 4, wl.H, wl.eps, 0, 4, 1 << 30, ws.data_ptr(), nbytes, 4,
        torch.cuda.current_stream().cuda_stream, tw.TW_BF16)
    assert rc == -1 and "page-locked" in tw.tw_last_error_string()


def test_binding_refuses_tensors_off_the_device():
    wl = CASES[0].with_tokens(4)
    d = inputs.make_inputs(wl)   # CPU tensors
    out = [torch.empty(4, wl.H, dtype=wl.torch_dtype)]
    with pytest.raises(ValueError, match="current CUDA device"):
        tw.tw_fused_reduce_add_rmsnorm(d["partials"], d["residual"], d["weight"], out,
                                       torch.empty_like(out[0]), wl.eps)


@pytest.mark.parametrize("chunk", [16, 0])
def test_host_in_place_residual(chunk):
    # residual_out is the pinned residual itself: each chunk's rows are read
    # (copied in, or loaded in place) before the kernel writes them back.
    wl = CASES[0]
    t0, t1 = 3, wl.T - 2
    d = inputs.make_inputs(wl)
    parts = [p.pin_memory() for p in d["partials"]]
    res = d["residual"].clone().pin_memory()
    w = d["weight"].pin_memory()
    out = [torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype).pin_memory()]
    tw.tw_fused_reduce_add_rmsnorm_host(parts, res, w, out, res, wl.eps, workspace(wl, chunk),
                                        chunk, t0, t1)
    torch.cuda.synchronize()
    ref_out, ref_res = oracle.reordered([inputs.to_f64(p) for p in d["partials"]],
                                        inputs.to_f64(d["residual"]), inputs.to_f64(d["weight"]),
                                        wl.eps, n_out=1, t0=t0, t1=t1)
    check_close(out[0][t0:t1], ref_out[0][t0:t1], wl.dtype, "in-place out")
    check_close(res[t0:t1], ref_res[t0:t1], wl.dtype, "in-place residual_out")
    assert torch.equal(torch.cat([res[:t0], res[t1:]]),
                       torch.cat([d["residual"][:t0], d["residual"][t1:]]))


@pytest.mark.parametrize("chunk", [8, 0])
def test_host_back_to_back_steps_on_one_stream(chunk):
    # Step 2 reads step 1's host outputs (its partial 0 is step 1's out, its
    # residual step 1's residual_out); enqueued back to back on one stream it
    # must equal the same two steps with the host synchronised between them.
    wl = CASES[0].with_tokens(48)
    d1 = inputs.make_inputs(wl)
    d2 = inputs.make_inputs(replace(wl, seed=wl.seed + 7))
    ws = workspace(wl, chunk)
    w1, w2 = d1["weight"].pin_memory(), d2["weight"].pin_memory()
    p1 = [p.pin_memory() for p in d1["partials"]]
    rest2 = [p.pin_memory() for p in d2["partials"][1:]]
    res1 = d1["residual"].pin_memory()
    results = []
    for sync in (True, False):
        out1 = [torch.zeros(wl.T, wl.H, dtype=wl.torch_dtype).pin_memory()]
        res_out1 = torch.zeros(wl.T, wl.H, dtype=wl.torch_dtype).pin_memory()
        out2 = [torch.zeros(wl.T, wl.H, dtype=wl.torch_dtype).pin_memory()]
        res_out2 = torch.zeros(wl.T, wl.H, dtype=wl.torch_dtype).pin_memory()
        torch.cuda.synchronize()
        tw.tw_fused_reduce_add_rmsnorm_host(p1, res1, w1, out1, res_out1, wl.eps, ws, chunk)
        if sync:
            torch.cuda.synchronize()
        tw.tw_fused_reduce_add_rmsnorm_host([out1[0]] + rest2, res_out1, w2, out2, res_out2,
                                            wl.eps, ws, chunk)
        torch.cuda.synchronize()
        results.append((out2[0].clone(), res_out2.clone()))
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])
    assert bool(torch.isfinite(results[0][0].float()).all())
