"""The no-allocation host-buffer entry point, for callers that cannot allocate
device memory (a host program with no CUDA allocator of its own, device memory
reserved up front by a framework, code where cudaMalloc is not allowed): it
must give the same result, within the tests' tolerance, as the host-buffer
entry point that takes a caller-allocated workspace, on two calls in a row
(the second on different data, so stale staging from the first cannot leak
through).  Collected last: it works in a fresh process (where its first call
sets up the device array's address) and after every other test."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import SENTINEL, check_close

pytestmark = pytest.mark.gpu


def _pinned(wl):
    d = inputs.make_inputs(wl)
    return ([p.pin_memory() for p in d["partials"]], d["residual"].pin_memory(),
            d["weight"].pin_memory())


def _outputs(wl):
    out = [torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype).pin_memory()
           for _ in range(wl.n_out)]
    return out, torch.full((wl.T, wl.H), SENTINEL, dtype=wl.torch_dtype).pin_memory()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_no_alloc_matches_workspace_entry_on_two_calls(dtype):
    calls = [Workload(f"noalloc_a_{dtype}", 8, 70, 8192, dtype, 1e-5, 2, 41),
             Workload(f"noalloc_b_{dtype}", 8, 70, 8192, dtype, 1e-6, 2, 42)]
    ranges = [(0, 70), (3, 61)]
    for wl, (t0, t1) in zip(calls, ranges):
        parts, res, w = _pinned(wl)
        out, res_out = _outputs(wl)
        tw.tw_fused_reduce_add_rmsnorm_host_noalloc(parts, res, w, out, res_out, wl.eps,
                                                    t0=t0, t1=t1)
        ref_out, ref_res = _outputs(wl)
        chunk = 32
        ws = torch.empty(tw.tw_host_workspace_bytes(wl.n_parts, wl.n_out, wl.H, chunk,
                                                    wl.torch_dtype),
                         dtype=torch.uint8, device="cuda")
        tw.tw_fused_reduce_add_rmsnorm_host(parts, res, w, ref_out, ref_res, wl.eps, ws, chunk,
                                            t0=t0, t1=t1)
        torch.cuda.synchronize()
        for k in range(wl.n_out):
            check_close(out[k][t0:t1], inputs.to_f64(ref_out[k][t0:t1]), dtype,
                        f"{wl.name} out[{k}]")
            assert bool((torch.cat([out[k][:t0], out[k][t1:]]).float() == SENTINEL).all())
        check_close(res_out[t0:t1], inputs.to_f64(ref_res[t0:t1]), dtype,
                    f"{wl.name} residual_out")
        assert bool((torch.cat([res_out[:t0], res_out[t1:]]).float() == SENTINEL).all())
    assert tw.tw_device_status() == 0


def test_no_alloc_refuses_chunks_beyond_its_array():
    wl = Workload("noalloc_big", 8, 64, 8192, "bf16", 1e-5, 1, 43)
    parts, res, w = _pinned(wl)
    out, res_out = _outputs(wl)
    # 47-token chunks need 16 KB + 2 * 11 * 47 * 16 KB of staging, above 16 MiB
    # (a chunk longer than the range would be cut to the range first).
    with pytest.raises(tw.TwError, match="TW_ERR_UNSUPPORTED"):
        tw.tw_fused_reduce_add_rmsnorm_host_noalloc(parts, res, w, out, res_out, wl.eps,
                                                    chunk_tokens=47)
    # 46 tokens fit; nothing was written by the refused call.
    assert bool((out[0].float() == SENTINEL).all())
    tw.tw_fused_reduce_add_rmsnorm_host_noalloc(parts, res, w, out, res_out, wl.eps,
                                                chunk_tokens=46)
    torch.cuda.synchronize()
    assert not bool((out[0].float() == SENTINEL).any())


# Default chunk (chunk_tokens = 0) on rows of 16 bytes to 20 KB, each range
# long enough to need two or three chunks of the 16 MiB array: small rows
# whose rounded staging grows by less than a row per token, and rows whose
# staging is not a whole number of 256-byte units (H = 136 bf16).
DEFAULT_CHUNK_CASES = [
    Workload("noalloc_h8_bf16", 8, 50000, 8, "bf16", 1e-6, 2, 44),
    Workload("noalloc_h64_bf16", 8, 6000, 64, "bf16", 1e-6, 2, 45),
    Workload("noalloc_h136_bf16", 8, 3000, 136, "bf16", 1e-6, 2, 46),
    Workload("noalloc_h8192_bf16", 8, 100, 8192, "bf16", 1e-5, 2, 47),
    Workload("noalloc_h4_f32", 4, 60000, 4, "f32", 1e-6, 4, 48),
    Workload("noalloc_h5120_f32", 4, 100, 5120, "f32", 1e-6, 4, 49),
]


@pytest.mark.parametrize("wl", DEFAULT_CHUNK_CASES, ids=lambda w: w.name)
def test_no_alloc_default_chunk_matches_oracle(wl):
    import oracle
    parts, res, w = _pinned(wl)
    out, res_out = _outputs(wl)
    t0, t1 = 1, wl.T - 2
    for _ in range(2):  # two calls in a row on the shared array
        tw.tw_fused_reduce_add_rmsnorm_host_noalloc(parts, res, w, out, res_out, wl.eps,
                                                    t0=t0, t1=t1)
        torch.cuda.synchronize()
        ref_out, ref_res = oracle.reordered([inputs.to_f64(p) for p in parts],
                                            inputs.to_f64(res), inputs.to_f64(w), wl.eps,
                                            n_out=wl.n_out, t0=t0, t1=t1)
        for k in range(wl.n_out):
            check_close(out[k][t0:t1], ref_out[k][t0:t1], wl.dtype, f"{wl.name} out[{k}]")
            assert bool((torch.cat([out[k][:t0], out[k][t1:]]).float() == SENTINEL).all())
        check_close(res_out[t0:t1], ref_res[t0:t1], wl.dtype, f"{wl.name} residual_out")
        assert bool((torch.cat([res_out[:t0], res_out[t1:]]).float() == SENTINEL).all())
    assert tw.tw_device_status() == 0
