"""The pages' two-chunk layer step on one GPU ("TokenWeave: Efficient
Compute-Communication Overlap for Distributed LLM Inference", gist.science
summary, "Der intelligente Split" and "Der Fused Kernel").

A row-parallel linear layer leaves its output in partial 0 (the other
partials stand for the other ranks' outputs).  The batch is cut into two token
chunks A and B: the GEMM of chunk A runs first; then the GEMM of chunk B runs
on its stream while the fused reduce + residual add + RMSNorm of chunk A runs
beside it on a second stream, held to a few SMs; the fused step of chunk B
follows its GEMM with the whole GPU.  Events order each fused step after the
GEMM that writes its rows.

The GEMM is a plain library GEMM (``torch.matmul``, cuBLAS): the compute the
pages overlap with, not part of the fused path.  Every step of the fused path
runs in libtw.so.
"""
import torch

from . import tw


def two_chunk_layer_step(x, wmat, partials, residual, weight, out, residual_out, eps,
                         budget, gemm_stream, fused_stream, t_split=None):
    """Enqueue one two-chunk layer step.

    ``x`` [T, K] and ``wmat`` [K, H] give partial 0 = x @ wmat ([T, H], written
    chunk by chunk); chunk A is tokens [0, t_split) (default T // 2), fused on
    ``fused_stream`` under a budget of ``budget`` SMs beside the GEMM of chunk
    B; chunk B is fused with the whole GPU once its GEMM is done.  On return
    ``gemm_stream`` is ordered after the whole step."""
    T = residual.shape[0]
    split = T // 2 if t_split is None else t_split
    done_a, done_b = torch.cuda.Event(), torch.cuda.Event()
    with torch.cuda.stream(gemm_stream):
        torch.matmul(x[:split], wmat, out=partials[0][:split])
        done_a.record(gemm_stream)
        torch.matmul(x[split:], wmat, out=partials[0][split:])
        done_b.record(gemm_stream)
    fused_stream.wait_event(done_a)
    tw.tw_fused_reduce_add_rmsnorm(partials, residual, weight, out, residual_out, eps, 0, split,
                                   max_sms=budget, stream=fused_stream)
    fused_stream.wait_event(done_b)
    tw.tw_fused_reduce_add_rmsnorm(partials, residual, weight, out, residual_out, eps, split, T,
                                   stream=fused_stream)
    gemm_stream.wait_stream(fused_stream)


def sequential_layer_step(x, wmat, partials, residual, weight, out, residual_out, eps, stream):
    """The same layer without the split: the whole GEMM, then the fused step
    with the whole GPU, on one stream."""
    with torch.cuda.stream(stream):
        torch.matmul(x, wmat, out=partials[0])
    tw.tw_fused_reduce_add_rmsnorm(partials, residual, weight, out, residual_out, eps,
                                   stream=stream)
