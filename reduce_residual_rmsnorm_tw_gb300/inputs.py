"""Seeded synthetic inputs for the fused reduce + residual add + RMSNorm path.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds shapes, value distributions and seeds only -- none of the method's
arithmetic -- so that both sides of a parity check see the same bits.

Recipe (one ``torch.Generator`` seeded with the workload's seed, values drawn
in fp32 and rounded to nearest-even into the storage dtype):
  1. partials r = 0 .. N-1, each [T, H]:
       dense      N(0, 1) * partial_std
       column     rank r draws N(0, 1) for columns
                  [floor(r*H/N), floor((r+1)*H/N)) and is zero elsewhere
                  (the zero-padded column split of "TokenWeave 策略详解",
                  appendix 实现方法：零填充 + AllReduce 求和)
  2. residual [T, H] ~ N(0, 1)
  3. weight [H] ~ U(0.5, 1.5)
Row-parallel partials with var 1/8 at N=8 follow "张量并行Tensor
Parallelism", MLP (Y = sum_i Y_i): their sum has unit variance.
"""
from dataclasses import dataclass, replace

import torch

DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload of the hot path."""
    name: str
    n_parts: int
    T: int
    H: int
    dtype: str          # "bf16" or "f32"
    eps: float
    n_out: int
    seed: int
    partial_std: float = 1.0
    column_split: bool = False

    @property
    def torch_dtype(self):
        return DTYPES[self.dtype]

    @property
    def elem_bytes(self):
        return 2 if self.dtype == "bf16" else 4

    def bytes_per_token(self):
        """Algorithmic HBM bytes per token: N partial rows + residual row
        read, n_out gather rows + residual_out row written."""
        return (self.n_parts + 1 + self.n_out + 1) * self.H * self.elem_bytes

    def with_tokens(self, T):
        return replace(self, T=T, name=f"{self.name}@T{T}")


WORKLOADS = {
    # N=2, T=2048, H=4096: the shape walk-through of "TokenWeave 策略详解" §3.
    "tp2_t2048_h4096_bf16": Workload(
        "tp2_t2048_h4096_bf16", 2, 2048, 4096, "bf16", 1e-6, 1, 0),
    # N=8 dense row-parallel partials at ~1024 tokens per iteration.
    "tp8_t1024_h8192_bf16": Workload(
        "tp8_t1024_h8192_bf16", 8, 1024, 8192, "bf16", 1e-5, 1, 1,
        partial_std=(1.0 / 8.0) ** 0.5),
    # Decode-size batches (T is swept over DECODE_TOKENS).
    "decode_tp8_h8192_bf16": Workload(
        "decode_tp8_h8192_bf16", 8, 256, 8192, "bf16", 1e-6, 1, 2),
    # Large batch run as two token chunks on two streams.
    "split_tp8_t16384_h8192_bf16": Workload(
        "split_tp8_t16384_h8192_bf16", 8, 16384, 8192, "bf16", 1e-6, 1, 3),
    # Zero-padded column-split partials, fp32, four gather destinations.
    "colsplit_tp4_t8192_h5120_f32_out4": Workload(
        "colsplit_tp4_t8192_h5120_f32_out4", 4, 8192, 5120, "f32", 1e-6, 4, 4,
        column_split=True),
}

DECODE_TOKENS = (1, 8, 64, 256)
SM_BUDGETS = (2, 4, 8, 16, 148)


def column_bounds(H, n_parts, r):
    """Columns [first, last) that rank r fills in a zero-padded column split."""
    return (H * r) // n_parts, (H * (r + 1)) // n_parts


def make_inputs(wl: Workload, device="cpu", gen_device=None):
    """Draw the workload's tensors.

    Returns a dict with ``partials`` (list of [T, H]), ``residual`` ([T, H])
    and ``weight`` ([H]) in the storage dtype on ``device``.  The generator runs
    on ``gen_device`` (default: ``device``); CPU and CUDA generators give
    different streams, so both sides of a comparison must use one source.
    """
    gen_device = torch.device(gen_device if gen_device is not None else device)
    g = torch.Generator(device=gen_device)
    g.manual_seed(wl.seed)
    T, H, N = wl.T, wl.H, wl.n_parts
    dt = wl.torch_dtype

    def normal(rows, cols):
        return torch.randn(rows, cols, generator=g, device=gen_device,
                           dtype=torch.float32)

    partials = []
    for r in range(N):
        if wl.column_split:
            c0, c1 = column_bounds(H, N, r)
            p = torch.zeros(T, H, device=gen_device, dtype=torch.float32)
            p[:, c0:c1] = normal(T, c1 - c0)
        else:
            p = normal(T, H)
            if wl.partial_std != 1.0:
                p.mul_(wl.partial_std)
        partials.append(p.to(dt).to(device))
        del p
    residual = normal(T, H).to(dt).to(device)
    weight = (torch.rand(H, generator=g, device=gen_device, dtype=torch.float32)
              .add_(0.5).to(dt).to(device))
    return {"partials": partials, "residual": residual, "weight": weight}


def to_f64(t):
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
