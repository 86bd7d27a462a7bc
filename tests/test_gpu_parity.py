"""CUDA path vs the fp64 oracle, element by element, at sizes the oracle
finishes in seconds: several chunks and CTAs per launch, ragged chunk tails,
sub-ranges, in-place residual, several destinations, both dtypes, both
kernels, and the edge cases (empty range, one token, maximum H and N)."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import check_workload

pytestmark = pytest.mark.gpu


def wl(n, T, H, dtype="bf16", n_out=1, eps=1e-6, seed=11, column=False, std=1.0):
    return Workload(f"n{n}_t{T}_h{H}_{dtype}_o{n_out}", n, T, H, dtype, eps, n_out, seed,
                    partial_std=std, column_split=column)


CASES = [
    wl(1, 5, 8),                       # one 16-byte vector per row
    wl(2, 37, 4096),                   # two full chunks per token
    wl(3, 50, 1000),                   # ragged single chunk (125 of 256 vectors)
    wl(8, 70, 8192, eps=1e-5, std=(1 / 8) ** 0.5),
    wl(16, 19, 2056, n_out=3),         # max partials, ragged second chunk
    wl(8, 9, 16384, n_out=2),          # max bf16 H: 8 chunks in registers
    wl(5, 13, 2040, n_out=8),          # max destinations
    wl(4, 33, 5120, "f32", n_out=4, column=True),
    wl(2, 9, 4, "f32"),                # one vector per row
    wl(5, 21, 8192, "f32"),            # max fp32 H
    wl(16, 7, 1028, "f32", n_out=2),   # ragged fp32 chunk
    wl(3, 40, 6000, "f32", eps=0.5),   # large eps, 6 ragged chunks
    wl(4, 23, 2048, eps=0.0),          # eps = 0 (rows are never all zero)
]


@pytest.mark.parametrize("path", ["rows", "warp", "cluster", "auto"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_parity_full_range(case, path):
    check_workload(case, path=path)


@pytest.mark.parametrize("path", ["rows", "warp", "cluster"])
@pytest.mark.parametrize("case", [CASES[1], CASES[4], CASES[7]], ids=lambda c: c.name)
def test_parity_sub_range(case, path):
    check_workload(case, path=path, t0=3, t1=case.T - 2)


# CASES[5] (bf16 rows of 32 KB) runs the warp kernel in its two-pass form,
# the others keep x in shared memory.
@pytest.mark.parametrize("path", ["rows", "warp", "cluster"])
@pytest.mark.parametrize("case", [CASES[3], CASES[5], CASES[9]], ids=lambda c: c.name)
def test_parity_in_place_residual(case, path):
    check_workload(case, path=path, t0=2, t1=case.T - 1, in_place=True)


@pytest.mark.parametrize("max_sms", [1, 2, 7])
def test_parity_small_sm_budget(max_sms):
    # Many tokens per CTA: the stage ring wraps around many times.
    check_workload(wl(8, 45, 8192, n_out=2), path="rows", max_sms=max_sms)
    check_workload(wl(3, 30, 1000), path="warp", max_sms=max_sms)
    # Cluster of 1, 2 or 4 CTAs: rows of up to 8 KB per CTA.
    check_workload(wl(3, 30, 4096), path="cluster", max_sms=max_sms)


# Small budgets over rows of 1 to 4 vectors per thread and 2 to 9 rows per
# token: many tokens per CTA, the ring's stages dealt to two producer warps
# (an odd ring depth cut to an even one), with and without an in-place
# residual.
BUDGET_SHAPES = [
    wl(1, 23, 8192),                   # two rows per token
    wl(2, 31, 4096, n_out=2),
    wl(8, 29, 8192, eps=1e-5, std=(1 / 8) ** 0.5),   # three stages per token
    wl(4, 17, 12288),                  # 3 vectors per thread
    wl(3, 11, 16384),                  # 4 vectors per thread
    wl(6, 19, 4096, "f32", n_out=3),
    wl(3, 27, 1000),                   # ragged row, one vector per thread
    wl(16, 3000, 64, n_out=2),         # 16 one-token stages: the ring wraps ~190 times per CTA
]


@pytest.mark.parametrize("max_sms", [1, 4, 76])
@pytest.mark.parametrize("case", BUDGET_SHAPES, ids=lambda c: c.name)
def test_parity_budget_shapes(case, max_sms):
    check_workload(case, path="rows", max_sms=max_sms)
    check_workload(case, path="rows", max_sms=max_sms, t0=1, t1=case.T - 1, in_place=True)


def test_cluster_rejects_rows_too_long_for_the_budget():
    from reduce_residual_rmsnorm_tw_gb300 import tw
    with pytest.raises(tw.TwError, match="TW_ERR_UNSUPPORTED"):
        check_workload(wl(2, 4, 8192), path="cluster", max_sms=1)   # 16 KB row, 1 CTA


COLSPLIT = [
    wl(4, 33, 5120, "f32", n_out=4, column=True),
    wl(2, 41, 4096, n_out=2, column=True),
    wl(8, 17, 8192, column=True),
    wl(4, 9, 16384, column=True),
]


@pytest.mark.parametrize("case", COLSPLIT, ids=lambda c: c.name)
def test_colsplit_parity_and_bits(case):
    out, res = check_workload(case, colsplit=True)
    dense_out, dense_res = check_workload(case, path="rows")
    for a, b in zip(out + [res], dense_out + [dense_res]):
        assert torch.equal(a, b), "column-split result differs from the dense rows kernel"


def test_colsplit_sub_range_in_place():
    check_workload(COLSPLIT[0], colsplit=True, t0=5, t1=30, in_place=True)


# Several units per CTA under a budget (the two-pipeline variant of the rows
# kernel, whose consumer groups take alternate units): fp32 rows of 20 KB in
# one-token units, bf16 rows of 8 KB in units of two tokens, a ragged tail.
COLSPLIT_BUDGET = [
    (wl(4, 67, 5120, "f32", n_out=2, column=True), 3),
    (wl(2, 203, 4096, column=True), 8),
    (wl(8, 61, 2048, column=True), 5),
]


@pytest.mark.parametrize("case", COLSPLIT_BUDGET, ids=lambda c: f"{c[0].name}_sms{c[1]}")
def test_colsplit_under_budget(case):
    w, sms = case
    out, res = check_workload(w, colsplit=True, max_sms=sms)
    dense_out, dense_res = check_workload(w, path="rows", max_sms=sms)
    for a, b in zip(out + [res], dense_out + [dense_res]):
        assert torch.equal(a, b), "column-split result differs from the dense rows kernel"
    check_workload(w, colsplit=True, max_sms=sms, t0=3, t1=w.T - 2, in_place=True)


def test_parity_traditional_order():
    check_workload(CASES[3], order="traditional")


@pytest.mark.parametrize("path", ["rows", "warp", "cluster"])
def test_single_token_and_empty_range(path):
    check_workload(wl(8, 1, 8192), path=path)
    check_workload(wl(2, 6, 64), path=path, t0=4, t1=4)   # no-op: nothing written
    check_workload(wl(2, 6, 64), path=path, t0=5, t1=6)   # last row only


def test_split_launch_parity():
    case = wl(8, 64, 8192)
    for t_split in (0, 1, 31, 64):
        check_workload(case, split=t_split)


def test_device_status_clean():
    from reduce_residual_rmsnorm_tw_gb300 import tw
    check_workload(CASES[1], path="rows")
    torch.cuda.synchronize()
    assert tw.tw_device_status() == 0
