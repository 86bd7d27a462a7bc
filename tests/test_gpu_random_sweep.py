"""Seeded random sweep of small shapes against the oracle: N, T, H, dtype,
destinations, sub-range, in-place residual, kernel and SM budget are drawn
from a fixed generator, always within the rules of include/tw.h."""
import numpy as np
import pytest

from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import check_workload

pytestmark = pytest.mark.gpu


def draw_cases(n_cases, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n_cases):
        dtype = "bf16" if rng.random() < 0.6 else "f32"
        es = 2 if dtype == "bf16" else 4
        max_vecs = 16384 * 2 // 16            # rows of at most 32 KB
        vecs = int(rng.integers(1, max_vecs + 1)) if rng.random() < 0.3 else int(rng.integers(1, 257))
        H = vecs * 16 // es
        n = int(rng.integers(1, 17))
        T = int(rng.integers(1, 48))
        n_out = int(rng.integers(1, 5))
        t0 = int(rng.integers(0, T))
        t1 = int(rng.integers(t0, T + 1))
        path = ["rows", "warp", "cluster", "auto"][int(rng.integers(0, 4))]
        max_sms = [None, 1, 3, 8, 20][int(rng.integers(0, 5))]
        if path == "cluster":
            cluster = 1
            budget = 152 if max_sms is None else max_sms
            while cluster * 2 <= min(8, budget):
                cluster *= 2
            if H * es > cluster * 8192:       # row too long for that cluster
                path = "rows"
        in_place = bool(rng.random() < 0.25)
        eps = float(10.0 ** rng.uniform(-7, -1))
        wl = Workload(f"rand{i}_n{n}_t{T}_h{H}_{dtype}_o{n_out}", n, T, H, dtype, eps, n_out,
                      1000 + i, partial_std=float(rng.uniform(0.2, 1.5)))
        cases.append((wl, path, t0, t1, max_sms, in_place))
    return cases


CASES = draw_cases(40)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}_{c[1]}_{c[2]}-{c[3]}_sms{c[4]}")
def test_random_shape(case):
    wl, path, t0, t1, max_sms, in_place = case
    check_workload(wl, path=path, t0=t0, t1=t1, max_sms=max_sms, in_place=in_place)
