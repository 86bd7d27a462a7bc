"""The rows kernel's multi-token units: for rows of at most 8 KB a CTA takes
2 or 4 consecutive tokens at a time, so that one bulk copy moves a buffer's
rows of the whole unit.  Checked against the oracle (ragged last units,
sub-ranges starting at odd tokens, small budgets where the ring wraps many
times, several destinations, in place), and bit for bit against launches of
fewer tokens than SMs, which always take one token per unit: the arithmetic
of a token does not depend on the unit it was staged in."""
import pytest
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
from reduce_residual_rmsnorm_tw_gb300.inputs import Workload
from tests.parity import alloc_outputs, check_workload

pytestmark = pytest.mark.gpu


def wl(n, T, H, dtype="bf16", n_out=1, seed=71):
    return Workload(f"units_n{n}_t{T}_h{H}_{dtype}_o{n_out}", n, T, H, dtype, 1e-6, n_out, seed)


# (workload, budget): rows of 16 B to 8 KB, budgets where the rule picks
# units of 4 (4 KB rows on 3 SMs), 2 (8 KB rows on the whole GPU) and 4 again
# on tiny rows; token counts leave a ragged last unit.
CASES = [
    (wl(2, 1199, 2048), 3),
    (wl(2, 1203, 4096), None),
    (wl(3, 2047, 4096, n_out=2), 8),
    (wl(5, 903, 1000), 2),
    (wl(1, 777, 8), 1),
    (wl(4, 1201, 1024, "f32", n_out=3), 5),
    (wl(2, 1499, 2048, "f32"), None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}_sms{c[1]}")
def test_units_match_oracle(case):
    w, sms = case
    check_workload(w, path="rows", max_sms=sms)
    check_workload(w, path="rows", max_sms=sms, t0=5, t1=w.T - 3)


@pytest.mark.parametrize("case", CASES[:3], ids=lambda c: f"{c[0].name}_sms{c[1]}")
def test_units_in_place(case):
    w, sms = case
    check_workload(w, path="rows", max_sms=sms, t0=1, t1=w.T, in_place=True)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}_sms{c[1]}")
def test_units_bit_identical_to_one_token_units(case):
    w, sms = case
    d = inputs.make_inputs(w, device="cuda")
    out_a, res_a = alloc_outputs(w)
    tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out_a, res_a,
                                      w.eps, max_sms=sms, path="rows")
    # Ranges of 100 tokens on the whole GPU: fewer tokens than SMs, one
    # token per unit.
    out_b, res_b = alloc_outputs(w)
    for t0 in range(0, w.T, 100):
        tw.tw_fused_reduce_add_rmsnorm_ex(d["partials"], d["residual"], d["weight"], out_b,
                                          res_b, w.eps, t0, min(t0 + 100, w.T), path="rows")
    torch.cuda.synchronize()
    for a, b in zip(out_a + [res_a], out_b + [res_b]):
        assert torch.equal(a, b)
    assert tw.tw_device_status() == 0
