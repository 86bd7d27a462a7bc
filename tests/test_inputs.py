"""Host checks of the seeded input generator (shapes, seeds, distributions)."""
import torch

from reduce_residual_rmsnorm_tw_gb300 import inputs


def test_workloads_match_their_names():
    for name, wl in inputs.WORKLOADS.items():
        assert wl.name == name
        assert f"h{wl.H}" in name and f"tp{wl.n_parts}" in name and wl.dtype in name


def test_seeded_and_deterministic():
    wl = inputs.WORKLOADS["tp8_t1024_h8192_bf16"].with_tokens(4)
    a = inputs.make_inputs(wl)
    b = inputs.make_inputs(wl)
    for x, y in zip(a["partials"] + [a["residual"], a["weight"]],
                    b["partials"] + [b["residual"], b["weight"]]):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)


def test_distributions():
    wl = inputs.WORKLOADS["tp8_t1024_h8192_bf16"].with_tokens(64)
    d = inputs.make_inputs(wl)
    p = torch.stack(d["partials"]).float()
    assert abs(p.std().item() - (1 / 8) ** 0.5) < 0.01
    assert abs(p.mean().item()) < 0.01
    assert abs(d["residual"].float().std().item() - 1.0) < 0.02
    w = d["weight"].float()
    assert w.min() >= 0.5 and w.max() <= 1.5 and abs(w.mean().item() - 1.0) < 0.02


def test_column_split_structure():
    wl = inputs.WORKLOADS["colsplit_tp4_t8192_h5120_f32_out4"].with_tokens(3)
    d = inputs.make_inputs(wl)
    for r, p in enumerate(d["partials"]):
        assert p.dtype == torch.float32
        c0, c1 = inputs.column_bounds(wl.H, wl.n_parts, r)
        assert (c0, c1) == (1280 * r, 1280 * (r + 1))
        assert torch.count_nonzero(p[:, :c0]) == 0 and torch.count_nonzero(p[:, c1:]) == 0
        assert torch.count_nonzero(p[:, c0:c1]) == 3 * 1280


def test_bytes_per_token():
    wl = inputs.WORKLOADS["tp8_t1024_h8192_bf16"]
    assert wl.bytes_per_token() == 180224
    assert inputs.WORKLOADS["tp2_t2048_h4096_bf16"].bytes_per_token() == 40960
    assert inputs.WORKLOADS["colsplit_tp4_t8192_h5120_f32_out4"].bytes_per_token() == 204800
