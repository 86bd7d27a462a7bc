"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` handle and raises AssertionError when
the oracle disagrees.  The same checks run on the real oracle (test_oracle_pins)
and on builds with planted mistakes (test_oracle_mutants), which must fail at
least one of them.

Pages: "TokenWeave 策略详解：以大模型推理为例" (§1 背景 formula, §2/§3 reorder and
token slices, appendix 数值示例 hidden=4 example); "张量并行Tensor Parallelism"
(MLP: the row-parallel partials sum to the layer output).
"""
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def dyadic(rng, shape, lo=-512, hi=512, shift=6):
    """Random multiples of 2**-shift in a small range: every sum of a few dozen
    of them is exact in fp64, so results that are sums are known exactly."""
    return rng.integers(lo, hi, size=shape).astype(np.float64) / (1 << shift)


def split_into_partials(rng, x, residual, n_parts):
    """Partials p_0..p_{N-1} with sum_r p_r + residual == x exactly (dyadic)."""
    parts = [dyadic(rng, x.shape) for _ in range(n_parts - 1)]
    last = x - residual
    for p in parts:
        last = last - p
    parts.append(last)
    return parts


def _both(orc, *args, **kwargs):
    return (orc.traditional(*args, **kwargs), orc.reordered(*args, **kwargs))


def pin_hidden4_example(orc):
    """Appendix 数值示例: [a,b,0,0] + [0,0,c,d] = [a,b,c,d] on every GPU.  With
    residual 0, weight 1 and eps 0 the normalised row is x / sqrt(mean(x^2)),
    whose mean square we work out by hand per case."""
    hand_mean_sq = {("1", "2", "3", "4"): 7.5,            # (1+4+9+16)/4
                    ("-0.5", "0.25", "-3.75", "1024"): 262147.59375}
    for case in _read_golden("hidden4_zero_pad.txt"):
        a, b, c, d = (float(v) for v in case)
        p0 = np.array([[a, b, 0.0, 0.0]])
        p1 = np.array([[0.0, 0.0, c, d]])
        for outs, res in _both(orc, [p0, p1], np.zeros((1, 4)), np.ones(4), 0.0,
                               n_out=2):
            assert np.array_equal(res[0], [a, b, c, d]), res
            want = np.array([a, b, c, d]) / math.sqrt(hand_mean_sq[tuple(case)])
            for o in outs:
                np.testing.assert_allclose(o[0], want, rtol=1e-15, atol=0)


def pin_eps_inside_sqrt(orc):
    """Constant rows x = c: y = c / sqrt(c^2 + eps) * w.  (c, eps) = (1, 3) and
    (3, 7) give 1/2 and 3/4 exactly, so eps outside the root, a sum in place of
    the mean, or a dropped eps all show."""
    H = 12
    w = np.linspace(0.5, 1.5, H)
    for c, eps, k in ((1.0, 3.0, 0.5), (3.0, 7.0, 0.75), (-3.0, 7.0, -0.75)):
        x = np.full((1, H), c)
        for outs, res in _both(orc, [x], np.zeros((1, H)), w, eps):
            assert np.array_equal(res, x)
            np.testing.assert_allclose(outs[0][0], k * w, rtol=1e-15, atol=0)


def pin_library_rms_norm(orc):
    """Against an independent library routine: for inputs built so that
    sum_r p_r + residual equals a chosen x exactly, residual_out must be x
    bit-for-bit and y must equal torch.nn.functional.rms_norm(x, w, eps) in
    fp64.  Covers tiny shapes (T 0..3, H 8/16, N 1..3) and a few larger ones."""
    rng = np.random.default_rng(1234)
    shapes = [(T, H, N) for T in (0, 1, 2, 3) for H in (8, 16) for N in (1, 2, 3)]
    shapes += [(7, 1000, 8), (5, 4096, 2), (4, 136, 16)]
    for T, H, N in shapes:
        x = dyadic(rng, (T, H))
        residual = dyadic(rng, (T, H))
        parts = split_into_partials(rng, x, residual, N)
        w = rng.uniform(0.5, 1.5, size=H)
        for eps in (1e-6, 0.75):
            want = torch.nn.functional.rms_norm(
                torch.from_numpy(x), (H,), torch.from_numpy(w), eps).numpy()
            for outs, res in _both(orc, parts, residual, w, eps, n_out=2):
                assert np.array_equal(res, x)
                for o in outs:
                    np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-300)


def pin_unit_rms(orc):
    """Before the weight (w = 1), z = x / rms(x) has mean(z^2) = ms / (ms + eps);
    with eps = 0 that is exactly 1 up to fp64 rounding."""
    rng = np.random.default_rng(7)
    T, H, N = 6, 512, 3
    parts = [rng.standard_normal((T, H)) for _ in range(N)]
    residual = rng.standard_normal((T, H))
    for eps in (0.0, 1e-6, 0.5):
        for outs, res in _both(orc, parts, residual, np.ones(H), eps):
            ms = np.mean(res * res, axis=1)
            got = np.mean(outs[0] * outs[0], axis=1)
            np.testing.assert_allclose(got, ms / (ms + eps), rtol=1e-12, atol=0)


def pin_order_equivalence(orc):
    """§3.4 / appendix 总结: the reordered order gives the same output as the
    traditional one.  Same per-token arithmetic, so fp64 bits must agree, for
    uneven splits, T < N, partial ranges and several destinations; all
    destinations are identical and rows outside [t0, t1) are untouched."""
    rng = np.random.default_rng(99)
    cases = [(1, 8, 8, 0, 1, 1), (3, 16, 8, 0, 3, 2), (10, 24, 3, 2, 9, 3),
             (2048 // 64, 64, 2, 0, 32, 1), (5, 40, 4, 1, 4, 4), (0, 8, 2, 0, 0, 2),
             (9, 32, 16, 0, 9, 8), (4, 8, 1, 4, 4, 1)]
    for T, H, N, t0, t1, n_out in cases:
        parts = [rng.standard_normal((T, H)) for _ in range(N)]
        residual = rng.standard_normal((T, H))
        w = rng.uniform(0.5, 1.5, H)
        (o_a, r_a), (o_b, r_b) = _both(orc, parts, residual, w, 1e-6,
                                       n_out=n_out, t0=t0, t1=t1, fill=-7.0)
        assert np.array_equal(r_a, r_b)
        for k in range(n_out):
            assert np.array_equal(o_a[k], o_b[k]), (T, H, N, t0, t1, k)
            assert np.array_equal(o_a[k], o_a[0])
        for arr in [r_a] + o_a:
            assert np.all(arr[:t0] == -7.0) and np.all(arr[t1:] == -7.0)
            assert not np.any(arr[t0:t1] == -7.0)


def pin_shape_walkthrough(orc):
    """§3.2: with N=2 and seq_len 2048, GPU0 owns tokens 0-1023, GPU1 1024-2047."""
    rows = {r[0]: r[1:] for r in _read_golden("shape_walkthrough.txt")
            if r[0] != "token_slice" and r[0] != "column_slice"}
    n = int(rows["n_ranks"][0])
    T = int(rows["seq_len"][0])
    for r in _read_golden("shape_walkthrough.txt"):
        if r[0] == "token_slice":
            rank, first, last = (int(v) for v in r[1:])
            assert orc.token_slice(T, n, rank) == (first, last)
            assert last - first == 1024
    # Floor bounds cover every token once, for even and uneven splits.
    for n_tok in (0, 1, 7, 8, 1023, 2048):
        for n_r in (1, 2, 3, 8, 16):
            bounds = [orc.token_slice(n_tok, n_r, r) for r in range(n_r)]
            assert bounds[0][0] == 0 and bounds[-1][1] == n_tok
            assert all(bounds[i][1] == bounds[i + 1][0] for i in range(n_r - 1))


def pin_zero_pad_concat(orc):
    """Appendix 实现方法：零填充 + AllReduce 求和: zero-padded column-split
    partials sum to the concatenation of each rank's filled columns, exactly."""
    rng = np.random.default_rng(5)
    T, H, N = 3, 40, 4
    blocks = [rng.standard_normal((T, H // N)) for _ in range(N)]
    parts = []
    for r, blk in enumerate(blocks):
        p = np.zeros((T, H))
        p[:, r * H // N:(r + 1) * H // N] = blk
        parts.append(p)
    for outs, res in _both(orc, parts, np.zeros((T, H)), np.ones(H), 1e-6):
        assert np.array_equal(res, np.concatenate(blocks, axis=1))


def pin_invariants(orc):
    """Permuting the partials leaves x unchanged (exact for dyadic data);
    with eps = 0, scaling x by 2**k leaves y unchanged; doubling w doubles y."""
    rng = np.random.default_rng(11)
    T, H, N = 4, 24, 5
    parts = [dyadic(rng, (T, H)) for _ in range(N)]
    residual = dyadic(rng, (T, H))
    w = rng.uniform(0.5, 1.5, H)
    o0, r0 = orc.reordered(parts, residual, w, 0.0)
    o1, r1 = orc.reordered(parts[::-1], residual, w, 0.0)
    assert np.array_equal(r0, r1) and np.array_equal(o0[0], o1[0])
    o2, _ = orc.reordered([p * 8.0 for p in parts], residual * 8.0, w, 0.0)
    np.testing.assert_allclose(o2[0], o0[0], rtol=1e-15, atol=0)
    o3, _ = orc.traditional(parts, residual, w * 2.0, 0.0)
    assert np.array_equal(o3[0], 2.0 * o0[0])


def pin_bad_arguments(orc):
    """Invalid ranges and shapes are refused, nothing is computed."""
    x = np.zeros((2, 8))
    for kwargs in ({"t0": 1, "t1": 0}, {"t0": 0, "t1": 3}, {"t0": -1, "t1": 1}):
        try:
            orc.reordered([x], x, np.ones(8), 1e-6, **kwargs)
        except ValueError:
            pass
        else:
            raise AssertionError(f"accepted {kwargs}")
    try:
        orc.traditional([x], x, np.ones(8), -1.0)
    except ValueError:
        pass
    else:
        raise AssertionError("accepted eps < 0")


def pin_special_values(orc):
    """IEEE special values follow from the definition with no special case: a
    NaN element makes its token's rms NaN (every y of the token NaN,
    residual_out NaN there only); an infinite element makes the rms infinite
    (y NaN there, x / inf = 0 elsewhere in the row); other tokens are finite.
    Both orders agree on the pattern."""
    rng = np.random.default_rng(13)
    T, H, N = 4, 16, 3
    parts = [rng.standard_normal((T, H)) for _ in range(N)]
    residual = rng.standard_normal((T, H))
    w = rng.uniform(0.5, 1.5, H)
    parts[1][1, 3] = math.nan
    parts[0][2, 7] = math.inf
    for fn in (orc.reordered, orc.traditional):
        out, res = fn(parts, residual, w, 1e-6)
        y = out[0]
        assert np.isnan(y[1]).all() and np.isnan(res[1, 3])
        assert np.isfinite(np.delete(res[1], 3)).all()
        assert np.isnan(y[2, 7]) and np.isposinf(res[2, 7])
        assert (np.delete(y[2], 7) == 0.0).all()
        assert np.isfinite(y[[0, 3]]).all() and np.isfinite(res[[0, 3]]).all()


PINS = [pin_hidden4_example, pin_eps_inside_sqrt, pin_library_rms_norm,
        pin_unit_rms, pin_order_equivalence, pin_shape_walkthrough,
        pin_zero_pad_concat, pin_invariants, pin_bad_arguments, pin_special_values]
