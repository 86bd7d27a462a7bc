"""The oracle's token loops are independent per token, so its results do not
depend on how many host threads run them; the benchmark's CPU legs set the
thread count to the host's cores whatever OMP_NUM_THREADS says."""
import numpy as np

import oracle


def test_results_do_not_depend_on_thread_count():
    rng = np.random.default_rng(5)
    parts = [rng.standard_normal((37, 96)) for _ in range(3)]
    res = rng.standard_normal((37, 96))
    w = rng.standard_normal(96)
    before = oracle.threads()
    try:
        oracle.set_threads(1)
        assert oracle.threads() == 1
        one = oracle.reordered(parts, res, w, 1e-6, n_out=2)
        oracle.set_threads(4)
        assert oracle.threads() == 4
        four = oracle.reordered(parts, res, w, 1e-6, n_out=2)
    finally:
        oracle.set_threads(before)
    for a, b in zip(one[0] + [one[1]], four[0] + [four[1]]):
        assert np.array_equal(a, b)


def test_non_positive_thread_count_is_ignored():
    before = oracle.threads()
    oracle.set_threads(0)
    oracle.set_threads(-3)
    assert oracle.threads() == before
