"""The online verify-cost curve's host logic (no GPU): P3 "Teaching the Speculator What a Draft
Costs", "What we changed" and "Reproduce".

The library's table is checked against a model written here from the page's rule: every
`rebuild_every` observations, the table is the boot curve with, for each token count that has
at least `min_samples` of its last `window` observations, their median laid on top (numpy's
median: the mean of the two middle values for an even count).  Only observe/table/create are
called, none of which touches a device.
"""

import ctypes

import numpy as np
import pytest

import speculative_decoding_block_verify_gb300 as sv
from speculative_decoding_block_verify_gb300 import build as svbuild


@pytest.fixture(scope="module", autouse=True)
def _lib():
    svbuild.build()
    sv.lib()


class Model:
    def __init__(self, boot, window, min_samples, rebuild_every):
        self.boot = np.asarray(boot, np.float32)
        self.table = self.boot.copy()
        self.window, self.min_samples, self.rebuild_every = window, min_samples, rebuild_every
        self.samples = {}
        self.n = 0
        self.rebuilds = 0

    def observe(self, n, ms):
        if not (0 <= n < len(self.boot)) or not (ms >= 0):
            return
        self.samples.setdefault(n, []).append(np.float32(ms))
        self.n += 1
        if self.n % self.rebuild_every == 0:
            self.rebuilds += 1
            t = self.boot.copy()
            for k, s in self.samples.items():
                last = s[-self.window:]
                if len(last) >= self.min_samples:
                    t[k] = np.median(np.asarray(last, np.float64))
            self.table = t


def _boot(n_max=16):
    return (2.0 + 0.25 * np.arange(n_max + 1)).astype(np.float32)


def test_table_is_the_boot_curve_until_the_first_rebuild():
    c = sv.CostCurve(_boot(), window=32, min_samples=3, rebuild_every=32)
    for i in range(31):
        c.observe(5, 9.0)
    t, cnt = c.table()
    assert np.array_equal(np.float32(t), _boot()) and cnt["rebuilds"] == 0 and cnt["observations"] == 31
    c.observe(5, 9.0)
    t, cnt = c.table()
    assert cnt["rebuilds"] == 1 and t[5] == 9.0
    assert np.array_equal(np.delete(np.float32(t), 5), np.delete(_boot(), 5))
    c.close()


def test_min_samples_and_even_median():
    c = sv.CostCurve(_boot(), window=8, min_samples=3, rebuild_every=6)
    for n, ms in [(3, 1.0), (3, 5.0), (7, 1.0), (7, 2.0), (7, 4.0), (7, 10.0)]:
        c.observe(n, ms)
    t, cnt = c.table()
    assert cnt["rebuilds"] == 1
    assert t[3] == _boot()[3]                  # two samples: below min_samples, boot kept
    assert t[7] == 3.0                         # median of 1, 2, 4, 10 = (2 + 4) / 2
    c.close()


def test_window_keeps_only_the_last_observations():
    c = sv.CostCurve(_boot(), window=4, min_samples=1, rebuild_every=10)
    for ms in [100.0] * 6 + [1.0, 2.0, 3.0, 4.0]:
        c.observe(2, ms)
    t, _ = c.table()
    assert t[2] == 2.5                         # the last four: 1, 2, 3, 4
    c.close()


def test_out_of_range_and_invalid_observations_are_dropped():
    c = sv.CostCurve(_boot(4), window=4, min_samples=1, rebuild_every=1)
    for n, ms in [(-1, 1.0), (5, 1.0), (2, float("nan")), (2, -1.0)]:
        c.observe(n, ms)
    t, cnt = c.table()
    assert cnt == {"observations": 0, "rebuilds": 0, "dropped": 4, "pending": 0}
    c.observe(4, 0.5)
    t, cnt = c.table()
    assert t[4] == 0.5 and cnt["rebuilds"] == 1
    c.close()


@pytest.mark.parametrize("window,min_samples,rebuild_every", [(32, 3, 32), (5, 2, 7), (1, 1, 1)])
def test_random_stream_matches_the_model(window, min_samples, rebuild_every):
    rng = np.random.default_rng(window * 100 + rebuild_every)
    boot = _boot(24)
    c = sv.CostCurve(boot, window=window, min_samples=min_samples, rebuild_every=rebuild_every)
    m = Model(boot, window, min_samples, rebuild_every)
    for i in range(700):
        n = int(rng.integers(-2, 28))
        ms = float(np.float32(rng.gamma(4.0, 0.5)))
        c.observe(n, ms)
        m.observe(n, ms)
        if i % 37 == 0 or i == 699:
            t, cnt = c.table()
            assert cnt["rebuilds"] == m.rebuilds
            np.testing.assert_allclose(np.float32(t), m.table, rtol=1e-6, atol=0)
    c.close()


def test_planted_mistake_mean_instead_of_median_is_caught():
    """A model that lays the mean on top (a plausible slip) disagrees with the library on a
    skewed window, so the comparison above can tell the two apart."""
    c = sv.CostCurve(_boot(), window=8, min_samples=3, rebuild_every=5)
    for ms in [1.0, 1.0, 1.0, 1.0, 50.0]:
        c.observe(6, ms)
    t, _ = c.table()
    assert t[6] == 1.0 and t[6] != np.mean([1.0, 1.0, 1.0, 1.0, 50.0])
    c.close()


def test_create_refuses_invalid_knobs():
    L = sv.lib()
    boot = (ctypes.c_float * 5)(*([1.0] * 5))
    assert L.spec_cost_curve_create(None, 4, 32, 3, 32) is None
    assert L.spec_cost_curve_create(boot, 0, 32, 3, 32) is None
    assert L.spec_cost_curve_create(boot, 4, 0, 1, 32) is None
    assert L.spec_cost_curve_create(boot, 4, 2, 3, 32) is None          # min_samples > window
    assert L.spec_cost_curve_create(boot, 4, 32, 3, 0) is None
    assert b"invalid" in L.spec_last_error()
    h = L.spec_cost_curve_create(boot, 4, 32, 3, 32)
    assert h is not None
    assert L.spec_cost_curve_end(h, 0, None, None) == -1                # end without begin
    L.spec_cost_curve_destroy(h)
    L.spec_cost_curve_destroy(None)
