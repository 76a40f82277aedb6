"""The host-side draft-length controller (CPU only): 2kiu.com §4.4 (a 100-batch sliding window of
acceptance rates; K + 1 above 0.8, K - 1 below 0.6, K within [2, 10]; switch speculation off
when acceptance stays poor and back on once it recovers) and §7 (the switch-off threshold 0.5).

Hand-built scenarios check each rule and boundary; a plain Python restatement of the same rules
(written here from the pages, independent of the C code) is run beside the controller on random
acceptance histories and must agree batch by batch."""
import math

import numpy as np
import pytest

import speculative_decoding_rejection_verify_gb300 as sv


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_rejection_verify_gb300 import _build
    _build.build()


def feed(c, rate, times=1, B=10):
    """Record `times` batches of B requests at the controller's current K, each with
    round(rate * B * K) accepted drafts; returns the last K the controller gave."""
    k = c.k
    for _ in range(times):
        K = c.k
        n = np.zeros(B, np.int32)
        for i in range(int(round(rate * B * K))):
            n[i % B] += 1
        k = c.update(n, K_used=K)
    return k


def test_defaults_are_the_pages_numbers():
    c = sv.Controller()
    cfg = c.config
    assert (cfg.k_init, cfg.k_min, cfg.k_max, cfg.window, cfg.probe_after) == (4, 2, 10, 100, 100)
    assert (cfg.raise_above, cfg.lower_below, cfg.disable_below) == pytest.approx((0.8, 0.6, 0.5))
    assert c.k == 4 and c.window_fill == 0 and math.isnan(c.window_mean)


def test_raise_after_a_full_window_only():
    c = sv.Controller()
    for i in range(99):
        assert feed(c, 0.9) == 4
    assert c.window_fill == 99 and c.window_mean == pytest.approx(0.9)
    assert feed(c, 0.9) == 5  # the 100th batch decides
    assert c.window_fill == 0  # a new K starts an empty window


def test_lower_and_bounds():
    c = sv.Controller(k_init=3)
    assert feed(c, 0.56, 100) == 2
    assert feed(c, 0.56, 300) == 2  # already at k_min: stays
    c = sv.Controller(k_init=10)
    assert feed(c, 1.0, 300) == 10  # at k_max: stays
    c = sv.Controller(k_init=99)
    assert c.k == 10  # clamped


def test_thresholds_are_strict():
    # a window mean of exactly 0.6 (or between 0.6 and 0.8) changes nothing
    c = sv.Controller()
    assert feed(c, 0.6, 200) == 4
    assert feed(c, 0.7, 100) == 4


def test_switch_off_and_probe_again():
    c = sv.Controller()
    assert feed(c, 0.3, 100) == 0 and c.k == 0
    for i in range(99):
        assert c.skip() == 0
    assert c.skip() == 2  # after 100 batches without drafts: probe at k_min
    assert c.window_fill == 0
    assert feed(c, 0.9, 100) == 3  # acceptance recovered: speculation stays on and grows


def test_rate_uses_k_per_row_and_clamps():
    c = sv.Controller(window=1, raise_above=0.9, lower_below=0.2, disable_below=0.0)
    # K_b = (4, 2, 0): proposed 6, accepted 3 + 2 + 0 (the 5 on a K_b = 0 row is clamped to 0)
    c.update(np.array([3, 2, 5], np.int32), np.array([4, 2, 0], np.int32), K_used=4)
    assert c.window_mean == pytest.approx(5 / 6)
    a, p, b = c.totals()
    assert (a, p, b) == (5, 6, 1)
    # a batch without drafts adds no rate
    c2 = sv.Controller()
    c2.update(np.array([0, 0], np.int32), np.array([0, 0], np.int32), K_used=4)
    assert c2.window_fill == 0 and c2.totals()[2] == 1


def test_bad_settings_rejected():
    for kw in (dict(k_min=0), dict(k_min=5, k_max=4), dict(k_max=65), dict(window=0),
               dict(lower_below=0.9), dict(disable_below=0.7), dict(raise_above=1.5), dict(probe_after=0)):
        with pytest.raises(ValueError):
            sv.Controller(**kw)


# ----------------------------------------------------------------------------------------------
# the rules restated in Python, run beside the controller on random histories
# ----------------------------------------------------------------------------------------------
class Restated:
    def __init__(self, k_init=4, k_min=2, k_max=10, window=100, raise_above=0.8, lower_below=0.6,
                 disable_below=0.5, probe_after=100):
        f32 = lambda x: float(np.float32(x))  # noqa: E731  (the C settings are floats)
        self.k = min(max(k_init, k_min), k_max)
        self.k_min, self.k_max, self.window, self.probe_after = k_min, k_max, window, probe_after
        self.up, self.down, self.off = f32(raise_above), f32(lower_below), f32(disable_below)
        self.rates, self.off_batches = [], 0

    def update(self, n, kb):
        prop = int(kb.sum())
        if prop > 0:
            self.rates.append(int(np.minimum(n, kb).sum()) / prop)
            self.rates = self.rates[-self.window:]
            if self.k > 0 and len(self.rates) == self.window:
                m = float(np.float32(sum(self.rates) / self.window))
                if m < self.off:
                    self.k, self.off_batches, self.rates = 0, 0, []
                elif m > self.up and self.k < self.k_max:
                    self.k, self.rates = self.k + 1, []
                elif m < self.down and self.k > self.k_min:
                    self.k, self.rates = self.k - 1, []
        return self.k

    def skip(self):
        if self.k == 0:
            self.off_batches += 1
            if self.off_batches >= self.probe_after:
                self.k, self.off_batches, self.rates = self.k_min, 0, []
        return self.k


@pytest.mark.parametrize("seed", range(4))
def test_matches_restated_rules(seed):
    rng = np.random.default_rng(seed)
    kw = dict(window=int(rng.integers(3, 20)), probe_after=int(rng.integers(2, 10)))
    c, r = sv.Controller(**kw), Restated(**kw)
    level = 0.7
    for step in range(3000):
        if step % 150 == 0:
            level = float(rng.uniform(0.2, 1.0))  # the traffic changes
        k = c.k
        assert k == r.k, step
        if k == 0:
            assert c.skip() == r.skip()
            continue
        B = int(rng.integers(1, 16))
        kb = rng.integers(0, k + 1, size=B).astype(np.int32)
        n = rng.binomial(kb, level).astype(np.int32)
        assert c.update(n, kb, K_used=k) == r.update(n, kb), step
