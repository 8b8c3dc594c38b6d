"""The acceptance rule itself (no GPU): planted errors are judged as the
rule of vLLM PR 60684 (Validation) says."""
import numpy as np

from tolerance import acceptance, assert_lse


def test_exact_passes():
    r = np.random.default_rng(0).standard_normal(100000)
    assert acceptance(r, r)["ok"]


def test_outlier_budget():
    r = np.zeros(100000)
    g = r.copy()
    g[:10] = 0.2          # 10 = 1e-4 * 1e5 outliers, below the hard bound
    assert acceptance(g, r)["ok"]
    g[10] = 0.2           # one too many
    assert not acceptance(g, r)["ok"]


def test_hard_bound():
    r = np.zeros(100000)
    g = r.copy()
    g[0] = 0.26
    assert not acceptance(g, r)["ok"]


def test_relative_part():
    r = np.full(1000, 10.0)
    assert not acceptance(r * 1.054, r)["ok"]               # 0.54 > 0.25 bound
    assert acceptance(r + 0.549, r)["ok"] is False          # hard bound
    small = np.full(1000, 1.0)
    assert acceptance(small + 0.099, small)["ok"]           # 0.05 + 0.05*1
    assert not acceptance(small + 0.101, small)["ok"]


def test_nonfinite_fails():
    r = np.zeros(10)
    g = r.copy()
    g[3] = np.nan
    assert not acceptance(g, r)["ok"]


def test_lse_rule():
    r = np.array([0.0, 1.0, -np.inf])
    assert_lse(np.array([0.005, 1.0, -np.inf]), r)
    try:
        assert_lse(np.array([0.02, 1.0, -np.inf]), r)
        raise RuntimeError("should fail")
    except AssertionError:
        pass
