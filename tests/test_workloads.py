"""The seeded input generator: shapes, dtypes, determinism, distributions."""

import numpy as np
import pytest

from transformer_linear_layer_tcgen05_gb300 import workloads as wl


@pytest.mark.parametrize("form", wl.FORMS)
def test_shapes_and_dtypes(form):
    M, N, K = 33, 24, 20
    d = wl.generate(form, M, N, K, seed=1)
    if wl.form_is_at(form):
        assert d["GATE" if wl.form_is_swiglu(form) else "X"].shape == (M, K)
        assert d["DY"].shape == (M, N)
        assert ("R" in d) == wl.form_has_residual(form)
        if "R" in d:
            assert d["R"].shape == (K, N) and d["R"].dtype == np.float32
    elif wl.form_is_t(form):
        assert d["DY"].shape == (M, N) and d["DY"].dtype == np.float32
        assert ("R" in d) == wl.form_has_residual(form)
        if "R" in d:
            assert d["R"].shape == (M, K) and d["R"].dtype == np.float32
    elif wl.form_is_swiglu(form):
        assert d["GATE"].shape == (M, K) and d["UP"].shape == (M, K)
        assert d["GATE"].dtype == np.float32 and d["UP"].dtype == np.float32
    else:
        assert d["X"].shape == (M, K) and d["X"].dtype == np.float32
    if wl.form_is_at(form):
        assert "W" not in d and "W16" not in d
    elif wl.form_is_w16(form):
        assert d["W16"].shape == (K, N) and d["W16"].dtype == np.uint16
    else:
        assert d["W"].shape == (K, N) and d["W"].dtype == np.float32
    assert ("R" in d) == wl.form_has_residual(form)
    for a in d.values():
        assert a.flags.c_contiguous


def test_deterministic_and_seed_sensitive():
    a = wl.generate("matmul_residual_swiglu_a_w16", 40, 32, 16, seed=5)
    b = wl.generate("matmul_residual_swiglu_a_w16", 40, 32, 16, seed=5)
    c = wl.generate("matmul_residual_swiglu_a_w16", 40, 32, 16, seed=6)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["GATE"], c["GATE"])


def test_variances_and_outliers():
    d = wl.generate("matmul_residual_swiglu_a", 400, 64, 1000, seed=3, w_var=1.0 / 1000,
                    outlier_frac=0.01)
    g = d["GATE"]
    big = np.abs(g) >= 20.0
    frac = big.mean()
    assert 0.007 < frac < 0.013
    assert np.all(np.abs(g[big]) < 100.0)
    assert abs(np.std(g[~big]) - 2.0) < 0.05            # N(0, 4): std 2
    assert abs(np.std(d["UP"]) - 1.0) < 0.02
    assert abs(np.std(d["W"]) - np.sqrt(1e-3)) < 0.02 * np.sqrt(1e-3) * 5


def test_w16_is_round_to_nearest_of_a_float32_draw():
    d = wl.generate("matmul_w16", 4, 64, 32, seed=9, w_var=0.02)
    vals = d["W16"].view(np.float16).astype(np.float64)
    assert np.all(np.isfinite(vals))
    assert abs(np.std(vals) - np.sqrt(0.02)) < 0.03


def test_named_workloads():
    names = [w.name for w in wl.WORKLOADS]
    assert len(set(names)) == 5
    w5 = wl.WORKLOADS_BY_NAME["ffn_down_swiglu_w16_16k"]
    assert (w5.M, w5.N, w5.K) == (16384, 2048, 8192) and w5.seed == 1005
    assert w5.flops == 549755813888
    assert wl.input_bytes(w5.form, w5.M, w5.N, w5.K) == 1375731712
    w1 = wl.WORKLOADS[0]
    assert wl.input_bytes(w1.form, w1.M, w1.N, w1.K) == 5505024
