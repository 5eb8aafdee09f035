"""The seeded input generator against the workload recipes it stands for: shapes, seeds and the
distributions of the DLR initialisation ("Simplifying and Understanding State Space Models with
Diagonal Linear RNNs", section 2.2: (log Lambda)_re = sqrt(e^r / 2) with r uniform on
[log 5e-4, log 0.5], (log Lambda)_im = 2 pi n / N, Re and Im of W with variance 1 / N^2; section
3.1: inputs divided by their largest magnitude) and of the S5 initialisation ("Simplified State
Space Layers for Sequence Modeling", sections 3 and 4.3: HiPPO-N eigenvalues, a timescale Delta
per state, log-uniform on [1e-3, 1e-1])."""
import numpy as np
import pytest
import scipy.stats

from state_space_sequence_gb300 import inputs


@pytest.mark.parametrize("name", ["dlr_b1_h1_n16_l256", "dlr_b8_h256_n64_l4096",
                                  "dlr_b1_h256_n64_l65536_unit8"])
def test_dlr_workloads_shapes_and_seeds(name):
    cfg = inputs.WORKLOADS[name]
    w = inputs.make_workload(name)
    assert w.u.shape == (cfg["B"], cfg["H"], cfg["L"]) and w.u.dtype == np.float32
    assert w.fwd.log_re.shape == (cfg["H"], cfg["N"]) and w.fwd.W.shape == (cfg["H"], cfg["N"], 2)
    again = inputs.make_workload(name)
    assert np.array_equal(w.u, again.u) and np.array_equal(w.fwd.W, again.fwd.W)
    assert (w.bwd is None) == (not cfg["bidir"])


def test_dlr_init_distribution():
    p = inputs.dlr_params(np.random.default_rng(5), 256, 64)
    a = p.log_re.astype(np.float64)
    r = np.log(2.0 * a * a)  # inverts (log Lambda)_re = sqrt(e^r / 2)
    lo, hi = np.log(5e-4), np.log(0.5)
    assert r.min() >= lo - 1e-5 and r.max() <= hi + 1e-5
    assert scipy.stats.kstest((r.ravel() - lo) / (hi - lo), "uniform").pvalue > 1e-3
    np.testing.assert_allclose(p.log_im, np.broadcast_to(2 * np.pi * np.arange(64) / 64,
                                                         (256, 64)), rtol=1e-6)
    for c in range(2):  # Re and Im of W: mean 0, variance 1 / N^2
        x = p.W[..., c].astype(np.float64).ravel() * 64
        assert abs(x.mean()) < 0.03 and abs(x.var() - 1.0) < 0.05


def test_dlr_inputs_normalised_where_the_recipe_says():
    w0 = inputs.make_workload("dlr_b1_h1_n16_l256")
    np.testing.assert_allclose(np.abs(w0.u).max(axis=-1), 1.0, rtol=0, atol=0)
    u = inputs.dlr_input(np.random.default_rng(6), 4, 8, 16384, normalize=True)
    np.testing.assert_array_equal(np.abs(u).max(axis=-1), np.ones((4, 8), np.float32))
    w1 = inputs.make_workload("dlr_b8_h256_n64_l4096")  # raw N(0, 1)
    x = w1.u.astype(np.float64).ravel()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_unit_circle_channels():
    p = inputs.dlr_params(np.random.default_rng(7), 256, 64, unit_channels=8)
    assert np.all(p.log_re[:8] == 0.0) and np.all(p.log_re[8:] > 0.0)


def test_s5_init_distribution():
    H, P = 512, 256
    p = inputs.s5_params(np.random.default_rng(8), H, P)
    np.testing.assert_array_equal(p.lam, inputs.hippo_n_eigenvalues(P).astype(np.float32))
    ld = p.log_delta.astype(np.float64)
    lo, hi = np.log(1e-3), np.log(1e-1)
    assert ld.min() >= lo - 1e-6 and ld.max() <= hi + 1e-6
    assert scipy.stats.kstest((ld - lo) / (hi - lo), "uniform").pvalue > 1e-3
    for arr in (p.Bt, p.Ct):  # Re and Im with variance 1 / H
        for c in range(2):
            x = arr[..., c].astype(np.float64).ravel() * np.sqrt(H)
            assert abs(x.mean()) < 0.02 and abs(x.var() - 1.0) < 0.02
    d = p.D.astype(np.float64)
    assert abs(d.mean()) < 0.15 and abs(d.var() - 1.0) < 0.2
