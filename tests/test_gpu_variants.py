"""Discretisation and parameterisation variants on the GPU against the float64 oracle:
S5 with the bilinear transform (s5_layer_ex; "The Annotated S4", part 1), S5 with a step that
changes from step to step (s5_layer_tv; "Simplified State Space Layers for Sequence Modeling",
sections 2.2 and 6.3), DSS_exp mapped onto the DLR and the decay-rate reparameterisations
("Simplifying and Understanding State Space Models with Diagonal Linear RNNs", section 2; the
StableSSM discussion). Float32 paths: relative L2 <= 1e-5; the bf16 tensor-core tier <= 1e-2,
on y and on its state part y - D u.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_gb300 import dlr, inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5
TOL_BF16 = 1e-2


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().astype(np.float64)


def s5_args(p):
    return p.lam, p.log_delta, p.Bt, p.Ct, p.D


def state_part(y, u, D):
    return np.asarray(y, np.float64) - np.asarray(u, np.float64) * np.asarray(D, np.float64)


@pytest.mark.parametrize("B,L,H,P", [(1, 1, 32, 32), (2, 1000, 96, 64), (1, 300, 512, 256),
                                     (2, 640, 96, 64)])
def test_s5_bilinear_matches_oracle(B, L, H, P):
    w = inputs.make_s5(B, L, H, P, seed=3 * B + L + H + P)
    a = s5_args(w.params)
    ref = oracle.s5_layer(w.u, *a, disc="bilinear")
    y = host(dlr.s5_layer_ex(dev(w.u), *(dev(x) for x in a), disc="bilinear"))
    assert oracle.rel_l2(y, ref) <= TOL
    yb = host(dlr.s5_layer_ex(dev(w.u), *(dev(x) for x in a), prec="bf16", disc="bilinear"))
    D = w.params.D
    assert oracle.rel_l2(yb, ref) <= TOL_BF16
    assert oracle.rel_l2(state_part(yb, w.u, D), state_part(ref, w.u, D)) <= TOL_BF16
    assert dlr.device_status() == 0


def test_s5_ex_zoh_is_s5_layer():
    w = inputs.make_s5(2, 500, 64, 32, seed=5)
    args = [dev(x) for x in s5_args(w.params)]
    u = dev(w.u)
    for prec in ("fp32", "bf16"):
        y0 = dlr.s5_layer(u, *args, prec=prec)
        y1 = dlr.s5_layer_ex(u, *args, prec=prec, disc="zoh")
        assert torch.equal(y0, y1), prec


def test_s5_bilinear_workload_sampled_batch_row():
    """The S5 workload (B8 L16384 H512 P256) with the bilinear transform, one batch row
    checked against the oracle."""
    w = inputs.make_workload("s5_b8_l16384_h512_p256")
    a = s5_args(w.params)
    y = host(dlr.s5_layer_ex(dev(w.u), *(dev(x) for x in a), disc="bilinear"))
    ref = oracle.s5_layer(w.u[5:6], *a, disc="bilinear")
    assert oracle.rel_l2(y[5:6], ref) <= TOL
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("B,L,H,P", [(1, 1, 32, 32), (2, 100, 32, 32), (3, 1000, 96, 64),
                                     (1, 4097, 64, 256), (2, 640, 128, 128)])
def test_s5_time_varying_matches_oracle(B, L, H, P):
    """Irregular gaps (sorted uniform observation times); ragged last chunks."""
    w = inputs.make_s5(B, L, H, P, seed=11 * B + L + H + P)
    dt = inputs.irregular_gaps(np.random.default_rng(L + P), B, L)
    a = s5_args(w.params)
    y = host(dlr.s5_layer_tv(dev(w.u), dev(dt), *(dev(x) for x in a)))
    ref = oracle.s5_layer_tv(w.u, dt, *a)
    assert oracle.rel_l2(y, ref) <= TOL
    D = w.params.D
    assert oracle.rel_l2(state_part(y, w.u, D), state_part(ref, w.u, D)) <= TOL
    assert dlr.device_status() == 0


def test_s5_time_varying_unit_gaps_equal_the_layer():
    w = inputs.make_s5(2, 777, 64, 64, seed=13)
    a = [dev(x) for x in s5_args(w.params)]
    u = dev(w.u)
    y_tv = host(dlr.s5_layer_tv(u, torch.ones((2, 777), dtype=torch.float32, device="cuda"), *a))
    y = host(dlr.s5_layer(u, *a))
    assert oracle.rel_l2(y_tv, y) <= TOL


def test_s5_time_varying_workload_sampled_batch_row():
    """The S5 workload's shapes with irregular gaps, one batch row against the oracle."""
    w = inputs.make_workload("s5_b8_l16384_h512_p256")
    dt = inputs.irregular_gaps(np.random.default_rng(3), w.B, w.L)
    a = s5_args(w.params)
    y = host(dlr.s5_layer_tv(dev(w.u), dev(dt), *(dev(x) for x in a)))
    ref = oracle.s5_layer_tv(w.u[1:2], dt[1:2], *a)
    assert oracle.rel_l2(y[1:2], ref) <= TOL
    D = w.params.D
    assert oracle.rel_l2(state_part(y[1:2], w.u[1:2], D), state_part(ref, w.u[1:2], D)) <= TOL
    assert np.all(np.isfinite(y))


def test_dss_exp_mapped_layer_matches_its_definition():
    """DSS_exp parameters mapped on the GPU equal the oracle's map, and the DLR layer run on
    them (the tensor-core scan) equals the DSS_exp recurrence by its definition."""
    rng = np.random.default_rng(21)
    B, H, N, L = 2, 4, 64, 1000
    Lam = np.stack([-rng.uniform(1e-3, 0.5, (H, N)), rng.uniform(-3, 3, (H, N))], -1)
    ld = rng.uniform(np.log(1e-3), np.log(0.1), H)
    W = rng.standard_normal((H, N, 2)) / N
    f32 = lambda x: np.asarray(x, np.float32)
    Lam, ld, W = f32(Lam), f32(ld), f32(W)
    u = rng.standard_normal((B, H, L)).astype(np.float32)
    lr, li, Wo = dlr.dlr_params_from_dss_exp(dev(Lam), dev(ld), dev(W))
    r_lr, r_li, r_W = oracle.dss_exp_params(Lam, ld, W)
    assert oracle.rel_l2(host(lr), r_lr) <= 1e-6
    assert oracle.rel_l2(host(li), r_li) <= 1e-6
    assert oracle.rel_l2(host(Wo), r_W) <= 1e-6
    y = host(dlr.dlr_scan(dev(u), (lr, li, Wo), algo="tensor"))
    assert oracle.rel_l2(y, oracle.dss_exp_layer(u, Lam, ld, W)) <= TOL
    assert dlr.device_status() == 0


def test_dss_exp_growing_mode_is_reported():
    """Re Lambda > 0 cannot be held by |lambda| <= 1: mapped to |lambda| = 1 and reported."""
    Lam = np.array([[[0.2, 1.0], [-0.1, 0.5]]], np.float32)
    ld = np.array([np.log(0.1)], np.float32)
    W = np.ones((1, 2, 2), np.float32)
    lr, _, _ = dlr.dlr_params_from_dss_exp(dev(Lam), dev(ld), dev(W))
    assert host(lr)[0, 0] == 0.0
    assert dlr.device_status() == 1   # DLR_ERR_INVALID_ARG, then cleared
    assert dlr.device_status() == 0


@pytest.mark.parametrize("kind", ["exp", "softplus", "best"])
def test_reparam_maps_match_oracle(kind):
    w = np.linspace(-6, 6, 1001).astype(np.float32)
    lr = host(dlr.dlr_log_re_from_reparam(dev(w), kind, a=0.5, b=2.0))
    assert oracle.rel_l2(lr, oracle.reparam_log_re(w, kind, 0.5, 2.0)) <= 1e-6
