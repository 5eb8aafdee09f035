"""Parameter gradients of the causal DLR layer on the GPU (dlr_scan_backward_params) against the
float64 oracle's gradients, which are written out from the definitions ("Simplifying and
Understanding State Space Models with Diagonal Linear RNNs", section 2, gradient analysis) and
pinned by central differences and the adjoint identity. Relative L2 <= 1e-5 for each of the
three gradient arrays.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_gb300 import dlr, inputs

pytestmark = pytest.mark.gpu

TOL = 1e-5


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,H,N,L", [
    # lag-correlation route (N >= 16, L <= 8192): transforms of M = 2^ceil(log2(2L-1)) points,
    # from M = 1 and 4 up to 16384
    (3, 1, 16, 1), (2, 1, 17, 2), (1, 1, 32, 33), (2, 3, 16, 256), (3, 2, 40, 1000),
    (1, 2, 64, 4096), (4, 3, 33, 777), (2, 1, 100, 3000), (2, 2, 16, 8192), (1, 1, 70, 5000),
    # rows longer than 8192: the correlation through the FFT convolution's kernels (one CTA per
    # row up to 16384, the 8-CTA cluster above)
    (1, 2, 20, 9000), (2, 2, 16, 20000), (1, 1, 24, 65536),
    # recurrence route: few states, rows longer than 65536
    (1, 1, 1, 1), (2, 2, 8, 1000), (1, 1, 2, 9000), (1, 1, 16, 66000)])
def test_backward_params_match_oracle(B, H, N, L):
    """Both routes; ragged L, N not a multiple of 32 or of the four states a warp takes, one
    unit-circle channel (d log_re = 0 there)."""
    w = inputs.make_dlr(B, H, N, L, seed=B * 101 + H * 7 + N + L, unit_channels=1)
    g = np.random.default_rng(L + N).standard_normal((B, H, L)).astype(np.float32)
    p = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    d_re, d_im, dW = dlr.dlr_scan_backward_params(dev(w.u), dev(g), tuple(dev(a) for a in p))
    _, r_re, r_im, r_W = oracle.dlr_backward(w.u, g, *p)
    assert oracle.rel_l2(host(d_re), r_re) <= TOL
    assert oracle.rel_l2(host(d_im), r_im) <= TOL
    assert oracle.rel_l2(host(dW), r_W) <= TOL
    assert dlr.device_status() == 0


def test_backward_params_bank_workload():
    """The bank workload at full size (B8 H256 N64 L4096) with a random output gradient."""
    w = inputs.make_workload("dlr_b8_h256_n64_l4096")
    g = np.random.default_rng(17).standard_normal(w.u.shape).astype(np.float32)
    p = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    d_re, d_im, dW = dlr.dlr_scan_backward_params(dev(w.u), dev(g), tuple(dev(a) for a in p))
    _, r_re, r_im, r_W = oracle.dlr_backward(w.u, g, *p)
    assert oracle.rel_l2(host(d_re), r_re) <= TOL
    assert oracle.rel_l2(host(d_im), r_im) <= TOL
    assert oracle.rel_l2(host(dW), r_W) <= TOL
    assert dlr.device_status() == 0


def test_backward_params_linear_in_g():
    """The gradients are linear in g: g1 + 2 g2 gives grad(g1) + 2 grad(g2)."""
    w = inputs.make_dlr(2, 2, 16, 500, seed=3, unit_channels=1)
    rng = np.random.default_rng(4)
    g1 = rng.standard_normal(w.u.shape).astype(np.float32)
    g2 = rng.standard_normal(w.u.shape).astype(np.float32)
    p = tuple(dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    u = dev(w.u)
    a = dlr.dlr_scan_backward_params(u, dev(g1), p)
    b = dlr.dlr_scan_backward_params(u, dev(g2), p)
    c = dlr.dlr_scan_backward_params(u, dev(g1 + 2 * g2), p)
    for x, y, z in zip(a, b, c):
        ref = host(x) + 2 * host(y)
        assert oracle.rel_l2(host(z), ref) <= 1e-5


@pytest.mark.parametrize("bidir,cast,B,H,N,L", [
    (False, "re", 2, 3, 16, 300),        # correlation route; du by the FFT convolution
    (True, "re", 2, 3, 16, 300),         # both directions: c at positive and negative lags
    (True, "re", 3, 2, 8, 1000),         # recurrence route, the second direction on reversed rows
    (True, "re", 1, 2, 20, 9000),        # recurrence route, rows longer than 8192
    (False, "re_im", 2, 2, 24, 777),     # DLR-prod: weights c_j K_j
    (True, "re_im", 3, 2, 40, 1000),
    (True, "re_im", 1, 1, 8, 8192),      # DLR-prod with few states, the largest transform
    (True, "re", 2, 2, 16, 20000),       # long rows: c through the convolution's kernels
    (True, "re_im", 2, 2, 24, 16384),
    (True, "re_im", 1, 2, 16, 40000),    # ... on the 8-CTA cluster transform
    (True, "re", 2, 1, 4, 20000),        # recurrence route on reversed rows, du on the cluster
])
def test_layer_backward_matches_oracle(bidir, cast, B, H, N, L):
    """dlr_layer_backward against the oracle's dlr_layer_backward: du and the three gradients
    of each direction, causal and bidirectional, Re and DLR-prod casts, both routes."""
    w = inputs.make_dlr(B, H, N, L, seed=B * 13 + N + L + (7 if bidir else 0), bidir=bidir,
                        unit_channels=1)
    g = np.random.default_rng(N + L).standard_normal((B, H, L)).astype(np.float32)
    fwd = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    bwd = (w.bwd.log_re, w.bwd.log_im, w.bwd.W) if bidir else None
    du, grads = dlr.dlr_layer_backward(dev(w.u), dev(g), tuple(dev(a) for a in fwd),
                                       tuple(dev(a) for a in bwd) if bidir else None, cast=cast)
    r_du, r_grads = oracle.dlr_layer_backward(w.u, g, fwd, bwd, cast=cast)
    assert oracle.rel_l2(host(du), r_du) <= TOL
    assert len(grads) == len(r_grads) == (2 if bidir else 1)
    for got, ref in zip(grads, r_grads):
        for a, b in zip(got, ref):
            assert oracle.rel_l2(host(a), b) <= TOL
    assert dlr.device_status() == 0


def test_layer_backward_causal_re_equals_the_scan_gradients():
    """The causal Re-cast case of dlr_layer_backward gives the parameter gradients of
    dlr_scan_backward_params (the same kernels) and, by another route (FFT convolution against
    the tensor-core scan's reversed pass), the input gradient of dlr_scan_backward_input."""
    w = inputs.make_dlr(4, 3, 32, 1500, seed=21, unit_channels=1)
    g = np.random.default_rng(5).standard_normal(w.u.shape).astype(np.float32)
    p = tuple(dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    u, gd = dev(w.u), dev(g)
    du, grads = dlr.dlr_layer_backward(u, gd, p)
    a = dlr.dlr_scan_backward_params(u, gd, p)
    for x, y in zip(grads[0], a):
        assert torch.equal(x, y)
    assert oracle.rel_l2(host(du), host(dlr.dlr_scan_backward_input(gd, p))) <= TOL


def test_layer_backward_dlrprod_workload_sampled_channels():
    """The bidirectional DLR-prod workload at full size (B4 H128 N1024 L16384): all gradients
    on the GPU, compared with the oracle on a seeded sample of channels (the channels are
    independent, so the oracle runs on those channels' slices) and on du of the same
    channels."""
    w = inputs.make_workload("dlrprod_bidir_b4_h128_n1024_l16384")
    g = np.random.default_rng(23).standard_normal(w.u.shape).astype(np.float32)
    fwd = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    bwd = (w.bwd.log_re, w.bwd.log_im, w.bwd.W)
    du, grads = dlr.dlr_layer_backward(dev(w.u), dev(g), tuple(dev(a) for a in fwd),
                                       tuple(dev(a) for a in bwd), cast="re_im")
    assert dlr.device_status() == 0
    hs = np.sort(np.random.default_rng(3).choice(w.H, 4, replace=False))
    sl = lambda p: tuple(np.ascontiguousarray(a[hs]) for a in p)
    r_du, r_grads = oracle.dlr_layer_backward(np.ascontiguousarray(w.u[:, hs]),
                                              np.ascontiguousarray(g[:, hs]), sl(fwd), sl(bwd),
                                              cast="re_im")
    assert oracle.rel_l2(host(du)[:, hs], r_du) <= TOL
    for got, ref in zip(grads, r_grads):
        for a, b in zip(got, ref):
            assert oracle.rel_l2(host(a)[hs], b) <= TOL


@pytest.mark.parametrize("bidir,cast,B,H,N,L", [
    (True, "re", 1, 1, 1, 1), (True, "re_im", 1, 1, 1, 1), (False, "re_im", 2, 1, 1, 2),
    (True, "re", 2, 1, 16, 8192), (True, "re", 2, 1, 16, 8193),        # correlation routes
    (False, "re_im", 1, 1, 20, 16384), (False, "re_im", 1, 1, 20, 16385),  # one CTA / cluster
    (True, "re", 2, 1, 63, 500), (True, "re", 2, 1, 64, 500),          # FFMA / tensor-core sums
    (False, "re_im", 1, 2, 127, 300), (False, "re_im", 1, 2, 128, 300), (True, "re", 1, 1, 129, 300),
])
def test_layer_backward_route_boundaries(bidir, cast, B, H, N, L):
    """dlr_layer_backward at the sizes where its routes change (the correlation by one CTA per
    channel or through the convolution, the convolution on one CTA or eight, the power sums on
    FFMA or on the tensor cores with 128 states per CTA) and at the smallest sizes."""
    w = inputs.make_dlr(B, H, N, L, seed=N * 3 + L, bidir=bidir, unit_channels=1)
    g = np.random.default_rng(N + 2 * L).standard_normal((B, H, L)).astype(np.float32)
    fwd = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    bwd = (w.bwd.log_re, w.bwd.log_im, w.bwd.W) if bidir else None
    du, grads = dlr.dlr_layer_backward(dev(w.u), dev(g), tuple(dev(a) for a in fwd),
                                       tuple(dev(a) for a in bwd) if bidir else None, cast=cast)
    r_du, r_grads = oracle.dlr_layer_backward(w.u, g, fwd, bwd, cast=cast)
    assert oracle.rel_l2(host(du), r_du) <= TOL
    for got, ref in zip(grads, r_grads):
        for a, b in zip(got, ref):
            assert oracle.rel_l2(host(a), b) <= TOL
    assert dlr.device_status() == 0


@pytest.mark.parametrize("bidir,cast", [(True, "re"), (True, "re_im"), (False, "re_im")])
def test_layer_backward_without_input_gradient(bidir, cast):
    """du is optional: with it skipped the parameter gradients are the same bits as with it."""
    w = inputs.make_dlr(2, 2, 24, 600, seed=31, bidir=bidir, unit_channels=1)
    g = dev(np.random.default_rng(2).standard_normal(w.u.shape).astype(np.float32))
    u = dev(w.u)
    fwd = tuple(dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    bwd = tuple(dev(a) for a in (w.bwd.log_re, w.bwd.log_im, w.bwd.W)) if bidir else None
    du, full = dlr.dlr_layer_backward(u, g, fwd, bwd, cast=cast)
    none, part = dlr.dlr_layer_backward(u, g, fwd, bwd, cast=cast, input_grad=False)
    assert none is None and du is not None
    for a, b in zip(full, part):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    assert dlr.device_status() == 0
