"""No result depends on what the caller's workspace held before the call: every entry point
that takes a workspace runs once on a zero-filled and once on an all-ones-bits workspace (each
float32 word a NaN), and the outputs must be bit-identical and finite. A read of a workspace
word before the call writes it would show up as a NaN or as a difference."""
import numpy as np
import pytest
import torch

from state_space_sequence_gb300 import dlr, inputs

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def ws_pair(nbytes):
    z = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    f = torch.full((max(nbytes, 1),), 255, dtype=torch.uint8, device="cuda")
    return z, f


def same(run, nbytes):
    z, f = ws_pair(nbytes)
    a = run(z)
    b = run(f)
    torch.cuda.synchronize()
    a = a if isinstance(a, (list, tuple)) else [a]
    b = b if isinstance(b, (list, tuple)) else [b]
    assert len(a) == len(b)
    for x, y in zip(a, b):
        assert torch.isfinite(x).all()
        assert torch.equal(x, y)
    assert dlr.device_status() == 0


@pytest.mark.parametrize("B,H,L,bidir", [(2, 3, 1000, False), (3, 2, 700, True),
                                         (1, 2, 20000, True)])
def test_conv(B, H, L, bidir):
    w = inputs.make_dlr(B, H, 16, L, seed=L + B, bidir=bidir, unit_channels=1)
    K1 = dlr.dlr_kernel(dev(w.fwd.log_re), dev(w.fwd.log_im), dev(w.fwd.W), L)
    K2 = dlr.dlr_kernel(dev(w.bwd.log_re), dev(w.bwd.log_im), dev(w.bwd.W), L) if bidir else None
    u = dev(w.u)
    same(lambda ws: dlr.dlr_conv(u, K1, K2, workspace=ws), dlr.dlr_conv_workspace_size(H, L, bidir))


@pytest.mark.parametrize("B,H,N,L,bidir", [(3, 5, 33, 1000, False), (2, 2, 64, 4096, True),
                                           (1, 3, 16, 9000, False)])
def test_scan(B, H, N, L, bidir):
    w = inputs.make_dlr(B, H, N, L, seed=N + L, bidir=bidir, unit_channels=1)
    f = tuple(dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    b = tuple(dev(a) for a in (w.bwd.log_re, w.bwd.log_im, w.bwd.W)) if bidir else None
    u = dev(w.u)
    same(lambda ws: dlr.dlr_scan(u, f, b, workspace=ws), dlr.dlr_scan_workspace_size(B, H, N, L))


@pytest.mark.parametrize("B,H,N,L", [(2, 3, 32, 1000), (2, 2, 8, 500), (1, 2, 20, 9000)])
def test_backward_params(B, H, N, L):
    w = inputs.make_dlr(B, H, N, L, seed=3 * N + L, unit_channels=1)
    f = tuple(dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    u = dev(w.u)
    g = dev(np.random.default_rng(L).standard_normal(w.u.shape).astype(np.float32))
    same(lambda ws: dlr.dlr_scan_backward_params(u, g, f, workspace=ws),
         dlr.dlr_scan_backward_params_workspace_size(B, H, N, L))


@pytest.mark.parametrize("cast,bidir,L", [("re_im", True, 700), ("re", True, 20000),
                                          ("re_im", False, 300)])
def test_layer_backward(cast, bidir, L):
    w = inputs.make_dlr(2, 2, 24, L, seed=L + 1, bidir=bidir, unit_channels=1)
    f = tuple(dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    b = tuple(dev(a) for a in (w.bwd.log_re, w.bwd.log_im, w.bwd.W)) if bidir else None
    u = dev(w.u)
    g = dev(np.random.default_rng(L).standard_normal(w.u.shape).astype(np.float32))

    def run(ws):
        du, grads = dlr.dlr_layer_backward(u, g, f, b, cast=cast, workspace=ws)
        return [du] + [t for gr in grads for t in gr]
    same(run, dlr.dlr_layer_backward_workspace_size(2, 2, 24, L, bidir, cast))


@pytest.mark.parametrize("prec,L", [("fp32", 256), ("bf16", 256), ("bf16", 200)])
def test_s5(prec, L):
    s = inputs.make_s5(2, L, 64, 32, seed=L)
    p = s.params
    a = [dev(x) for x in (p.lam, p.log_delta, p.Bt, p.Ct, p.D)]
    u = dev(s.u)
    same(lambda ws: dlr.s5_layer(u, *a, prec=prec, workspace=ws),
         dlr.s5_workspace_size(2, L, 64, 32, prec))


def test_s5_time_varying():
    s = inputs.make_s5(2, 300, 64, 32, seed=5)
    p = s.params
    a = [dev(x) for x in (p.lam, p.log_delta, p.Bt, p.Ct, p.D)]
    dt = dev(inputs.irregular_gaps(np.random.default_rng(1), 2, 300))
    u = dev(s.u)
    nbytes = int(dlr._load().s5_layer_tv_workspace_size(2, 300, 64, 32))
    same(lambda ws: dlr.s5_layer_tv(u, dt, *a, workspace=ws), nbytes)


def test_scan_host_buffers():
    w = inputs.make_dlr(4, 3, 32, 1024, seed=9, unit_channels=1)
    u_h = torch.from_numpy(w.u).pin_memory()
    p_h = tuple(torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))

    def run(ws):
        y = torch.empty(u_h.shape, dtype=torch.float32).pin_memory()
        dlr.dlr_scan_host(u_h, p_h, y, ws)
        torch.cuda.synchronize()
        return y.cuda()
    same(run, dlr.dlr_scan_host_workspace_size(4, 3, 32, 1024))
