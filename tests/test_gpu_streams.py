"""Every call runs in order on the caller's stream: the inputs are written on a side stream
behind a ~10 ms device sleep, the call is enqueued on that stream, and its outputs must equal
the results of the same call on inputs that were ready. A launch on any other stream would read
the inputs before they are written."""
import numpy as np
import pytest
import torch

from state_space_sequence_gb300 import dlr, inputs

pytestmark = pytest.mark.gpu

SLEEP_CYCLES = 20_000_000  # about 10 ms at 2 GHz


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def late_copies(s, *srcs):
    """Copies of srcs that become valid on stream s only after a device sleep."""
    outs = [torch.zeros_like(t) for t in srcs]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(SLEEP_CYCLES)
        for o, t in zip(outs, srcs):
            o.copy_(t)
    return outs


def check(ref, got, s):
    assert not s.query()  # the call was enqueued while its inputs were still being written
    s.synchronize()
    ref = ref if isinstance(ref, (list, tuple)) else [ref]
    got = got if isinstance(got, (list, tuple)) else [got]
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    assert dlr.device_status() == 0


def test_kernel_conv_scan_on_the_callers_stream():
    w = inputs.make_dlr(2, 3, 32, 1000, seed=4, bidir=True, unit_channels=1)
    f = [dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W)]
    b = [dev(a) for a in (w.bwd.log_re, w.bwd.log_im, w.bwd.W)]
    u = dev(w.u)
    K_ref = dlr.dlr_kernel(*f, 1000)
    y_conv = dlr.dlr_conv(u, K_ref)
    y_scan = dlr.dlr_scan(u, f, b)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    fl = late_copies(s, *f)
    K = dlr.dlr_kernel(*fl, 1000, stream=s)
    check(K_ref, K, s)
    (ul,) = late_copies(s, u)
    check(y_conv, dlr.dlr_conv(ul, K_ref, stream=s), s)
    fl, bl, (ul,) = late_copies(s, *f), late_copies(s, *b), late_copies(s, u)
    check(y_scan, dlr.dlr_scan(ul, fl, bl, stream=s), s)


def test_gradients_on_the_callers_stream():
    w = inputs.make_dlr(2, 2, 24, 700, seed=6, bidir=True, unit_channels=1)
    f = [dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W)]
    b = [dev(a) for a in (w.bwd.log_re, w.bwd.log_im, w.bwd.W)]
    u = dev(w.u)
    g = dev(np.random.default_rng(2).standard_normal(w.u.shape).astype(np.float32))
    p_ref = dlr.dlr_scan_backward_params(u, g, f)
    du_ref, gr_ref = dlr.dlr_layer_backward(u, g, f, b, cast="re_im")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    ul, gl = late_copies(s, u, g)
    check(list(p_ref), list(dlr.dlr_scan_backward_params(ul, gl, f, stream=s)), s)
    ul, gl = late_copies(s, u, g)
    du, gr = dlr.dlr_layer_backward(ul, gl, f, b, cast="re_im", stream=s)
    check([du_ref] + [t for x in gr_ref for t in x], [du] + [t for x in gr for t in x], s)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_s5_on_the_callers_stream(prec):
    w = inputs.make_s5(2, 256, 64, 32, seed=8)
    p = w.params
    a = [dev(x) for x in (p.lam, p.log_delta, p.Bt, p.Ct, p.D)]
    u = dev(w.u)
    y_ref = dlr.s5_layer(u, *a, prec=prec)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    (ul,) = late_copies(s, u)
    check(y_ref, dlr.s5_layer(ul, *a, prec=prec, stream=s), s)


def test_step_on_the_callers_stream():
    w = inputs.make_dlr(2, 3, 16, 40, seed=10, unit_channels=1)
    f = [dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W)]
    u = dev(w.u)
    tab = dlr.dlr_step_prepare(f)
    x0 = torch.zeros((2, 3, 16, 2), dtype=torch.float32, device="cuda")
    y_ref = dlr.dlr_step(u, tab, x0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    ul, = late_copies(s, u)
    x1 = torch.zeros_like(x0)
    check(y_ref, dlr.dlr_step(ul, tab, x1, stream=s), s)
    assert torch.equal(x0, x1)


def test_concurrent_calls_on_two_streams():
    """Calls on two streams with their own workspaces run at the same time without sharing
    state: the tensor-core scan on one, the DLR-prod gradients (tensor-core generator and power
    sums, FFT convolutions) on the other, each equal to the same call run alone."""
    w = inputs.make_dlr(4, 16, 64, 4096, seed=12, unit_channels=1)
    f = [dev(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W)]
    u = dev(w.u)
    wp = inputs.make_dlr(2, 8, 256, 2048, seed=13, bidir=True, unit_channels=1)
    fp = [dev(a) for a in (wp.fwd.log_re, wp.fwd.log_im, wp.fwd.W)]
    bp = [dev(a) for a in (wp.bwd.log_re, wp.bwd.log_im, wp.bwd.W)]
    up = dev(wp.u)
    gp = dev(np.random.default_rng(3).standard_normal(wp.u.shape).astype(np.float32))
    y_ref = dlr.dlr_scan(u, f)
    du_ref, gr_ref = dlr.dlr_layer_backward(up, gp, fp, bp, cast="re_im")
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = torch.empty(dlr.dlr_scan_workspace_size(4, 16, 64, 4096), dtype=torch.uint8,
                      device="cuda")
    ws2 = torch.empty(dlr.dlr_layer_backward_workspace_size(2, 8, 256, 2048, True, "re_im"),
                      dtype=torch.uint8, device="cuda")
    ys, outs = [], []
    for _ in range(3):
        ys.append(dlr.dlr_scan(u, f, workspace=ws1, stream=s1))
        outs.append(dlr.dlr_layer_backward(up, gp, fp, bp, cast="re_im", workspace=ws2,
                                           stream=s2))
        s1.synchronize()
        s2.synchronize()
    for y, (du, gr) in zip(ys, outs):
        assert torch.equal(y, y_ref) and torch.equal(du, du_ref)
        for a, b in zip([t for x in gr for t in x], [t for x in gr_ref for t in x]):
            assert torch.equal(a, b)
    assert dlr.device_status() == 0
