"""Cases for the bounds-checked build, run in a child process with DLR_BOUNDS_CHECK=1 (the
binding then loads libdlr_checked.so): every entry point on small, ragged shapes that reach the
kernels' tail paths, each result checked against the float64 oracle, and after each call the
device status and the first failing site of the index checks. Prints one JSON line:
{"checked": bool, "cases": [[name, rel_l2, status, site], ...], "selftest": [status, site]}.
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from state_space_sequence_gb300 import dlr, inputs  # noqa: E402


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().astype(np.float64)


def pdev(p):
    return dev(p.log_re), dev(p.log_im), dev(p.W)


def pnp(p):
    return p.log_re, p.log_im, p.W


def run():
    cases = []

    def record(name, got, ref):
        err = float(oracle.rel_l2(got, ref)) if ref is not None else 0.0
        cases.append([name, err, int(dlr.device_status()), int(dlr.bounds_site())])

    # kernel generation: FFMA (few states), tensor cores (many states; long rows)
    for H, N, L in [(3, 5, 1000), (2, 300, 5000), (2, 64, 20000)]:
        w = inputs.make_dlr(1, H, N, 1, seed=H + N + L, unit_channels=1)
        for cast in ("re", "re_im"):
            K = host(dlr.dlr_kernel(*pdev(w.fwd), L, cast))
            record(f"kernel H{H} N{N} L{L} {cast}", K, oracle.dlr_kernel(*pnp(w.fwd), L, cast=cast))

    # FFT convolution: one CTA per row (odd and even rows), pairs of rows, the 8-CTA cluster
    for B, H, N, L, bidir in [(3, 2, 16, 1000, False), (2, 2, 8, 999, True), (2, 3, 16, 4096, False),
                              (1, 2, 8, 20000, True), (3, 1, 4, 7, True)]:
        w = inputs.make_dlr(B, H, N, L, seed=B * 7 + L, bidir=bidir, unit_channels=1)
        y = host(dlr.dlr_layer(dev(w.u), pdev(w.fwd), pdev(w.bwd) if bidir else None, path="fft"))
        record(f"fft B{B} H{H} L{L} bidir={bidir}", y,
               oracle.dlr_layer(w.u, pnp(w.fwd), pnp(w.bwd) if bidir else None))
    # the DLR-prod cast
    w = inputs.make_dlr(2, 2, 8, 500, seed=5, bidir=True, unit_channels=1)
    y = host(dlr.dlr_layer(dev(w.u), pdev(w.fwd), pdev(w.bwd), cast="re_im", path="fft"))
    record("fft prod bidir", y, oracle.dlr_layer(w.u, pnp(w.fwd), pnp(w.bwd), cast="re_im"))

    # the direct spectrum route
    for H, N, L in [(2, 16, 3000), (1, 8, 20000)]:
        w = inputs.make_dlr(2, H, N, L, seed=H + L, unit_channels=1)
        ws = dlr.dlr_conv_spectrum_direct(pdev(w.fwd), None, L=L)
        y = host(dlr.dlr_conv_apply(dev(w.u), ws))
        record(f"direct spectrum H{H} L{L}", y, oracle.dlr_layer(w.u, pnp(w.fwd)))

    # scans: tensor cores (ragged rows, long rows walked tile by tile, bidirectional) and
    # float32 (more states)
    for B, H, N, L, bidir, algo in [(3, 2, 64, 1000, False, "tensor"), (1, 1, 33, 20000, False, "tensor"),
                                    (2, 2, 16, 700, True, "tensor"), (2, 1, 100, 700, False, "fp32")]:
        w = inputs.make_dlr(B, H, N, L, seed=B + H + N + L, bidir=bidir, unit_channels=1)
        y = host(dlr.dlr_scan(dev(w.u), pdev(w.fwd), pdev(w.bwd) if bidir else None, algo=algo))
        record(f"scan {algo} B{B} N{N} L{L} bidir={bidir}", y,
               oracle.dlr_layer(w.u, pnp(w.fwd), pnp(w.bwd) if bidir else None))

    # the host-buffer entry point
    w = inputs.make_dlr(5, 2, 16, 300, seed=9, unit_channels=1)
    u_h = torch.from_numpy(np.ascontiguousarray(w.u)).pin_memory()
    y_h = torch.empty_like(u_h).pin_memory()
    p_h = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in pnp(w.fwd)]
    ws_h = torch.empty(dlr.dlr_scan_host_workspace_size(5, 2, 16, 300), dtype=torch.uint8,
                       device="cuda")
    dlr.dlr_scan_host(u_h, p_h, y_h, ws_h)
    torch.cuda.synchronize()
    record("scan host buffers", y_h.numpy().astype(np.float64), oracle.dlr_layer(w.u, pnp(w.fwd)))

    # recurrent mode from a carried state
    w = inputs.make_dlr(2, 3, 16, 37, seed=3, unit_channels=1)
    wss = dlr.dlr_step_prepare(pdev(w.fwd))
    x = torch.zeros((2, 3, 16, 2), dtype=torch.float32, device="cuda")
    y = host(dlr.dlr_step(dev(w.u), wss, x))
    record("step T37", y, oracle.dlr_layer(w.u, pnp(w.fwd)))

    # backward pass
    w = inputs.make_dlr(2, 2, 16, 300, seed=13, unit_channels=1)
    g = np.random.default_rng(1).standard_normal(w.u.shape).astype(np.float32)
    du = host(dlr.dlr_scan_backward_input(dev(g), pdev(w.fwd)))
    r_du, r_re, r_im, r_W = oracle.dlr_backward(w.u, g, *pnp(w.fwd))
    record("backward input", du, r_du)
    d_lr, d_li, dW = dlr.dlr_scan_backward_params(dev(w.u), dev(g), pdev(w.fwd))
    got = np.concatenate([host(d_lr).ravel(), host(d_li).ravel(), host(dW).ravel()])
    record("backward parameters", got, np.concatenate([r_re.ravel(), r_im.ravel(), r_W.ravel()]))
    # the recurrence route (few states) and the correlation route's largest transform
    for B, H, N, L in [(2, 2, 8, 300), (1, 1, 18, 8000), (2, 1, 70, 700)]:
        w = inputs.make_dlr(B, H, N, L, seed=N + L, unit_channels=1)
        g = np.random.default_rng(N).standard_normal(w.u.shape).astype(np.float32)
        _, r_re, r_im, r_W = oracle.dlr_backward(w.u, g, *pnp(w.fwd))
        d_lr, d_li, dW = dlr.dlr_scan_backward_params(dev(w.u), dev(g), pdev(w.fwd))
        got = np.concatenate([host(d_lr).ravel(), host(d_li).ravel(), host(dW).ravel()])
        record(f"backward parameters N{N} L{L}", got,
               np.concatenate([r_re.ravel(), r_im.ravel(), r_W.ravel()]))

    # the layer's gradients: both directions, both casts, both routes
    for bidir, cast, B, H, N, L in [(True, "re", 2, 2, 16, 300), (True, "re", 2, 1, 8, 300),
                                    (True, "re_im", 2, 2, 20, 500), (False, "re_im", 1, 1, 8, 33)]:
        w = inputs.make_dlr(B, H, N, L, seed=N + L, bidir=bidir, unit_channels=1)
        g = np.random.default_rng(L).standard_normal(w.u.shape).astype(np.float32)
        bwd = pnp(w.bwd) if bidir else None
        du, grads = dlr.dlr_layer_backward(dev(w.u), dev(g), pdev(w.fwd),
                                           pdev(w.bwd) if bidir else None, cast=cast)
        r_du, r_grads = oracle.dlr_layer_backward(w.u, g, pnp(w.fwd), bwd, cast=cast)
        record(f"layer backward du {cast} bidir={bidir} N{N} L{L}", host(du), r_du)
        for d, (gr, rg) in enumerate(zip(grads, r_grads)):
            got = np.concatenate([host(t).ravel() for t in gr])
            record(f"layer backward grads {d} {cast} bidir={bidir} N{N} L{L}", got,
                   np.concatenate([t.ravel() for t in rg]))

    # S5: float32 and bf16 tiers (L a multiple of 64 takes the fused output projection),
    # bilinear, a step that changes from step to step
    for B, L, H, P in [(2, 63, 32, 32), (1, 128, 64, 32)]:
        s = inputs.make_s5(B, L, H, P, seed=B + L)
        p = s.params
        args = (dev(p.lam), dev(p.log_delta), dev(p.Bt), dev(p.Ct), dev(p.D))
        ref = oracle.s5_layer(s.u, p.lam, p.log_delta, p.Bt, p.Ct, p.D)
        record(f"s5 fp32 L{L}", host(dlr.s5_layer(dev(s.u), *args)), ref)
        record(f"s5 bf16 L{L}", host(dlr.s5_layer(dev(s.u), *args, prec="bf16")), ref)
        refb = oracle.s5_layer(s.u, p.lam, p.log_delta, p.Bt, p.Ct, p.D, disc="bilinear")
        record(f"s5 bilinear L{L}", host(dlr.s5_layer_ex(dev(s.u), *args, disc="bilinear")), refb)
        dt = inputs.irregular_gaps(np.random.default_rng(L), B, L)
        reft = oracle.s5_layer_tv(s.u, dt, p.lam, p.log_delta, p.Bt, p.Ct, p.D)
        record(f"s5 time-varying L{L}", host(dlr.s5_layer_tv(dev(s.u), dev(dt), *args)), reft)

    # parameter maps
    rng = np.random.default_rng(2)
    Lam = np.stack([-rng.uniform(0.01, 1.0, (2, 5)), rng.uniform(-3, 3, (2, 5))], -1).astype(np.float32)
    ld = rng.uniform(np.log(0.01), np.log(0.5), 2).astype(np.float32)
    W = rng.standard_normal((2, 5, 2)).astype(np.float32)
    lr, li, Wo = dlr.dlr_params_from_dss_exp(dev(Lam), dev(ld), dev(W))
    rlr, rli, rW = oracle.dss_exp_params(Lam, ld, W)
    record("dss_exp map", np.concatenate([host(lr).ravel(), host(li).ravel(), host(Wo).ravel()]),
           np.concatenate([rlr.ravel(), rli.ravel(), rW.ravel()]))
    wv = rng.standard_normal(37).astype(np.float32)
    record("reparam softplus", host(dlr.dlr_log_re_from_reparam(dev(wv), "softplus")),
           oracle.reparam_log_re(wv, "softplus"))

    dlr.selftest_bounds()
    selftest = [int(dlr.device_status()), int(dlr.bounds_site())]
    return {"checked": dlr.bounds_checked(), "library": dlr.library_path(), "cases": cases,
            "selftest": selftest}


if __name__ == "__main__":
    print(json.dumps(run()))
