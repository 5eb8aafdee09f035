"""The direct spectrum route on the GPU (dlr_conv_spectrum_direct + dlr_conv_apply) against the
float64 oracle: the spectra themselves (the truncated generating function of the kernel at the
roots of unity, "The Annotated S4", part 2) and the layer they give through the FFT
convolution ("Simplifying and Understanding State Space Models with Diagonal Linear RNNs",
sections 2 and 2.1). Relative L2 over the whole tensor <= 1e-5, as for every float32 path.
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
    return t.detach().cpu().numpy()


def pdev(p):
    return dev(p.log_re), dev(p.log_im), dev(p.W)


def pnp(p):
    return p.log_re, p.log_im, p.W


def spectra_from_workspace(ws, H, L):
    """The [H, n + 1] spectra in bin order from the convolution workspace (twiddle tables of n
    and 2n points, each padded to 256 bytes, then the spectra; above n = 2^14 the cluster
    transform's order k = k1 + 8 k2 at k1 * n / 8 + k2)."""
    lg = int(np.ceil(np.log2(L))) if L > 1 else 0
    n = 1 << lg
    off = ((8 * n + 255) // 256) * 256 + ((16 * n + 255) // 256) * 256
    raw = host(ws)[off:off + 8 * H * (n + 1)].view(np.complex64).reshape(H, n + 1)
    if lg > 14:
        k = np.arange(n)
        idx = (k % 8) * (n // 8) + k // 8
        raw = np.concatenate([raw[:, idx], raw[:, n:]], axis=1)
    return np.ascontiguousarray(raw.astype(np.complex128)), n


@pytest.mark.parametrize("H,N,L,bidir", [(2, 16, 256, False), (3, 8, 1000, True),
                                         (4, 64, 4096, False), (2, 64, 4096, True),
                                         (2, 33, 30000, False), (1, 5, 1, False)])
def test_direct_spectrum_matches_oracle(H, N, L, bidir):
    """The spectra in the workspace equal the oracle's geometric-series spectra scaled by
    1 / (4n); unit-circle channels put bins on poles of the series."""
    w = inputs.make_dlr(1, H, N, 1, seed=H + 7 * N + L, bidir=bidir, unit_channels=1)
    bwd = pdev(w.bwd) if bidir else None
    ws = dlr.dlr_conv_spectrum_direct(pdev(w.fwd), bwd, L=L)
    S, n = spectra_from_workspace(ws, H, L)
    ref = oracle.dlr_spectrum(*pnp(w.fwd), L, 2 * n, bwd=pnp(w.bwd) if bidir else None)
    ref = np.ascontiguousarray(ref / (4.0 * n))
    assert oracle.rel_l2(S.view(np.float64), ref.view(np.float64)) <= TOL
    assert dlr.device_status() == 0


@pytest.mark.parametrize("B,H,N,L,bidir", [(3, 4, 16, 256, False), (2, 3, 64, 4096, True),
                                           (5, 2, 40, 3000, False), (1, 3, 64, 20000, True),
                                           (2, 2, 8, 7, True)])
def test_direct_spectrum_layer_matches_oracle(B, H, N, L, bidir):
    """dlr_conv_spectrum_direct + dlr_conv_apply = the DLR layer (causal or bidirectional)."""
    w = inputs.make_dlr(B, H, N, L, seed=B * 31 + H + N + L, bidir=bidir, unit_channels=1)
    bwd = pdev(w.bwd) if bidir else None
    ws = dlr.dlr_conv_spectrum_direct(pdev(w.fwd), bwd, L=L)
    y = host(dlr.dlr_conv_apply(dev(w.u), ws)).astype(np.float64)
    ref = oracle.dlr_layer(w.u, pnp(w.fwd), pnp(w.bwd) if bidir else None)
    assert oracle.rel_l2(y, ref) <= TOL
    assert dlr.device_status() == 0


@pytest.mark.parametrize("name", ["dlr_b8_h256_n64_l4096", "dlr_b1_h256_n64_l65536_unit8"])
def test_direct_spectrum_workloads(name):
    """The bank and the long unit-circle workload at full size: the direct route's layer
    against the oracle, and against the kernel route's layer (pairwise)."""
    w = inputs.make_workload(name)
    B, H, L = w.u.shape
    u = dev(w.u)
    fwd = pdev(w.fwd)
    ws = dlr.dlr_conv_spectrum_direct(fwd, None, L=L)
    y = host(dlr.dlr_conv_apply(u, ws)).astype(np.float64)
    y_k = host(dlr.dlr_layer(u, fwd, path="fft")).astype(np.float64)
    ref = oracle.dlr_layer(w.u, pnp(w.fwd))
    assert oracle.rel_l2(y, ref) <= TOL
    assert oracle.rel_l2(y, y_k) <= TOL
    assert dlr.device_status() == 0
