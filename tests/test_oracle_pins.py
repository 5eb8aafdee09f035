"""Pins for the float64 oracle: each test checks the oracle against something other than
itself -- a closed form, a library routine (numpy FFT / convolve, scipy lfilter / toeplitz /
expm, a general eigensolver), brute force on tiny inputs, or an invariant the pages state.

Sources: "Simplifying and Understanding State Space Models with Diagonal Linear RNNs"
(section 2: recurrence, kernel, Re cast; 2.1: DLR-prod, bidirectional, Toeplitz/FFT; 2.2:
parameterisation, DFT identity at (log Lambda)_re = 0, L = N), "The Annotated S4" (part 1:
unrolling the recurrence into a convolution; part 1b: HiPPO matrix; part 2: HiPPO-N) and
"Simplified State Space Layers for Sequence Modeling" (sections 2.2, 3: scan, diagonalised
MIMO system, ZOH, per-state Delta).
"""
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.signal

import oracle
from state_space_sequence_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _params(H, N, seed, unit=0):
    rng = np.random.default_rng(seed)
    p = inputs.dlr_params(rng, H, N, unit)
    return p.log_re, p.log_im, p.W


def _lam_np(log_re, log_im):
    a = log_re.astype(np.float64)
    t = log_im.astype(np.float64)
    return np.exp(-a * a) * np.exp(1j * t)


def _w_np(W):
    return W[..., 0].astype(np.float64) + 1j * W[..., 1].astype(np.float64)


# ---------------------------------------------------------------------------------------
# Kernel K_j = sum_n w_n lambda_n^j

@pytest.mark.parametrize("N", [4, 8, 16, 64])
def test_kernel_dft_identity(N):
    """(log Lambda)_re = 0, (log Lambda)_im = 2 pi n / N, L = N  =>  K = N * IDFT(w)
    (DLR paper section 2.2; with lambda_n = e^{+2 pi i n/N} the sum is numpy's ifft times N).
    theta is stored as float32, so K may differ from the exact DFT by at most
    sum_n |w_n| * j * |theta_n - 2 pi n/N| at lag j -- the test uses that bound."""
    rng = np.random.default_rng(100 + N)
    log_re = np.zeros((1, N), np.float32)
    log_im = (2 * np.pi * np.arange(N) / N).astype(np.float32)[None, :]
    W = rng.standard_normal((1, N, 2)).astype(np.float32)
    K = oracle.dlr_kernel(log_re, log_im, W, N, cast="complex")[0]
    w = _w_np(W)[0]
    ref = N * np.fft.ifft(w)
    dtheta = np.max(np.abs(log_im.astype(np.float64) - 2 * np.pi * np.arange(N) / N))
    bound = np.sum(np.abs(w)) * np.arange(N) * dtheta * 1.01 + 1e-12 * np.sum(np.abs(w))
    assert np.all(np.abs(K - ref) <= bound)
    # a sign or index slip gives an O(|w|) error, far above the bound
    assert np.max(bound) < 1e-4 * np.sum(np.abs(w))


def test_kernel_periodic_on_unit_circle():
    """At (log Lambda)_re = 0 and theta_n = 2 pi n/N the kernel has period N (DLR paper 2.2)."""
    N = 8
    log_re = np.zeros((1, N), np.float32)
    log_im = (2 * np.pi * np.arange(N) / N).astype(np.float32)[None, :]
    W = np.random.default_rng(3).standard_normal((1, N, 2)).astype(np.float32)
    K = oracle.dlr_kernel(log_re, log_im, W, 4 * N, cast="complex")[0]
    w = np.abs(_w_np(W)[0])
    dtheta = np.abs(log_im[0].astype(np.float64) - 2 * np.pi * np.arange(N) / N)
    for r in range(1, 4):
        # |K_{j+rN} - K_j| <= sum_n |w_n| |lambda_n^{rN} - 1| <= sum_n |w_n| r N dtheta_n
        bound = np.sum(w * r * N * dtheta) * 1.01 + 1e-12
        assert np.max(np.abs(K[r * N:(r + 1) * N] - K[:N])) <= bound
        assert bound < 1e-4 * np.sum(w)


def test_kernel_brute_force_powers():
    """Tiny case: K_j against sum_n w_n * (lambda_n ** j) with Python's complex power."""
    lr, li, W = _params(2, 5, seed=7)
    L = 40
    K = oracle.dlr_kernel(lr, li, W, L, cast="complex")
    lam = _lam_np(lr, li)
    w = _w_np(W)
    for h in range(2):
        for j in range(L):
            ref = sum(complex(w[h, n]) * complex(lam[h, n]) ** j for n in range(5))
            assert abs(K[h, j] - ref) <= 1e-12 * (1 + abs(ref))


def test_kernel_casts():
    """Re cast and DLR-prod cast are the real part and Re*Im of the complex kernel."""
    lr, li, W = _params(3, 6, seed=8)
    Kc = oracle.dlr_kernel(lr, li, W, 50, cast="complex")
    np.testing.assert_array_equal(oracle.dlr_kernel(lr, li, W, 50, cast="re"), Kc.real)
    np.testing.assert_allclose(oracle.dlr_kernel(lr, li, W, 50, cast="re_im"),
                               Kc.real * Kc.imag, rtol=1e-15, atol=0)


@pytest.mark.parametrize("N", [1, 2, 3, 4])
def test_dlr_prod_is_a_dlr_with_n_squared_states(N):
    """DLR paper 2.1 / A.2: the DLR-prod kernel Re(K)Im(K) = Im(K^2)/2 is the Re-cast kernel
    of a DLR whose states are the products lambda_n lambda_m with weights -i w_n w_m / 2."""
    lr, li, W = _params(2, N, seed=20 + N)
    L = 64
    kp = oracle.dlr_kernel(lr, li, W, L, cast="re_im")
    lam = _lam_np(lr, li)
    w = _w_np(W)
    j = np.arange(L)
    for h in range(2):
        mu = (lam[h][:, None] * lam[h][None, :]).ravel()
        nu = (-0.5j * w[h][:, None] * w[h][None, :]).ravel()
        ref = np.real((nu[None, :] * mu[None, :] ** j[:, None]).sum(1))
        np.testing.assert_allclose(kp[h], ref, rtol=1e-10, atol=1e-14)


# ---------------------------------------------------------------------------------------
# Recurrence (scan) and its convolution view

def test_recurrence_matches_scipy_lfilter():
    """Each state is the first-order IIR filter 1/(1 - lambda z^-1) driven by u (DLR paper
    section 2, Eq. 1); y = sum_n Re(w_n x_n). scipy.signal.lfilter runs the same recurrence
    independently (complex coefficients)."""
    lr, li, W = _params(3, 7, seed=9)
    u = np.random.default_rng(10).standard_normal((2, 3, 300)).astype(np.float32)
    y = oracle.dlr_recurrence(u, lr, li, W, nthreads=2)
    lam = _lam_np(lr, li)
    w = _w_np(W)
    for b in range(2):
        for h in range(3):
            ref = np.zeros(300)
            for n in range(7):
                x = scipy.signal.lfilter([1.0], [1.0, -lam[h, n]], u[b, h].astype(np.float64))
                ref += np.real(w[h, n] * x)
            np.testing.assert_allclose(y[b, h], ref, rtol=1e-11, atol=1e-12)


def test_impulse_response_is_kernel():
    """u = delta_0  =>  y_k = Re K_k (Annotated S4 part 1: the unrolled recurrence is a
    convolution with K = (CB, CAB, CA^2B, ...))."""
    lr, li, W = _params(4, 9, seed=11)
    L = 200
    u = np.zeros((1, 4, L), np.float32)
    u[..., 0] = 1.0
    y = oracle.dlr_recurrence(u, lr, li, W)[0]
    K = oracle.dlr_kernel(lr, li, W, L, cast="re")
    np.testing.assert_allclose(y, K, rtol=1e-12, atol=1e-14)


def test_recurrence_equals_library_convolution():
    """Recurrence == numpy.convolve(u, Re K)[:L] (the Re cast of section 2)."""
    lr, li, W = _params(2, 6, seed=12)
    L = 257
    u = np.random.default_rng(13).standard_normal((3, 2, L)).astype(np.float32)
    y = oracle.dlr_recurrence(u, lr, li, W)
    K = oracle.dlr_kernel(lr, li, W, L, cast="re")
    for b in range(3):
        for h in range(2):
            ref = np.convolve(u[b, h].astype(np.float64), K[h])[:L]
            np.testing.assert_allclose(y[b, h], ref, rtol=1e-10, atol=1e-12)


def test_toeplitz_equals_library_convolution():
    rng = np.random.default_rng(14)
    u = rng.standard_normal((2, 3, 129)).astype(np.float32)
    kap = rng.standard_normal((3, 129))
    y = oracle.toeplitz_causal(u, kap)
    for b in range(2):
        for h in range(3):
            np.testing.assert_allclose(y[b, h], np.convolve(u[b, h], kap[h])[:129],
                                       rtol=1e-12, atol=1e-12)


def test_constant_input_geometric_series():
    """u = 1  =>  y_k = Re sum_n w_n (1 - lambda_n^{k+1}) / (1 - lambda_n)."""
    lr, li, W = _params(2, 5, seed=15)
    L = 500
    y = oracle.dlr_recurrence(np.ones((1, 2, L), np.float32), lr, li, W)[0]
    lam = _lam_np(lr, li)
    w = _w_np(W)
    k = np.arange(L)
    for h in range(2):
        ref = np.real((w[h][None, :] * (1 - lam[h][None, :] ** (k[:, None] + 1))
                       / (1 - lam[h][None, :])).sum(1))
        np.testing.assert_allclose(y[h], ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("splits", [[1], [64], [100, 101], [7, 63, 64, 200, 511]])
def test_scan_chunking_associativity(splits):
    """S5 paper section 2.2: the recurrence is a scan with an associative operator, so running
    it chunk by chunk with the carried state gives the sequential result exactly."""
    lr, li, W = _params(2, 8, seed=16)
    L = 512
    u = np.random.default_rng(17).standard_normal((2, 2, L)).astype(np.float32)
    y_full = oracle.dlr_recurrence(u, lr, li, W)
    bounds = [0] + list(splits) + [L]
    x = None
    parts = []
    for s, e in zip(bounds[:-1], bounds[1:]):
        yp, x = oracle.dlr_recurrence(np.ascontiguousarray(u[..., s:e]), lr, li, W, x0=x,
                                      return_state=True)
        parts.append(yp)
    np.testing.assert_allclose(np.concatenate(parts, -1), y_full, rtol=1e-12, atol=1e-13)


def test_thread_count_does_not_change_results():
    lr, li, W = _params(5, 4, seed=18)
    u = np.random.default_rng(19).standard_normal((3, 5, 100)).astype(np.float32)
    np.testing.assert_array_equal(oracle.dlr_recurrence(u, lr, li, W, nthreads=1),
                                  oracle.dlr_recurrence(u, lr, li, W, nthreads=7))


# ---------------------------------------------------------------------------------------
# Bidirectional DLR

def test_bidirectional_is_toeplitz_matvec():
    """DLR paper 2.1: the bidirectional output is a Toeplitz matrix-vector product whose
    lower part holds Re K^1, upper part Re K^2, diagonal Re K^1_0 + Re K^2_0. Built with
    scipy.linalg.toeplitz and multiplied densely."""
    f = _params(2, 5, seed=21)
    g = _params(2, 5, seed=22)
    L = 90
    u = np.random.default_rng(23).standard_normal((2, 2, L)).astype(np.float32)
    y = oracle.dlr_bidirectional(u, f, g)
    K1 = oracle.dlr_kernel(*f, L, cast="re")
    K2 = oracle.dlr_kernel(*g, L, cast="re")
    for h in range(2):
        col = K1[h].copy()
        row = K2[h].copy()
        col[0] = row[0] = K1[h, 0] + K2[h, 0]
        T = scipy.linalg.toeplitz(col, row)
        for b in range(2):
            np.testing.assert_allclose(y[b, h], T @ u[b, h].astype(np.float64),
                                       rtol=1e-10, atol=1e-12)


def test_bidirectional_symmetry():
    """Same parameters both ways and a palindromic input give a palindromic output."""
    f = _params(1, 6, seed=24)
    half = np.random.default_rng(25).standard_normal(50).astype(np.float32)
    u = np.concatenate([half, half[::-1]])[None, None, :]
    y = oracle.dlr_bidirectional(u, f, f)[0, 0]
    np.testing.assert_allclose(y, y[::-1], rtol=1e-12, atol=1e-12)


def test_prod_layer_bidirectional_matches_toeplitz_matrix():
    f = _params(1, 4, seed=26)
    g = _params(1, 4, seed=27)
    L = 70
    u = np.random.default_rng(28).standard_normal((1, 1, L)).astype(np.float32)
    y = oracle.dlr_prod_layer(u, f, g)[0, 0]
    k1 = oracle.dlr_kernel(*f, L, cast="re_im")[0]
    k2 = oracle.dlr_kernel(*g, L, cast="re_im")[0]
    col, row = k1.copy(), k2.copy()
    col[0] = row[0] = k1[0] + k2[0]
    np.testing.assert_allclose(y, scipy.linalg.toeplitz(col, row) @ u[0, 0].astype(np.float64),
                               rtol=1e-10, atol=1e-13)


# ---------------------------------------------------------------------------------------
# S5

def _s5_small(H, P, seed, equal_delta=False):
    rng = np.random.default_rng(seed)
    lam = np.stack([-np.abs(rng.uniform(0.1, 2.0, P)), rng.uniform(-5, 5, P)], -1)
    if equal_delta:
        log_delta = np.full(P, np.log(0.05))
    else:
        log_delta = rng.uniform(np.log(1e-3), np.log(1e-1), P)
    Bt = rng.standard_normal((P, H, 2)) / np.sqrt(H)
    Ct = rng.standard_normal((H, P, 2)) / np.sqrt(H)
    D = rng.standard_normal(H)
    f = lambda a: np.asarray(a, np.float32)
    return f(lam), f(log_delta), f(Bt), f(Ct), f(D)


def test_zoh_matches_augmented_matrix_exponential():
    """ZOH of state p with step Delta_p: expm([[lambda_p Delta_p, Delta_p B~_p],[0, 0]]) has
    exp(lambda Delta) and B_bar_p as its first row (Van Loan's block exponential)."""
    lam, ld, Bt, _, _ = _s5_small(3, 5, seed=30)
    abar, bbar = oracle.s5_zoh(lam, ld, Bt)
    lamc = lam[:, 0].astype(np.float64) + 1j * lam[:, 1]
    delta = np.exp(ld.astype(np.float64))
    Btc = Bt[..., 0].astype(np.float64) + 1j * Bt[..., 1]
    H = Bt.shape[1]
    for p in range(5):
        M = np.zeros((1 + H, 1 + H), complex)
        M[0, 0] = lamc[p] * delta[p]
        M[0, 1:] = delta[p] * Btc[p]
        E = scipy.linalg.expm(M)
        np.testing.assert_allclose(abar[p], E[0, 0], rtol=1e-12)
        np.testing.assert_allclose(bbar[p], E[0, 1:], rtol=1e-10, atol=1e-14)


def test_s5_equals_dense_system_in_original_coordinates():
    """S5 paper section 3: A = V Lambda V^-1, B~ = V^-1 B, C~ = C V. With one shared Delta the
    diagonal layer must equal the dense system discretised by expm and run as a dense
    recurrence in the original coordinates."""
    H, P, L = 3, 4, 40
    lam, ld, Bt, Ct, D = _s5_small(H, P, seed=31, equal_delta=True)
    rng = np.random.default_rng(32)
    V = rng.standard_normal((P, P)) + 1j * rng.standard_normal((P, P))
    lamc = lam[:, 0].astype(np.float64) + 1j * lam[:, 1]
    A = V @ np.diag(lamc) @ np.linalg.inv(V)
    Btc = Bt[..., 0].astype(np.float64) + 1j * Bt[..., 1]
    Ctc = Ct[..., 0].astype(np.float64) + 1j * Ct[..., 1]
    Bd = V @ Btc
    Cd = Ctc @ np.linalg.inv(V)
    delta = float(np.exp(np.float64(ld[0])))
    M = np.zeros((P + H, P + H), complex)
    M[:P, :P] = A * delta
    M[:P, P:] = Bd * delta
    E = scipy.linalg.expm(M)
    Abar, Bbar = E[:P, :P], E[:P, P:]
    u = rng.standard_normal((2, L, H)).astype(np.float32)
    y = oracle.s5_layer(u, lam, ld, Bt, Ct, D)
    for b in range(2):
        x = np.zeros(P, complex)
        for k in range(L):
            x = Abar @ x + Bbar @ u[b, k].astype(np.float64)
            ref = np.real(Cd @ x) + D.astype(np.float64) * u[b, k]
            np.testing.assert_allclose(y[b, k], ref, rtol=1e-9, atol=1e-11)


def test_s5_zoh_exact_for_constant_input():
    """One state, constant input c: the discrete states equal the continuous solution
    x((k+1) Delta) = (e^{lambda (k+1) Delta} - 1)/lambda * B~ c."""
    lam = np.array([[-0.7, 3.0]], np.float32)
    ld = np.array([np.log(0.03)], np.float32)
    Bt = np.array([[[0.8, -0.4]]], np.float32)
    D = np.zeros(1, np.float32)
    L = 300
    c = 1.5
    u = np.full((1, L, 1), c, np.float32)
    lamc = complex(lam[0, 0], lam[0, 1])
    delta = float(np.exp(np.float64(ld[0])))
    t = (np.arange(L) + 1) * delta
    xs = (np.exp(lamc * t) - 1) / lamc * complex(Bt[0, 0, 0], Bt[0, 0, 1]) * c
    y_re = oracle.s5_layer(u, lam, ld, Bt, np.array([[[1.0, 0.0]]], np.float32), D)[0, :, 0]
    y_im = oracle.s5_layer(u, lam, ld, Bt, np.array([[[0.0, -1.0]]], np.float32), D)[0, :, 0]
    np.testing.assert_allclose(y_re, xs.real, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(y_im, xs.imag, rtol=1e-10, atol=1e-13)


def test_s5_feedthrough_and_linearity():
    H, P, L = 4, 3, 30
    lam, ld, Bt, Ct, D = _s5_small(H, P, seed=33)
    rng = np.random.default_rng(34)
    u1 = rng.standard_normal((1, L, H)).astype(np.float32)
    u2 = rng.standard_normal((1, L, H)).astype(np.float32)
    zero_c = np.zeros_like(Ct)
    np.testing.assert_allclose(oracle.s5_layer(u1, lam, ld, Bt, zero_c, D)[0],
                               u1[0] * D.astype(np.float64), rtol=1e-15)
    np.testing.assert_allclose(oracle.s5_layer(u1, lam, ld, np.zeros_like(Bt), Ct, D)[0],
                               u1[0] * D.astype(np.float64), rtol=1e-15)
    a, b = 0.75, -2.0
    ysum = oracle.s5_layer(u1 * np.float32(a) + u2 * np.float32(b), lam, ld, Bt, Ct, D)
    y1 = oracle.s5_layer(u1, lam, ld, Bt, Ct, D)
    y2 = oracle.s5_layer(u2, lam, ld, Bt, Ct, D)
    np.testing.assert_allclose(ysum, a * y1 + b * y2, rtol=1e-5, atol=1e-6)


def test_s5_zoh_small_step_limit():
    """S5 section 3.2: for a small step the ZOH input matrix tends to Delta B~; the next two
    terms of the series of (e^{lambda Delta} - 1)/lambda are Delta^2 lambda/2 and
    Delta^3 lambda^2/6, so B_bar - Delta B~ (1 + lambda Delta/2) is bounded by the third."""
    lam = np.array([[-0.5, 2.0], [-0.5, -7.0], [-0.5, 19.0]], np.float32)
    Bt = np.array([[[0.3, -1.1]], [[-0.8, 0.2]], [[1.4, 0.9]]], np.float32)
    for step in (1e-3, 1e-5):
        ld = np.full(3, np.log(step), np.float32)
        abar, bbar = oracle.s5_zoh(lam, ld, Bt)
        delta = np.exp(ld.astype(np.float64))
        lamc = lam[:, 0].astype(np.float64) + 1j * lam[:, 1]
        Btc = Bt[:, 0, 0].astype(np.float64) + 1j * Bt[:, 0, 1]
        first = delta * Btc
        second = first * (1 + lamc * delta / 2)
        # plus the double rounding of e^{lambda Delta} - 1, relative eps / |lambda Delta|
        bound = np.abs(first) * (np.abs(lamc * delta) ** 2 / 6 * 1.01 +
                                 4e-16 / np.abs(lamc * delta))
        assert np.all(np.abs(bbar[:, 0] - second) <= bound)
        assert np.all(np.abs(bbar[:, 0] - first) > 0.4 * np.abs(first * lamc * delta))
        np.testing.assert_allclose(np.abs(abar), np.exp(-0.5 * delta), rtol=1e-14)


def test_s5_one_state_one_feature_is_a_scalar_filter():
    """P = 1, H = 1: the layer is the first-order complex filter x_k = a x_{k-1} + b u_k
    (scipy lfilter) with a, b from the block exponential of [[lambda Delta, Delta B~], [0, 0]],
    read out as Re(c x_k) + d u_k."""
    lam = np.array([[-0.3, 1.7]], np.float32)
    ld = np.array([np.log(0.2)], np.float32)
    Bt = np.array([[[0.6, -0.9]]], np.float32)
    Ct = np.array([[[-1.2, 0.4]]], np.float32)
    D = np.array([0.35], np.float32)
    rng = np.random.default_rng(35)
    u = rng.standard_normal((2, 64, 1)).astype(np.float32)
    y = oracle.s5_layer(u, lam, ld, Bt, Ct, D)
    delta = float(np.exp(np.float64(ld[0])))
    lamc = complex(float(lam[0, 0]), float(lam[0, 1]))
    E = scipy.linalg.expm(np.array([[lamc * delta, delta * complex(float(Bt[0, 0, 0]),
                                                                    float(Bt[0, 0, 1]))],
                                    [0, 0]]))
    a, b = E[0, 0], E[0, 1]
    c = complex(float(Ct[0, 0, 0]), float(Ct[0, 0, 1]))
    for r in range(2):
        ur = u[r, :, 0].astype(np.float64)
        x = scipy.signal.lfilter([b], [1.0, -a], ur.astype(complex))
        np.testing.assert_allclose(y[r, :, 0], (c * x).real + float(D[0]) * ur, rtol=1e-11,
                                   atol=1e-13)


# ---------------------------------------------------------------------------------------
# Backward pass of the causal Re-cast layer

@pytest.mark.parametrize("B,H,N,L,unit", [(2, 3, 4, 37, 1), (1, 2, 16, 200, 0), (3, 1, 1, 5, 1)])
def test_backward_input_gradient_is_the_adjoint(B, H, N, L, unit):
    """The layer is linear in u, so for any g the input gradient du satisfies
    <g, DLR(u)> = <u, du> (DLR paper section 2: y is a causal convolution of u with Re K)."""
    log_re, log_im, W = _params(H, N, seed=60 + L, unit=unit)
    rng = np.random.default_rng(61 + L)
    u = rng.standard_normal((B, H, L)).astype(np.float32)
    g = rng.standard_normal((B, H, L))
    du, _, _, _ = oracle.dlr_backward(u, g, log_re, log_im, W)
    y = oracle.dlr_layer(u, (log_re, log_im, W))
    lhs, rhs = float((g * y).sum()), float((u.astype(np.float64) * du).sum())
    assert abs(lhs - rhs) <= 1e-11 * (np.abs(g * y).sum() + 1)
    # and du is a function of g alone: the reversed-time layer applied to g
    du_rev = oracle.dlr_layer(g[..., ::-1].astype(np.float32), (log_re, log_im, W))[..., ::-1]
    g32 = g.astype(np.float32).astype(np.float64)
    du32, _, _, _ = oracle.dlr_backward(u, g32, log_re, log_im, W)
    np.testing.assert_allclose(du32, du_rev, rtol=1e-9, atol=1e-9 * np.abs(du_rev).max())


def test_backward_parameter_gradients_match_finite_differences():
    """d/d(log_re, log_im, W_re, W_im) of sum(g * y) against central differences of a float64
    brute-force forward (K_j = sum_n W_n exp(j(-a^2 + i theta)), y = causal convolution of u
    with Re K), one channel on the unit circle (a = 0, where d/da vanishes)."""
    B, H, N, L = 2, 2, 3, 20
    log_re, log_im, W = _params(H, N, seed=62, unit=1)
    rng = np.random.default_rng(63)
    u = rng.standard_normal((B, H, L)).astype(np.float32)
    g = rng.standard_normal((B, H, L))
    _, d_re, d_im, dW = oracle.dlr_backward(u, g, log_re, log_im, W)
    ud = u.astype(np.float64)
    j = np.arange(L)

    def loss(a, th, wr, wi):
        tot = 0.0
        for h in range(H):
            lam_j = np.exp(np.outer(-a[h] ** 2 + 1j * th[h], j))      # [N, L]
            K = ((wr[h] + 1j * wi[h])[:, None] * lam_j).sum(0).real
            for b in range(B):
                tot += float(g[b, h] @ np.convolve(ud[b, h], K)[:L])
        return tot

    base = [log_re.astype(np.float64), log_im.astype(np.float64),
            W[..., 0].astype(np.float64), W[..., 1].astype(np.float64)]
    grads = [d_re, d_im, dW[..., 0], dW[..., 1]]
    for which in range(4):
        fd = np.empty((H, N))
        for h in range(H):
            for n in range(N):
                step = 1e-6 * max(1.0, abs(base[which][h, n]))
                plus = [x.copy() for x in base]
                minus = [x.copy() for x in base]
                plus[which][h, n] += step
                minus[which][h, n] -= step
                fd[h, n] = (loss(*plus) - loss(*minus)) / (2 * step)
        scale = np.abs(fd).max()
        np.testing.assert_allclose(grads[which], fd, rtol=0, atol=1e-6 * scale,
                                   err_msg=["log_re", "log_im", "W_re", "W_im"][which])
    assert np.all(d_re[log_re == 0] == 0)


@pytest.mark.parametrize("cast", ["re", "re_im"])
def test_backward_bidirectional_and_prod_cast_match_finite_differences(cast):
    """Both parameter sets of the bidirectional layer (section 2.1: y = DLR1(u) +
    rev(DLR2(rev(u)))), with the Re or the DLR-prod cast (kappa_j = Re K_j Im K_j), against
    central differences of a float64 brute-force forward; and the input gradient against the
    adjoint identity."""
    B, H, N, L = 2, 2, 3, 16
    w = inputs.make_dlr(B, H, N, L, seed=64, bidir=True, unit_channels=1)
    rng = np.random.default_rng(65)
    g = rng.standard_normal((B, H, L))
    fwd = (w.fwd.log_re, w.fwd.log_im, w.fwd.W)
    bwd = (w.bwd.log_re, w.bwd.log_im, w.bwd.W)
    du, grads = oracle.dlr_layer_backward(w.u, g, fwd, bwd, cast)
    ud = w.u.astype(np.float64)
    j = np.arange(L)

    def kernel(a, th, wr, wi, h):
        K = ((wr[h] + 1j * wi[h])[:, None] * np.exp(np.outer(-a[h] ** 2 + 1j * th[h], j))).sum(0)
        return K.real if cast == "re" else K.real * K.imag

    def loss(p1, p2):
        tot = 0.0
        for h in range(H):
            k1, k2 = kernel(*p1, h), kernel(*p2, h)
            for b in range(B):
                y = np.convolve(ud[b, h], k1)[:L] + np.convolve(ud[b, h][::-1], k2)[:L][::-1]
                tot += float(g[b, h] @ y)
        return tot

    base = [[x.astype(np.float64) for x in (p[0], p[1], p[2][..., 0], p[2][..., 1])]
            for p in (fwd, bwd)]
    for d in range(2):
        dr, di, dw = grads[d]
        mine = [dr, di, dw[..., 0], dw[..., 1]]
        for which in range(4):
            fd = np.empty((H, N))
            for h in range(H):
                for n in range(N):
                    step = 1e-6 * max(1.0, abs(base[d][which][h, n]))
                    plus = [[x.copy() for x in q] for q in base]
                    minus = [[x.copy() for x in q] for q in base]
                    plus[d][which][h, n] += step
                    minus[d][which][h, n] -= step
                    fd[h, n] = (loss(*plus) - loss(*minus)) / (2 * step)
            np.testing.assert_allclose(mine[which], fd, rtol=0, atol=1e-6 * np.abs(fd).max(),
                                       err_msg=f"direction {d}, parameter {which}")
    y = oracle.dlr_layer(w.u, fwd, bwd, cast=cast)
    assert abs(float((g * y).sum()) - float((ud * du).sum())) <= 1e-11 * np.abs(g * y).sum()


# ---------------------------------------------------------------------------------------
# Input generator structure (HiPPO-N spectrum)

@pytest.mark.parametrize("P", [4, 16, 64])
def test_hippo_n_normal_plus_low_rank(P):
    """Annotated S4 part 2: HiPPO-LegS is a normal matrix minus a rank-one term, A = S - p p^T
    with S normal, so S = V Lambda V^* for a unitary V. Rebuild A from the generator's
    eigenvalues and a unitary eigenbasis of S, and check S S^T = S^T S."""
    n = np.arange(P, dtype=np.float64)
    p = np.sqrt(n + 0.5)
    A = inputs.hippo_legs(P)
    S = A + np.outer(p, p)
    np.testing.assert_allclose(S @ S.T, S.T @ S, atol=1e-9 * P * P)
    mu, V = np.linalg.eigh(-1j * (S + 0.5 * np.eye(P)))  # Hermitian: V unitary
    np.testing.assert_allclose(V.conj().T @ V, np.eye(P), atol=1e-12 * P)
    lam = inputs.hippo_n_eigenvalues(P).astype(np.float64)
    lam = lam[np.argsort(lam[:, 1])]
    lamc = lam[:, 0] + 1j * lam[:, 1]
    A_rec = (V * lamc) @ V.conj().T - np.outer(p, p)
    scale = np.max(np.abs(lam[:, 1]))
    np.testing.assert_allclose(A_rec.real, A, atol=1e-6 * scale)
    np.testing.assert_allclose(A_rec.imag, 0.0, atol=1e-6 * scale)


def test_hippo_legs_golden():
    rows = []
    with open(os.path.join(GOLDEN, "hippo_legs_p4.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([eval(tok, {"sqrt": np.sqrt}) for tok in line.split()])
    np.testing.assert_allclose(inputs.hippo_legs(4), np.array(rows), rtol=1e-15)


@pytest.mark.parametrize("P", [8, 64, 256])
def test_hippo_n_spectrum(P):
    """Annotated S4 part 2: S = A + p p^T is -1/2 I plus a skew-symmetric matrix, so every
    eigenvalue has real part -1/2 and they come in conjugate pairs; a general (non-Hermitian)
    eigensolver on the dense S agrees with the generator's Hermitian route."""
    lam = inputs.hippo_n_eigenvalues(P)
    np.testing.assert_allclose(lam[:, 0], -0.5, rtol=0, atol=1e-12)
    n = np.arange(P, dtype=np.float64)
    S = inputs.hippo_legs(P) + np.outer(np.sqrt(n + 0.5), np.sqrt(n + 0.5))
    np.testing.assert_allclose(np.diagonal(S), -0.5, atol=1e-12)
    ev = np.linalg.eigvals(S)
    np.testing.assert_allclose(np.sort(ev.imag), np.sort(lam[:, 1]), rtol=1e-8,
                               atol=1e-8 * np.max(np.abs(lam[:, 1])))
    np.testing.assert_allclose(np.sort(lam[:, 1]), -np.sort(lam[:, 1])[::-1], atol=1e-6)


def test_dlr_init_ranges():
    """DLR paper 2.2: |lambda| = exp(-(log Lambda)_re^2) lies in [e^-0.25, e^-0.00025]."""
    p = inputs.dlr_params(np.random.default_rng(0), 64, 64)
    mag = np.exp(-p.log_re.astype(np.float64) ** 2)
    assert mag.min() >= np.exp(-0.25) * (1 - 1e-6)
    assert mag.max() <= np.exp(-0.00025) * (1 + 1e-6)
    np.testing.assert_allclose(p.log_im[0], 2 * np.pi * np.arange(64) / 64, rtol=1e-6)


def test_oracle_lambda_magnitude_spans_the_init_range():
    """The oracle's lambda against the range the DLR paper (section 2.2) fixes through its
    initialisation: r ~ U(log 5e-4, log 0.5) and (log Lambda)_re = sqrt(e^r / 2) put
    (log Lambda)_re^2 in [2.5e-4, 0.25], so |lambda| must lie in [e^-0.25, e^-0.00025] with
    both ends reached by many draws, and the end points themselves map to those magnitudes.
    A convention such as exp(-(log Lambda)_re) or exp(-2 (log Lambda)_re^2) leaves the range."""
    p = inputs.dlr_params(np.random.default_rng(7), 128, 64)
    lam = oracle.dlr_lambda(p.log_re, p.log_im)
    mag = np.abs(lam)
    lo, hi = np.exp(-0.25), np.exp(-0.00025)
    assert mag.min() >= lo * (1 - 1e-6) and mag.max() <= hi * (1 + 1e-6)
    # 8192 log-uniform draws: both ends of the range are approached
    assert mag.min() < np.exp(-0.24) and mag.max() > np.exp(-0.0003)
    # the phase is (log Lambda)_im
    np.testing.assert_allclose(np.angle(lam[0, 1:32]), p.log_im[0, 1:32].astype(np.float64),
                               rtol=0, atol=1e-12)
    # end points of the init range: r = log 0.5 -> a = 0.5; r = log 5e-4 -> a = sqrt(2.5e-4)
    a = np.array([[0.5, np.sqrt(2.5e-4)]], np.float32)
    ends = np.abs(oracle.dlr_lambda(a, np.zeros_like(a)))[0]
    np.testing.assert_allclose(ends, np.exp(-a[0].astype(np.float64) ** 2), rtol=1e-15)
    np.testing.assert_allclose(ends, [lo, hi], rtol=1e-7)


# ---------------------------------------------------------------------------------------
# Direct spectrum (The Annotated S4, part 2: the truncated generating function at the roots
# of unity)

@pytest.mark.parametrize("bidir", [False, True])
def test_direct_spectrum_equals_fft_of_the_circulant_column(bidir):
    """The spectrum from the geometric series equals numpy's real FFT of the circulant column
    built from the oracle's kernel (section 2.1 of the DLR paper: K zero-padded to 2L, the
    anti-causal kernel wrapped to the end, lag 0 counted by both). Channels on the unit circle
    (log_re = 0 with theta = 2 pi n / N) put some bins exactly on a pole of the series."""
    H, N, L, M = 3, 16, 100, 256
    rng = np.random.default_rng(31)
    f = inputs.dlr_params(rng, H, N, unit_channels=1)
    b = inputs.dlr_params(rng, H, N, unit_channels=1) if bidir else None
    fwd = (f.log_re, f.log_im, f.W)
    bwd = (b.log_re, b.log_im, b.W) if bidir else None
    C = oracle.dlr_spectrum(*fwd, L, M, bwd=bwd)
    col = np.zeros((H, M))
    col[:, :L] = oracle.dlr_kernel(*fwd, L, cast="re")
    if bidir:
        k2 = oracle.dlr_kernel(*bwd, L, cast="re")
        col[:, 0] += k2[:, 0]
        col[:, M - L + 1:] += k2[:, 1:][:, ::-1]
    ref = np.fft.rfft(col, axis=-1)
    scale = np.max(np.abs(ref))
    np.testing.assert_allclose(C, ref, rtol=0, atol=1e-10 * scale)


def test_direct_spectrum_single_state_geometric_sum():
    """One state with W = 1 and lambda = exp(-a^2 + i theta): C_k is the real part's DFT,
    (G(lambda w^k) + conj(G(lambda w^-k))) / 2, and G is checked against the explicit sum of
    L powers in float64; at a = 0, theta = 2 pi m / M the bin k = m holds the pole value L."""
    L, M = 50, 128
    for a, th in [(0.3, 0.7), (0.0, 2 * np.pi * 5 / M), (0.05, -1.1)]:
        lr = np.array([[a]], np.float32)
        li = np.array([[th]], np.float32)
        W = np.array([[[1.0, 0.0]]], np.float32)
        C = oracle.dlr_spectrum(lr, li, W, L, M)[0]
        lam = np.exp(-np.float64(lr[0, 0]) ** 2 + 1j * np.float64(li[0, 0]))
        j = np.arange(L)
        k = np.arange(M // 2 + 1)
        w = np.exp(-2j * np.pi * k / M)
        Gp = np.array([np.sum((lam * wk) ** j) for wk in w])
        Gm = np.array([np.sum((lam / wk) ** j) for wk in w])
        np.testing.assert_allclose(C, 0.5 * (Gp + np.conj(Gm)), rtol=1e-9, atol=1e-9)
    # the pole: with a = 0 and theta = 2 pi 5 / M (up to its float32 rounding) the causal
    # series at bin 5 is L: 2 C_5 - conj(G(lambda w^-5)) = G(lambda w^5) ~ L
    lr = np.zeros((1, 1), np.float32)
    li = np.array([[2 * np.pi * 5 / M]], np.float32)
    C = oracle.dlr_spectrum(lr, li, np.array([[[1.0, 0.0]]], np.float32), L, M)[0]
    lam = np.exp(1j * np.float64(li[0, 0]))
    Gm5 = np.sum((lam * np.exp(2j * np.pi * 5 / M)) ** np.arange(L))
    assert abs(2 * C[5] - np.conj(Gm5) - L) < 1e-4 * L


# ---------------------------------------------------------------------------------------
# Discretisation and parameterisation variants

def test_bilinear_matches_scipy_cont2discrete():
    """Per state, the complex scalar system x' = lambda x + b u in its real 2x2 form,
    discretised by scipy.signal.cont2discrete(method='bilinear'), gives the oracle's
    Lambda_bar (as a rotation-scaling block) and B_bar (The Annotated S4, part 1)."""
    H, P = 3, 5
    lam, ld, Bt, _, _ = _s5_small(H, P, seed=41)
    abar, bbar = oracle.s5_bilinear(lam, ld, Bt)
    for p in range(P):
        lr, li = np.float64(lam[p, 0]), np.float64(lam[p, 1])
        A = np.array([[lr, -li], [li, lr]])
        Bm = np.stack([Bt[p, :, 0], Bt[p, :, 1]], 0).astype(np.float64)   # [2, H]
        dt = float(np.exp(np.float64(ld[p])))
        Ad, Bd, _, _, _ = scipy.signal.cont2discrete((A, Bm, np.eye(2), np.zeros((2, H))), dt,
                                                     method="bilinear")
        np.testing.assert_allclose(Ad, [[abar[p].real, -abar[p].imag],
                                        [abar[p].imag, abar[p].real]], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(Bd[0] + 1j * Bd[1], bbar[p], rtol=1e-12, atol=1e-14)
    # the Pade property: |Lambda_bar| < 1 in the left half-plane, exp(z) to O(z^3)
    assert np.all(np.abs(abar) < 1.0)
    z = 1e-3 * (np.float64(lam[:, 0]) + 1j * np.float64(lam[:, 1]))
    small = (1 + z / 2) / (1 - z / 2)
    # (1 + z/2) / (1 - z/2) - exp(z) = z^3 / 12 + O(z^4)
    assert np.all(np.abs(small - np.exp(z)) <= np.abs(z) ** 3 / 12 * 1.01 + 1e-15)
    assert np.all(np.abs(small - np.exp(z)) >= np.abs(z) ** 3 / 12 * 0.99)


def test_s5_bilinear_equals_dense_system():
    """The bilinear S5 layer equals the dense system in its original coordinates (A = V Lambda
    V^-1, B = V B~, C = C~ V^-1) discretised by scipy's bilinear transform and run densely."""
    H, P, L = 3, 4, 40
    lam, ld, Bt, Ct, D = _s5_small(H, P, seed=43, equal_delta=True)
    rng = np.random.default_rng(44)
    V = rng.standard_normal((P, P)) + 1j * rng.standard_normal((P, P))
    lamc = lam[:, 0].astype(np.float64) + 1j * lam[:, 1]
    A = V @ np.diag(lamc) @ np.linalg.inv(V)
    Btc = Bt[..., 0].astype(np.float64) + 1j * Bt[..., 1]
    Ctc = Ct[..., 0].astype(np.float64) + 1j * Ct[..., 1]
    Bd, Cd = V @ Btc, Ctc @ np.linalg.inv(V)
    dt = float(np.exp(np.float64(ld[0])))
    Ad, Bdd, _, _, _ = scipy.signal.cont2discrete((A, Bd, Cd, np.zeros((H, H))), dt,
                                                  method="bilinear")
    u = rng.standard_normal((2, L, H)).astype(np.float32)
    y = oracle.s5_layer(u, lam, ld, Bt, Ct, D, disc="bilinear")
    for b in range(2):
        x = np.zeros(P, complex)
        for k in range(L):
            x = Ad @ x + Bdd @ u[b, k].astype(np.float64)
            ref = np.real(Cd @ x) + D.astype(np.float64) * u[b, k]
            np.testing.assert_allclose(y[b, k], ref, rtol=1e-9, atol=1e-11)


def test_s5_time_varying_unit_gaps_equal_the_layer():
    """dt = 1 at every step reduces the time-varying layer to the ZOH layer."""
    H, P, L = 4, 6, 50
    lam, ld, Bt, Ct, D = _s5_small(H, P, seed=45)
    u = np.random.default_rng(46).standard_normal((2, L, H)).astype(np.float32)
    y = oracle.s5_layer_tv(u, np.ones((2, L), np.float32), lam, ld, Bt, Ct, D)
    np.testing.assert_allclose(y, oracle.s5_layer(u, lam, ld, Bt, Ct, D), rtol=1e-12,
                               atol=1e-12)


def test_s5_time_varying_exact_for_piecewise_constant_input():
    """One state, one feature, u = c constant, irregular gaps: the ZOH at every step keeps the
    sampled continuous solution x(T_k) = (exp(Lambda Delta T_k) - 1) / Lambda B~ c, T_k the
    elapsed time (S5 section 6.3's irregular sampling)."""
    lam = np.array([[-0.7, 3.1]], np.float32)
    ld = np.array([np.log(0.2)], np.float32)
    Bt = np.array([[[0.8, -0.3]]], np.float32)
    Ct = np.array([[[1.0, 0.0]]], np.float32)
    D = np.zeros(1, np.float32)
    rng = np.random.default_rng(47)
    dt = inputs.irregular_gaps(rng, 1, 30)
    c = np.float32(1.5)
    u = np.full((1, 30, 1), c, np.float32)
    y = oracle.s5_layer_tv(u, dt, lam, ld, Bt, Ct, D)[0, :, 0]
    lc = np.float64(lam[0, 0]) + 1j * np.float64(lam[0, 1])
    T = np.cumsum(dt[0].astype(np.float64)) * np.exp(np.float64(ld[0]))
    x = np.expm1(lc * T) / lc * (np.float64(Bt[0, 0, 0]) + 1j * np.float64(Bt[0, 0, 1])) * c
    np.testing.assert_allclose(y, x.real, rtol=1e-10, atol=1e-12)


def test_s5_time_varying_equals_dense_per_step_expm():
    """Irregular gaps on a dense system: every step's ZOH by scipy's matrix exponential of the
    augmented matrix [[A d, B d], [0, 0]] with d = Delta dt_k, run densely, equals the layer."""
    H, P, L = 2, 3, 25
    lam, ld, Bt, Ct, D = _s5_small(H, P, seed=48, equal_delta=True)
    rng = np.random.default_rng(49)
    V = rng.standard_normal((P, P)) + 1j * rng.standard_normal((P, P))
    lamc = lam[:, 0].astype(np.float64) + 1j * lam[:, 1]
    A = V @ np.diag(lamc) @ np.linalg.inv(V)
    Btc = Bt[..., 0].astype(np.float64) + 1j * Bt[..., 1]
    Ctc = Ct[..., 0].astype(np.float64) + 1j * Ct[..., 1]
    Bd, Cd = V @ Btc, Ctc @ np.linalg.inv(V)
    delta = float(np.exp(np.float64(ld[0])))
    dt = inputs.irregular_gaps(rng, 1, L)
    u = rng.standard_normal((1, L, H)).astype(np.float32)
    y = oracle.s5_layer_tv(u, dt, lam, ld, Bt, Ct, D)
    x = np.zeros(P, complex)
    for k in range(L):
        d = delta * np.float64(dt[0, k])
        M = np.zeros((P + H, P + H), complex)
        M[:P, :P] = A * d
        M[:P, P:] = Bd * d
        E = scipy.linalg.expm(M)
        x = E[:P, :P] @ x + E[:P, P:] @ u[0, k].astype(np.float64)
        ref = np.real(Cd @ x) + D.astype(np.float64) * u[0, k]
        np.testing.assert_allclose(y[0, k], ref, rtol=1e-9, atol=1e-11)


def test_dss_exp_as_dlr():
    """DSS_exp (DLR paper section 2): the zero-order-hold recurrence of x' = Lambda x + u equals
    the DLR with lambda = exp(Delta Lambda) and W' = W (exp(Delta Lambda) - 1) / Lambda (run by
    the oracle's DLR recurrence on the mapped parameters rounded to float32), and for a
    constant input the state is the sampled continuous solution (exp(Lambda t) - 1) / Lambda."""
    rng = np.random.default_rng(50)
    H, N, L, B = 2, 6, 80, 2
    Lam = np.stack([-rng.uniform(0.01, 1.0, (H, N)), rng.uniform(-3, 3, (H, N))], -1)
    ld = rng.uniform(np.log(0.01), np.log(0.5), H)
    W = rng.standard_normal((H, N, 2)) / N
    f = lambda a: np.asarray(a, np.float32)
    Lam, ld, W = f(Lam), f(ld), f(W)
    u = rng.standard_normal((B, H, L)).astype(np.float32)
    y_def = oracle.dss_exp_layer(u, Lam, ld, W)
    lr, li, Wn = oracle.dss_exp_params(Lam, ld, W)
    y_dlr = oracle.dlr_recurrence(u, f(lr), f(li), f(Wn))
    assert oracle.rel_l2(y_dlr, y_def) < 1e-6       # float32 rounding of the mapped parameters
    # constant input: x_k = (exp(Lambda (k+1) Delta) - 1) / Lambda
    uc = np.ones((1, H, L), np.float32)
    yc = oracle.dss_exp_layer(uc, Lam, ld, W)[0]
    Lc = Lam[..., 0].astype(np.float64) + 1j * Lam[..., 1]
    t = (np.arange(L) + 1)[None, None, :] * np.exp(ld.astype(np.float64))[:, None, None]
    x = np.expm1(Lc[..., None] * t) / Lc[..., None]
    Wc = W[..., 0].astype(np.float64) + 1j * W[..., 1]
    np.testing.assert_allclose(yc, (Wc[..., None] * x).sum(1).real, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("kind", ["exp", "softplus", "best"])
def test_reparam_maps_give_the_decay_rate(kind):
    """The reparameterised decay rates (StableSSM thread: exponential, softplus, and
    f(w) = 1 / (a w^2 + b)) as (log Lambda)_re: the oracle's lambda then has magnitude
    exp(-f(w)) with f computed here from its own definition, and stays inside the unit disk."""
    w = np.linspace(-4, 4, 33)[None, :]
    a, b = 0.5, 2.0
    lr = oracle.reparam_log_re(w, kind, a, b)
    lam = oracle.dlr_lambda(lr.astype(np.float32), np.full_like(lr, 0.3, dtype=np.float32))
    f = {"exp": np.exp(w), "softplus": np.log1p(np.exp(w)), "best": 1.0 / (a * w ** 2 + b)}[kind]
    # log_re is rounded to float32 (relative 2^-24), which moves f by up to 2^-23 of itself
    rel = np.abs(np.abs(lam) / np.exp(-f) - 1.0)
    assert np.all(rel <= 1.1 * f * 2.0 ** -23 + 1e-12)
    assert np.all(np.abs(lam) < 1.0)


def test_block_diagonal_hippo_n():
    """S5 section 4.3: J HiPPO-N blocks on the diagonal. The eigenvalues of the explicit block
    diagonal matrix (each block the normal part of the (P/J)-point HiPPO-LegS) from a general
    eigensolver equal the generator's spectrum; Re = -1/2 throughout."""
    P, J = 24, 3
    lam = inputs.hippo_n_block_eigenvalues(P, J)
    m = P // J
    n = np.arange(m, dtype=np.float64)
    A = inputs.hippo_legs(m)
    p = np.sqrt(n + 0.5)
    S = A + np.outer(p, p)
    ev = np.linalg.eigvals(scipy.linalg.block_diag(*([S] * J)))
    np.testing.assert_allclose(np.sort(ev.imag), np.sort(lam[:, 1]), rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(lam[:, 0], -0.5, atol=1e-12)
    np.testing.assert_allclose(ev.real, -0.5, atol=1e-9)
