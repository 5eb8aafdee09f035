"""Float64 CPU oracle for the DLR / S5 hot path.

TEST INFRASTRUCTURE ONLY: imported by the test-suite, by ``__graft_entry__.smoke()`` and by
the benchmark's CPU-baseline leg, never by the library. It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain float64 loops) plus numpy library primitives
(complex matmul, exp, FFT) where a step is a plain matrix product or a convolution. Each
function cites the passage it follows and states the reading it takes where the pages are
silent.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, library routines (numpy FFT, scipy lfilter / toeplitz / expm) or brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None

DEFAULT_THREADS = max(1, min(os.cpu_count() or 1, 16))


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so (portable flags only)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        path = build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.orc_lambda.argtypes = [i64, i64, P, P, P]
        lib.orc_dlr_kernel.argtypes = [i64, i64, i64, P, P, P, ctypes.c_int, P]
        lib.orc_dlr_recurrence.argtypes = [i64, i64, i64, i64, P, P, P, P, P, P, P,
                                           ctypes.c_int]
        lib.orc_toeplitz_causal.argtypes = [i64, i64, i64, P, P, P, ctypes.c_int]
        lib.orc_diag_scan.argtypes = [i64, i64, P, P, P]
        lib.orc_diag_scan_tv.argtypes = [i64, i64, P, P, P]
        _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


# ------------------------------------------------------------------------------------------
# DLR ("Simplifying and Understanding State Space Models with Diagonal Linear RNNs")

def dlr_lambda(log_re, log_im) -> np.ndarray:
    """lambda = exp(-(log Lambda)_re^2 + i (log Lambda)_im), complex128 [H, N] (section 2.2)."""
    log_re, log_im = _f32(log_re), _f32(log_im)
    out = np.empty(log_re.shape + (2,), np.float64)
    _load().orc_lambda(log_re.shape[0], log_re.shape[1], _p(log_re), _p(log_im), _p(out))
    return out[..., 0] + 1j * out[..., 1]


def dlr_kernel(log_re, log_im, W, L: int, cast: str = "re") -> np.ndarray:
    """K_j = sum_n W_n lambda_n^j for j < L (section 2, Eq. 3/4), cast 're', 're_im' or
    'complex' (section 2 Re cast; section 2.1 DLR-prod cast Re(K)*Im(K))."""
    log_re, log_im, W = _f32(log_re), _f32(log_im), _f32(W)
    H, N = log_re.shape
    code = {"re": 0, "re_im": 1, "complex": 2}[cast]
    shape = (H, L, 2) if code == 2 else (H, L)
    K = np.empty(shape, np.float64)
    _load().orc_dlr_kernel(H, N, L, _p(log_re), _p(log_im), _p(W), code, _p(K))
    if code == 2:
        return K[..., 0] + 1j * K[..., 1]
    return K


def dlr_recurrence(u, log_re, log_im, W, x0=None, return_state: bool = False,
                   nthreads: int = DEFAULT_THREADS):
    """Sequential DLR recurrence with the Re cast (section 2, Eq. 1):
    x_{n,k} = lambda_n x_{n,k-1} + u_k, y_k = sum_n Re(w_n x_{n,k}); u [B, H, L]."""
    u = _f32(u)
    log_re, log_im, W = _f32(log_re), _f32(log_im), _f32(W)
    B, H, L = u.shape
    N = log_re.shape[1]
    y = np.empty((B, H, L), np.float64)
    x0a = None
    if x0 is not None:
        x0 = np.asarray(x0)
        x0a = _f64(np.stack([x0.real, x0.imag], -1))
    xT = np.empty((B, H, N, 2), np.float64) if return_state else None
    _load().orc_dlr_recurrence(B, H, N, L, _p(u), _p(log_re), _p(log_im), _p(W), _p(x0a),
                               _p(y), _p(xT), int(nthreads))
    if return_state:
        return y, xT[..., 0] + 1j * xT[..., 1]
    return y


def toeplitz_causal(u, kappa, nthreads: int = DEFAULT_THREADS) -> np.ndarray:
    """Direct causal Toeplitz sum y_k = sum_{j<=k} kappa_{h,j} u_{k-j} (section 2)."""
    u = _f32(u)
    kappa = _f64(kappa)
    B, H, L = u.shape
    assert kappa.shape == (H, L)
    y = np.empty((B, H, L), np.float64)
    _load().orc_toeplitz_causal(B, H, L, _p(u), _p(kappa), _p(y), int(nthreads))
    return y


def dlr_bidirectional(u, fwd, bwd, nthreads: int = DEFAULT_THREADS) -> np.ndarray:
    """Bidirectional DLR (section 2.1): the sum of two independent DLRs, the second one run
    on the time-reversed sequence and its output reversed back. Lag 0 is counted by both."""
    u = _f32(u)
    y1 = dlr_recurrence(u, *fwd, nthreads=nthreads)
    y2 = dlr_recurrence(u[..., ::-1], *bwd, nthreads=nthreads)[..., ::-1]
    return y1 + y2


def dlr_prod_layer(u, fwd, bwd=None, nthreads: int = DEFAULT_THREADS) -> np.ndarray:
    """DLR-prod (section 2.1): kernel kappa_j = Re(K_j) * Im(K_j), applied by the direct
    Toeplitz sum; with ``bwd`` the anti-causal direction is added as in the bidirectional DLR."""
    u = _f32(u)
    L = u.shape[-1]
    k1 = dlr_kernel(*fwd, L, cast="re_im")
    y = toeplitz_causal(u, k1, nthreads)
    if bwd is not None:
        k2 = dlr_kernel(*bwd, L, cast="re_im")
        y = y + toeplitz_causal(np.ascontiguousarray(u[..., ::-1]), k2, nthreads)[..., ::-1]
    return y


def dlr_layer(u, fwd, bwd=None, cast: str = "re", nthreads: int = DEFAULT_THREADS):
    """The DLR layer as the pages define it for the given cast and direction(s).
    ``fwd``/``bwd`` are (log_re, log_im, W) tuples."""
    if cast == "re":
        if bwd is None:
            return dlr_recurrence(u, *fwd, nthreads=nthreads)
        return dlr_bidirectional(u, fwd, bwd, nthreads)
    return dlr_prod_layer(u, fwd, bwd, nthreads)


def dlr_backward(u, g, log_re, log_im, W, cast: str = "re"):
    """Gradients of the causal DLR layer with the Re cast (section 2: y_k = sum_{j<=k} Re K_j
    u_{k-j}, K_j = sum_n W_n lambda_n^j; section 2.2: lambda = exp(-a^2 + i theta) with
    a = (log Lambda)_re, theta = (log Lambda)_im) for a loss whose gradient with respect to
    y is g [B, H, L]. Written out from those definitions:
      du_k        = sum_{j <= L-1-k} Re K_j g_{k+j}           (the same DLR run backwards)
      c_j         = sum_b sum_k g_{b,k} u_{b,k-j}              (per channel, j < L)
      S0, S1      = sum_j c_j lambda^j,  sum_j j c_j lambda^j
      dW          = (Re S0, -Im S0)          since d Re K_j / d(W_re, W_im) = (Re, -Im) lambda^j
      d log_re    = -2 a Re(W S1)            since d lambda^j / da = -2 a j lambda^j
      d log_im    = -Im(W S1)                since d lambda^j / d theta = i j lambda^j
    With the DLR-prod cast (section 2.1: kappa_j = Re K_j Im K_j in place of Re K_j) the
    gradient with respect to kappa_j is again c_j, and through K it becomes, with
    T_j = c_j K_j: dW = (Im, Re) sum_j T_j lambda^j, d log_re = -2 a Im(W sum_j j T_j
    lambda^j), d log_im = Re(W sum_j j T_j lambda^j); du uses kappa in place of Re K.
    The convolution and correlation are numpy FFTs (zero-padded past 2L, so exact linear
    sums); lambda^j is exp(j (-a^2 + i theta)) evaluated directly. Returns float64 du
    [B, H, L], d_log_re [H, N], d_log_im [H, N], dW [H, N, 2]."""
    if cast not in ("re", "re_im"):
        raise ValueError(cast)
    u, g = _f32(u), _f64(g)
    log_re, log_im, W = _f32(log_re), _f32(log_im), _f32(W)
    B, H, L = u.shape
    N = log_re.shape[1]
    ud = u.astype(np.float64)
    M = 1 << int(np.ceil(np.log2(2 * L)))
    K = dlr_kernel(log_re, log_im, W, L, "complex")          # [H, L]
    kap = K.real if cast == "re" else K.real * K.imag        # the convolution kernel
    Kf = np.fft.rfft(kap, M, axis=-1)                        # [H, M/2+1]
    # du_k = sum_j ReK_j g_{k+j}: the causal convolution of the reversed g, reversed back
    gr = g[..., ::-1]
    du = np.fft.irfft(np.fft.rfft(gr, M, axis=-1) * Kf[None], M, axis=-1)[..., :L][..., ::-1]
    # c_j = sum_b sum_k g_k u_{k-j}
    c = np.fft.irfft((np.fft.rfft(g, M, axis=-1) * np.conj(np.fft.rfft(ud, M, axis=-1))).sum(0),
                     M, axis=-1)[:, :L]                      # [H, L]
    a = log_re.astype(np.float64)
    th = log_im.astype(np.float64)
    Wc = W[..., 0].astype(np.float64) + 1j * W[..., 1]
    j = np.arange(L, dtype=np.float64)
    d_re = np.empty((H, N))
    d_im = np.empty((H, N))
    dW = np.empty((H, N, 2))
    for h in range(H):
        z = -a[h] * a[h] + 1j * th[h]                        # log lambda, [N]
        P = np.exp(np.outer(z, j))                           # lambda^j, [N, L]
        wt = c[h] if cast == "re" else c[h] * K[h]           # c_j, or T_j = c_j K_j
        S0 = P @ wt
        S1 = P @ (j * wt)
        WS1 = Wc[h] * S1
        if cast == "re":
            dW[h, :, 0] = S0.real
            dW[h, :, 1] = -S0.imag
            d_re[h] = -2.0 * a[h] * WS1.real
            d_im[h] = -WS1.imag
        else:
            dW[h, :, 0] = S0.imag
            dW[h, :, 1] = S0.real
            d_re[h] = -2.0 * a[h] * WS1.imag
            d_im[h] = WS1.real
    return np.ascontiguousarray(du), d_re, d_im, dW


def dlr_layer_backward(u, g, fwd, bwd=None, cast: str = "re"):
    """Gradients of dlr_layer (causal, or bidirectional with a second parameter set: section
    2.1, y = DLR1(u) + rev(DLR2(rev(u)))) for the output gradient g. The second direction is
    the causal layer on the reversed sequences, so its gradients are those of dlr_backward on
    rev(u) and rev(g), and its input gradient enters du reversed. Returns du and a list of
    (d_log_re, d_log_im, dW) per direction."""
    du, dr, di, dw = dlr_backward(u, g, *fwd, cast=cast)
    grads = [(dr, di, dw)]
    if bwd is not None:
        ur = np.ascontiguousarray(_f32(u)[..., ::-1])
        gr = np.ascontiguousarray(_f64(g)[..., ::-1])
        du2, dr2, di2, dw2 = dlr_backward(ur, gr, *bwd, cast=cast)
        du = du + du2[..., ::-1]
        grads.append((dr2, di2, dw2))
    return np.ascontiguousarray(du), grads


def dlr_spectrum(log_re, log_im, W, L: int, M: int, bwd=None) -> np.ndarray:
    """Spectrum of the length-M circulant column of the Re-cast DLR kernel, bins k = 0..M/2,
    evaluated directly from the parameters ("The Annotated S4", part 2: the kernel's truncated
    generating function evaluated at the roots of unity instead of the kernel itself; for a
    diagonal state matrix it is a sum of geometric series). With omega = exp(-2 pi i / M) and
    A(k) = sum_n W_n G(lambda_n omega^k), G(z) = sum_{j<L} z^j = (1 - z^L) / (1 - z):
      causal column [K_0 .. K_{L-1}, 0 ..]:       C_k = (A(k) + conj(A(-k))) / 2
      with bwd, the anti-causal column K2_j at M - j (j >= 1) and K2_0 added at 0 (the
      bidirectional DLR of section 2.1 as one circulant): + (A2(-k) + conj(A2(k))) / 2.
    G is formed as expm1(L log z) / expm1(log z) with log z = -a^2 + i(theta - 2 pi k / M)
    (complex128), and as L where log z = 0. Returns complex128 [H, M/2 + 1]."""
    def A(lr, li, w, sign):
        lr, li, w = _f32(lr), _f32(li), _f32(w)
        a = lr.astype(np.float64)
        th = li.astype(np.float64)
        wc = w[..., 0].astype(np.float64) + 1j * w[..., 1].astype(np.float64)   # [H, N]
        k = np.arange(M // 2 + 1, dtype=np.float64)
        ell = (-a * a)[..., None] + 1j * (th[..., None] - sign * 2.0 * np.pi * k / M)
        ell = ell.real + 1j * (np.mod(ell.imag + np.pi, 2.0 * np.pi) - np.pi)     # [H, N, K]
        num = np.expm1(L * ell)
        den = np.expm1(ell)
        zero = np.abs(ell) == 0.0
        G = np.where(zero, float(L), num / np.where(zero, 1.0, den))
        return np.einsum("hn,hnk->hk", wc, G)
    C = 0.5 * (A(log_re, log_im, W, +1) + np.conj(A(log_re, log_im, W, -1)))
    if bwd is not None:
        C = C + 0.5 * (A(*bwd, -1) + np.conj(A(*bwd, +1)))
    return C


# ------------------------------------------------------------------------------------------
# S5 ("Simplified State Space Layers for Sequence Modeling")

def s5_zoh(lam, log_delta, Bt):
    """Zero-order hold of the diagonal system (section 3.2 'Discretization'), the standard
    diagonal ZOH: Lambda_bar = exp(Lambda Delta), B_bar = Lambda^{-1} (Lambda_bar - 1) B~,
    Delta = exp(log_delta) per state. Returns complex128 Lambda_bar [P], B_bar [P, H]."""
    lam = _f64(lam)
    lamc = lam[:, 0] + 1j * lam[:, 1]
    delta = np.exp(_f64(log_delta))
    abar = np.exp(lamc * delta)
    Bt = _f64(Bt)
    Btc = Bt[..., 0] + 1j * Bt[..., 1]
    bbar = ((abar - 1.0) / lamc)[:, None] * Btc
    return abar, bbar


def s5_bilinear(lam, log_delta, Bt):
    """Bilinear discretisation of the diagonal system ("The Annotated S4", part 1, the discrete
    SSM: A_bar = (I - Delta/2 A)^-1 (I + Delta/2 A), B_bar = (I - Delta/2 A)^-1 Delta B; S5
    section 2.1 lists it beside ZOH). For a diagonal A, per state with z = Lambda Delta:
    Lambda_bar = (1 + z/2) / (1 - z/2), B_bar = Delta / (1 - z/2) B~. Returns complex128
    Lambda_bar [P], B_bar [P, H]."""
    lam = _f64(lam)
    lamc = lam[:, 0] + 1j * lam[:, 1]
    delta = np.exp(_f64(log_delta))
    z = lamc * delta
    abar = (1.0 + 0.5 * z) / (1.0 - 0.5 * z)
    Bt = _f64(Bt)
    Btc = Bt[..., 0] + 1j * Bt[..., 1]
    bbar = (delta / (1.0 - 0.5 * z))[:, None] * Btc
    return abar, bbar


def s5_layer(u, lam, log_delta, Bt, Ct, D, disc: str = "zoh") -> np.ndarray:
    """S5 SSM outputs (sections 2.2 and 3): per batch row,
    x_k = Lambda_bar x_{k-1} + B_bar u_k (x_{-1} = 0), y_k = Re(C~ x_k) + D (.) u_k.
    u: [B, L, H] float32; disc 'zoh' (s5_zoh) or 'bilinear' (s5_bilinear). B_bar u_k is a
    library complex matmul over all k at once."""
    u = _f32(u)
    Bsz, L, H = u.shape
    if disc == "zoh":
        abar, bbar = s5_zoh(lam, log_delta, Bt)
    elif disc == "bilinear":
        abar, bbar = s5_bilinear(lam, log_delta, Bt)
    else:
        raise ValueError(disc)
    P = abar.shape[0]
    Ct = _f64(Ct)
    Ctc = Ct[..., 0] + 1j * Ct[..., 1]  # [H, P]
    D = _f64(D)
    ab = _f64(np.stack([abar.real, abar.imag], -1))
    y = np.empty((Bsz, L, H), np.float64)
    lib = _load()
    for b in range(Bsz):
        ub = u[b].astype(np.float64)
        v = ub @ bbar.T                                   # [L, P] complex
        va = _f64(np.stack([v.real, v.imag], -1))
        x = np.empty_like(va)
        lib.orc_diag_scan(L, P, _p(ab), _p(va), _p(x))
        xc = x[..., 0] + 1j * x[..., 1]
        y[b] = (xc @ Ctc.T).real + ub * D[None, :]
    return y


def s5_layer_tv(u, dt, lam, log_delta, Bt, Ct, D) -> np.ndarray:
    """S5 with a step that changes from step to step (S5 section 2.2: "supplying a different
    A_bar_k at each step" for irregularly sampled sequences; section 6.3). Reading: the
    observation gap dt_{b,k} > 0 (time since the previous sample, in units of the base step)
    scales each state's learned step, Delta_{p,k} = Delta_p dt_{b,k}, and every step is a ZOH:
      Lambda_bar_{p,k} = exp(Lambda_p Delta_{p,k}),  B_bar_{p,k} = (Lambda_bar_{p,k} - 1) / Lambda_p B~_p,
      x_k = Lambda_bar_k x_{k-1} + B_bar_k u_k,      y_k = Re(C~ x_k) + D (.) u_k.
    u: [B, L, H] float32, dt: [B, L] float32. Returns float64 [B, L, H]."""
    u = _f32(u)
    dt = _f32(dt)
    Bsz, L, H = u.shape
    lam = _f64(lam)
    lamc = lam[:, 0] + 1j * lam[:, 1]
    delta = np.exp(_f64(log_delta))
    Bt = _f64(Bt)
    Btc = Bt[..., 0] + 1j * Bt[..., 1]
    Ct = _f64(Ct)
    Ctc = Ct[..., 0] + 1j * Ct[..., 1]
    Dd = _f64(D)
    y = np.empty((Bsz, L, H), np.float64)
    lib = _load()
    for b in range(Bsz):
        z = lamc[None, :] * delta[None, :] * dt[b].astype(np.float64)[:, None]   # [L, P]
        abar = np.exp(z)
        f = np.expm1(z) / lamc[None, :]
        ub = u[b].astype(np.float64)
        v = (ub @ Btc.T) * f                                                     # [L, P]
        ab = _f64(np.stack([abar.real, abar.imag], -1))
        va = _f64(np.stack([v.real, v.imag], -1))
        x = np.empty_like(va)
        lib.orc_diag_scan_tv(L, lamc.shape[0], _p(ab), _p(va), _p(x))
        xc = x[..., 0] + 1j * x[..., 1]
        y[b] = (xc @ Ctc.T).real + ub * Dd[None, :]
    return y


# ------------------------------------------------------------------------------------------
# Other parameterisations of the DLR

def dss_exp_params(Lam, log_delta, W):
    """DSS_exp as a DLR ("Simplifying and Understanding State Space Models with Diagonal Linear
    RNNs", section 2: DSS_exp discretises the continuous diagonal state space x' = Lambda x + u,
    y = Re <W, x> with a zero-order hold over steps of size Delta, and the DLR of Eq. 1 drops
    Delta and the extra input scaling). Reading of the missing equations: the discrete state is
    x_k = exp(Delta Lambda) x_{k-1} + (exp(Delta Lambda) - 1) / Lambda u_k, which is the DLR with
    lambda = exp(Delta Lambda), i.e. (log Lambda)_re = sqrt(-Delta Re Lambda),
    (log Lambda)_im = Delta Im Lambda, and the scaling moved into the weights:
    W' = W (exp(Delta Lambda) - 1) / Lambda. Lam [H, N, 2], log_delta [H] (one step per
    channel), W [H, N, 2]. Returns float64 log_re, log_im [H, N] and W' [H, N, 2]."""
    Lam = _f64(Lam)
    Lc = Lam[..., 0] + 1j * Lam[..., 1]
    delta = np.exp(_f64(log_delta))[:, None]
    z = Lc * delta
    W = _f64(W)
    Wc = W[..., 0] + 1j * W[..., 1]
    Wn = Wc * np.expm1(z) / Lc
    return np.sqrt(-z.real), z.imag, np.stack([Wn.real, Wn.imag], -1)


def dss_exp_layer(u, Lam, log_delta, W) -> np.ndarray:
    """The DSS_exp layer by its definition: the zero-order-hold recurrence
    x_k = exp(Delta Lambda) x_{k-1} + (exp(Delta Lambda) - 1) / Lambda u_k (x_{-1} = 0),
    y_k = Re sum_n W_n x_{n,k}, for u [B, H, L] (complex128 arithmetic, a loop over k)."""
    u = _f32(u).astype(np.float64)
    Lam = _f64(Lam)
    Lc = Lam[..., 0] + 1j * Lam[..., 1]
    z = Lc * np.exp(_f64(log_delta))[:, None]
    a = np.exp(z)
    f = np.expm1(z) / Lc
    W = _f64(W)
    Wc = W[..., 0] + 1j * W[..., 1]
    B, H, L = u.shape
    x = np.zeros((B, H, Lc.shape[1]), complex)
    y = np.empty((B, H, L))
    for k in range(L):
        x = a[None] * x + f[None] * u[:, :, k, None]
        y[:, :, k] = (Wc[None] * x).sum(-1).real
    return y


def reparam_log_re(w, kind: str, a: float = 1.0, b: float = 1.0) -> np.ndarray:
    """(log Lambda)_re for a decay rate given by a reparameterisation f(w) of the recurrent
    weight (the StableSSM thread: lambda = f(w) with the exponential, softplus and 'best'
    f(w) = 1 / (a w^2 + b) maps). Reading: f(w) > 0 is the decay rate, |lambda| = exp(-f(w)),
    so with the DLR's |lambda| = exp(-(log Lambda)_re^2), (log Lambda)_re = sqrt(f(w)).
    kind: 'exp' (f = e^w), 'softplus' (f = log(1 + e^w)), 'best'. Returns float64."""
    w = _f64(w)
    if kind == "exp":
        f = np.exp(w)
    elif kind == "softplus":
        f = np.logaddexp(0.0, w)
    elif kind == "best":
        f = 1.0 / (a * w * w + b)
    else:
        raise ValueError(kind)
    return np.sqrt(f)


def rel_l2(y, y_ref) -> float:
    """||y - y_ref||_2 / ||y_ref||_2 over the whole tensor."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    den = np.linalg.norm(y_ref.ravel())
    num = np.linalg.norm((y - y_ref).ravel())
    return float(num / den) if den > 0 else float(num)
