"""Seeded synthetic inputs for the diagonal-linear-recurrence (DLR) and S5 workloads.

This module only draws random numbers and lays them out; it performs none of the
method's arithmetic (no powers of Lambda, no kernels, no convolutions, no scans).
Both the CUDA path and the float64 oracle consume exactly the float32 arrays made here.

Recipes (from "Simplifying and Understanding State Space Models with Diagonal Linear
RNNs", section 2.2 "Parameterization and initialization" and section 3.1 "Shift" task; and
"Simplified State Space Layers for Sequence Modeling", section 4.3 "Initialization"):

* DLR parameters per channel h and state n:
    (log Lambda)_re = sqrt(exp(r)/2),  r ~ U(log 5e-4, log 0.5)
    (log Lambda)_im = 2*pi*n/N
    Re W, Im W      ~ N(0, 1/N^2)
* DLR input u ~ N(0, 1); where the workload asks for it, each length-L sequence is divided
  by its own max-abs value (the Shift-task input distribution).
* S5 parameters: Lambda = eigenvalues of the HiPPO-N normal matrix (the normal part of the
  HiPPO-LegS matrix, as built in "The Annotated S4", part 2 "Turning HiPPO to DPLR"),
  log Delta ~ U(log 1e-3, log 1e-1) per state, Re/Im of B~ and C~ ~ N(0, 1/H), D ~ N(0, 1).

Draw order within one workload (a fixed reading, since the pages fix only "seed 0"):
``r -> W_re -> W_im`` for each direction in turn, then ``u``; for S5:
``log_delta -> B_re -> B_im -> C_re -> C_im -> D -> u``. All draws are float64 from
``numpy.random.default_rng(seed)`` and are cast to float32 afterwards.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# The five workloads the library is measured and checked on.
WORKLOADS = {
    "dlr_b1_h1_n16_l256": dict(kind="dlr", B=1, H=1, N=16, L=256, normalize=True,
                               bidir=False, cast="re", unit_channels=0, seed=0),
    "dlr_b8_h256_n64_l4096": dict(kind="dlr", B=8, H=256, N=64, L=4096, normalize=False,
                                  bidir=False, cast="re", unit_channels=0, seed=1),
    "dlrprod_bidir_b4_h128_n1024_l16384": dict(kind="dlr", B=4, H=128, N=1024, L=16384,
                                               normalize=True, bidir=True, cast="re_im",
                                               unit_channels=0, seed=2),
    "s5_b8_l16384_h512_p256": dict(kind="s5", B=8, L=16384, H=512, P=256, seed=3),
    "dlr_b1_h256_n64_l65536_unit8": dict(kind="dlr", B=1, H=256, N=64, L=65536,
                                         normalize=False, bidir=False, cast="re",
                                         unit_channels=8, seed=4),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclasses.dataclass
class DLRParams:
    """One direction of a DLR bank: arrays of shape [H, N] (W is [H, N, 2] = re, im)."""
    log_re: np.ndarray
    log_im: np.ndarray
    W: np.ndarray

    @property
    def H(self) -> int:
        return self.log_re.shape[0]

    @property
    def N(self) -> int:
        return self.log_re.shape[1]


@dataclasses.dataclass
class S5Params:
    lam: np.ndarray        # [P, 2] continuous-time eigenvalues (re, im)
    log_delta: np.ndarray  # [P]
    Bt: np.ndarray         # [P, H, 2]
    Ct: np.ndarray         # [H, P, 2]
    D: np.ndarray          # [H]


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float64) * std


def dlr_params(rng: np.random.Generator, H: int, N: int, unit_channels: int = 0) -> DLRParams:
    """Draw one direction's (log Lambda)_re, (log Lambda)_im and W for H channels of N states.

    The first ``unit_channels`` channels get (log Lambda)_re = 0, i.e. |lambda| = 1.
    """
    r = rng.uniform(np.log(5e-4), np.log(0.5), size=(H, N))
    log_re = np.sqrt(np.exp(r) / 2.0)
    if unit_channels:
        log_re[:unit_channels] = 0.0
    log_im = np.broadcast_to(2.0 * np.pi * np.arange(N) / N, (H, N))
    w_re = _normal(rng, (H, N), 1.0 / N)
    w_im = _normal(rng, (H, N), 1.0 / N)
    W = np.stack([w_re, w_im], axis=-1)
    return DLRParams(log_re.astype(np.float32), np.ascontiguousarray(log_im, dtype=np.float32),
                     W.astype(np.float32))


def dlr_input(rng: np.random.Generator, B: int, H: int, L: int, normalize: bool) -> np.ndarray:
    """u of shape [B, H, L], N(0,1); optionally each row divided by its max |u|."""
    u = rng.standard_normal((B, H, L), dtype=np.float64)
    if normalize:
        m = np.max(np.abs(u), axis=-1, keepdims=True)
        m[m == 0] = 1.0
        u = u / m
    return u.astype(np.float32)


def hippo_n_eigenvalues(P: int) -> np.ndarray:
    """Eigenvalues of the HiPPO-N matrix (normal part of HiPPO-LegS), returned [P, 2].

    HiPPO-LegS: A_nk = -sqrt(2n+1)sqrt(2k+1) (n>k), -(n+1) (n=k), 0 (n<k). Adding the rank-one
    term p p^T with p_n = sqrt(n + 1/2) leaves S = -1/2 I + (skew-symmetric). Its eigenvalues are
    -1/2 + i*mu with mu the eigenvalues of the Hermitian matrix -i*(S + I/2).
    """
    n = np.arange(P, dtype=np.float64)
    q = np.sqrt(2.0 * n + 1.0)
    A = -(np.tril(np.outer(q, q)) - np.diag(n))
    p = np.sqrt(n + 0.5)
    S = A + np.outer(p, p)
    re = np.mean(np.diagonal(S))
    mu = np.linalg.eigvalsh(-1j * (S - re * np.eye(P)))
    lam = np.stack([np.full(P, re), mu], axis=-1)
    return lam


def hippo_n_block_eigenvalues(P: int, J: int) -> np.ndarray:
    """Eigenvalues of the block-diagonal initialisation of S5 (section 4.3 and appendix D.4: J
    blocks on the diagonal, each the HiPPO-N matrix of size P / J): the J blocks' spectra one
    after the other, [P, 2]."""
    if P % J:
        raise ValueError("P must be a multiple of J")
    return np.concatenate([hippo_n_eigenvalues(P // J)] * J, axis=0)


def irregular_gaps(rng: np.random.Generator, B: int, L: int) -> np.ndarray:
    """Observation gaps for irregularly sampled sequences (the setting of S5 section 6.3): per
    batch row, L observation times drawn uniformly over [0, L) and sorted; dt_k is the time
    since the previous observation (since 0 for the first), so the mean gap is about 1.
    [B, L] float32."""
    t = np.sort(rng.uniform(0.0, float(L), size=(B, L)), axis=1)
    dt = np.diff(np.concatenate([np.zeros((B, 1)), t], axis=1), axis=1)
    return dt.astype(np.float32)


def s5_params(rng: np.random.Generator, H: int, P: int) -> S5Params:
    lam = hippo_n_eigenvalues(P)
    log_delta = rng.uniform(np.log(1e-3), np.log(1e-1), size=P)
    std = 1.0 / np.sqrt(H)
    b_re = _normal(rng, (P, H), std)
    b_im = _normal(rng, (P, H), std)
    c_re = _normal(rng, (H, P), std)
    c_im = _normal(rng, (H, P), std)
    D = rng.standard_normal(H, dtype=np.float64)
    return S5Params(lam.astype(np.float32), log_delta.astype(np.float32),
                    np.stack([b_re, b_im], -1).astype(np.float32),
                    np.stack([c_re, c_im], -1).astype(np.float32),
                    D.astype(np.float32))


def s5_input(rng: np.random.Generator, B: int, L: int, H: int) -> np.ndarray:
    return rng.standard_normal((B, L, H), dtype=np.float64).astype(np.float32)


@dataclasses.dataclass
class DLRWorkload:
    name: str
    B: int
    H: int
    N: int
    L: int
    bidir: bool
    cast: str
    fwd: DLRParams
    bwd: Optional[DLRParams]
    u: np.ndarray


@dataclasses.dataclass
class S5Workload:
    name: str
    B: int
    L: int
    H: int
    P: int
    params: S5Params
    u: np.ndarray


def make_dlr(B: int, H: int, N: int, L: int, *, seed: int, normalize: bool = False,
             bidir: bool = False, cast: str = "re", unit_channels: int = 0,
             name: str = "custom") -> DLRWorkload:
    rng = np.random.default_rng(seed)
    fwd = dlr_params(rng, H, N, unit_channels)
    bwd = dlr_params(rng, H, N, unit_channels) if bidir else None
    u = dlr_input(rng, B, H, L, normalize)
    return DLRWorkload(name, B, H, N, L, bidir, cast, fwd, bwd, u)


def make_s5(B: int, L: int, H: int, P: int, *, seed: int, name: str = "custom") -> S5Workload:
    rng = np.random.default_rng(seed)
    params = s5_params(rng, H, P)
    u = s5_input(rng, B, L, H)
    return S5Workload(name, B, L, H, P, params, u)


def make_workload(name: str):
    """Build one of the named workloads with its fixed seed."""
    cfg = dict(WORKLOADS[name])
    kind = cfg.pop("kind")
    seed = cfg.pop("seed")
    if kind == "dlr":
        return make_dlr(cfg["B"], cfg["H"], cfg["N"], cfg["L"], seed=seed,
                        normalize=cfg["normalize"], bidir=cfg["bidir"], cast=cfg["cast"],
                        unit_channels=cfg["unit_channels"], name=name)
    return make_s5(cfg["B"], cfg["L"], cfg["H"], cfg["P"], seed=seed, name=name)


def hippo_legs(P: int) -> np.ndarray:
    """The HiPPO-LegS state matrix (float64 [P, P]) as printed in "The Annotated S4",
    part 1b "The HiPPO matrix": A_nk = -sqrt(2n+1)sqrt(2k+1) (n>k), -(n+1) (n=k), 0 (n<k)."""
    n = np.arange(P, dtype=np.float64)
    q = np.sqrt(2.0 * n + 1.0)
    return -(np.tril(np.outer(q, q)) - np.diag(n))
