"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Tolerance: relative L2 error over the whole output tensor <= 1e-5 for the float32 tier
(the bar the workloads state), computed against the oracle's float64 result on the same
float32 inputs. Full-size workloads whose oracle is too slow are compared on sampled rows.
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


def params_dev(p):
    return dev(p.log_re), dev(p.log_im), dev(p.W)


def params_np(p):
    return p.log_re, p.log_im, p.W


def check_status():
    assert dlr.device_status() == 0


# ------------------------------------------------------------------------------------------
# dlr_kernel

# N >= 256 runs the tensor-core generator: a whole tile of 128 chunks, ragged blocks of
# states and a ragged last chunk, the DLR-prod shape, a tile that is mostly past L, and more
# states than one pass of the row-scale pre-pass takes (1024)
@pytest.mark.parametrize("H,N,L", [(1, 1, 1), (3, 5, 1000), (2, 16, 256), (4, 64, 4096),
                                   (2, 33, 4097), (2, 64, 70000), (2, 256, 8192), (3, 300, 5000),
                                   (1, 1024, 16384), (2, 257, 100), (2, 1100, 9000)])
@pytest.mark.parametrize("cast", ["re", "re_im"])
def test_kernel_matches_oracle(H, N, L, cast):
    w = inputs.make_dlr(1, H, N, 1, seed=H * 1000 + N, unit_channels=min(1, H))
    K = host(dlr.dlr_kernel(*params_dev(w.fwd), L, cast))
    ref = oracle.dlr_kernel(*params_np(w.fwd), L, cast=cast)
    assert oracle.rel_l2(K, ref) <= TOL
    check_status()


@pytest.mark.parametrize("N", [64, 256, 512])
def test_kernel_dft_identity_on_gpu(N):
    """(log Lambda)_re = 0, theta_n = 2 pi n / N, L = N: K = N * IDFT(w) (real part); N >= 256
    on the tensor-core generator, all states on the unit circle."""
    rng = np.random.default_rng(5)
    log_re = np.zeros((1, N), np.float32)
    log_im = (2 * np.pi * np.arange(N) / N).astype(np.float32)[None]
    W = rng.standard_normal((1, N, 2)).astype(np.float32)
    K = host(dlr.dlr_kernel(dev(log_re), dev(log_im), dev(W), N, "re"))[0]
    ref = oracle.dlr_kernel(log_re, log_im, W, N, cast="re")[0]
    assert oracle.rel_l2(K, ref) <= TOL
    w = W[0, :, 0].astype(np.float64) + 1j * W[0, :, 1]
    assert oracle.rel_l2(K, (N * np.fft.ifft(w)).real) <= 1e-4  # float32 theta, see pins


# ------------------------------------------------------------------------------------------
# dlr_conv (given kernels) and dlr_scan on small and ragged shapes

@pytest.mark.parametrize("B,H,L", [(1, 1, 1), (1, 1, 2), (2, 3, 3), (1, 2, 5), (2, 2, 64),
                                   (3, 2, 100), (1, 3, 1000), (2, 2, 4095), (1, 2, 4096),
                                   (1, 1, 8192), (1, 1, 16383), (1, 2, 16384),
                                   # two rows per transform (B >= 2, 1024 < L <= 8192), odd B
                                   (3, 2, 1025), (2, 1, 2048), (3, 1, 5000), (2, 2, 8192),
                                   (5, 1, 4096)])
@pytest.mark.parametrize("bidir", [False, True])
def test_conv_matches_oracle_toeplitz(B, H, L, bidir):
    rng = np.random.default_rng(B * 7 + H * 11 + L)
    u = rng.standard_normal((B, H, L)).astype(np.float32)
    K1 = (rng.standard_normal((H, L)) * np.exp(-np.arange(L) / 300.0)).astype(np.float32)
    K2 = (rng.standard_normal((H, L)) * np.exp(-np.arange(L) / 500.0)).astype(np.float32)
    y = host(dlr.dlr_conv(dev(u), dev(K1), dev(K2) if bidir else None))
    ref = oracle.toeplitz_causal(u, K1.astype(np.float64))
    if bidir:
        ref = ref + oracle.toeplitz_causal(np.ascontiguousarray(u[..., ::-1]),
                                           K2.astype(np.float64))[..., ::-1]
    assert oracle.rel_l2(y, ref) <= TOL
    check_status()


@pytest.mark.parametrize("B,H,L", [(1, 1, 16385), (2, 1, 20000), (1, 2, 32768), (1, 1, 40001),
                                   (1, 1, 65536)])
@pytest.mark.parametrize("bidir", [False, True])
def test_conv_long_rows_cluster_path(B, H, L, bidir):
    """Rows longer than 16384: the transform is spread over a cluster of 8 CTAs."""
    rng = np.random.default_rng(B * 5 + H * 13 + L)
    u = rng.standard_normal((B, H, L)).astype(np.float32)
    K1 = (rng.standard_normal((H, L)) * np.exp(-np.arange(L) / 3000.0)).astype(np.float32)
    K2 = (rng.standard_normal((H, L)) * np.exp(-np.arange(L) / 9000.0)).astype(np.float32)
    y = host(dlr.dlr_conv(dev(u), dev(K1), dev(K2) if bidir else None))
    ref = oracle.toeplitz_causal(u, K1.astype(np.float64))
    if bidir:
        ref = ref + oracle.toeplitz_causal(np.ascontiguousarray(u[..., ::-1]),
                                           K2.astype(np.float64))[..., ::-1]
    assert oracle.rel_l2(y, ref) <= TOL
    check_status()


@pytest.mark.parametrize("B,H,N,L", [(1, 1, 1, 1), (1, 1, 1, 7), (2, 3, 5, 63), (1, 2, 16, 64),
                                     (2, 2, 16, 65), (1, 2, 64, 4095), (1, 2, 64, 4097),
                                     (2, 1, 65, 1000), (1, 2, 128, 5000), (1, 1, 64, 12289)])
@pytest.mark.parametrize("bidir", [False, True])
@pytest.mark.parametrize("algo", ["fp32", "tensor"])
def test_scan_matches_oracle(B, H, N, L, bidir, algo):
    if algo == "tensor" and N > 64:
        pytest.skip("the tensor-core scan holds at most 64 states")
    w = inputs.make_dlr(B, H, N, L, seed=B + 10 * H + 100 * N + L, bidir=bidir,
                        unit_channels=1)
    bwd_d = params_dev(w.bwd) if bidir else None
    y = host(dlr.dlr_scan(dev(w.u), params_dev(w.fwd), bwd_d, algo=algo))
    ref = oracle.dlr_layer(w.u, params_np(w.fwd), params_np(w.bwd) if bidir else None)
    assert oracle.rel_l2(y, ref) <= TOL
    check_status()


@pytest.mark.parametrize("B,H,N,L", [(5, 3, 64, 256), (3, 2, 40, 3000), (9, 2, 64, 8192),
                                     (2, 2, 64, 8193), (1, 3, 64, 30000), (2, 1, 8, 100)])
@pytest.mark.parametrize("bidir", [False, True])
def test_tensor_scan_tile_layouts(B, H, N, L, bidir):
    """Tensor-core scan: several rows packed in one tile (L <= 8192: floor(128 / chunks) rows
    per tile, ragged last tile), rows that walk several tiles with their state carried
    (L > 8192), ragged last chunks, N < 64 (zero state rows)."""
    w = inputs.make_dlr(B, H, N, L, seed=7 * B + 11 * H + N + L, bidir=bidir, unit_channels=1)
    bwd_d = params_dev(w.bwd) if bidir else None
    y = host(dlr.dlr_scan(dev(w.u), params_dev(w.fwd), bwd_d, algo="tensor"))
    ref = oracle.dlr_layer(w.u, params_np(w.fwd), params_np(w.bwd) if bidir else None)
    assert oracle.rel_l2(y, ref) <= TOL
    check_status()


def test_tensor_scan_input_scaling_extremes():
    """Per-chunk power-of-two scaling of u before the f16 split: rows of very different
    magnitude (1e-30 .. 1e30) and exactly zero chunks stay within the tolerance row by row."""
    B, H, N, L = 4, 2, 64, 4096
    w = inputs.make_dlr(B, H, N, L, seed=99, unit_channels=1)
    u = w.u.copy()
    u[0] *= 1e-30
    u[1] *= 1e30
    u[2, :, 1024:2048] = 0.0
    y = host(dlr.dlr_scan(dev(u), params_dev(w.fwd), algo="tensor"))
    ref = oracle.dlr_layer(u, params_np(w.fwd))
    for b in range(B):
        assert oracle.rel_l2(y[b], ref[b]) <= TOL, b
    check_status()


@pytest.mark.parametrize("B,H,N,L,bidir", [(8, 160, 16, 4096, False), (6, 300, 8, 2048, False),
                                           (4, 200, 8, 4096, True), (2, 100, 8, 16384, False),
                                           (2, 90, 4, 12288, True)])
def test_tensor_scan_channel_changes_inside_a_cta(B, H, N, L, bidir):
    """More tiles than SMs: each persistent CTA walks several tiles and crosses channels, so
    the per-channel operands (Q, the Toeplitz block, G) are replaced between tiles while
    earlier tiles of the old channel may still be in flight; both directions (the reversed
    pass adds through TMA reductions), rows packed in tiles and rows walked tile by tile."""
    w = inputs.make_dlr(B, H, N, L, seed=B + H + N, bidir=bidir, unit_channels=1)
    bwd_d = params_dev(w.bwd) if bidir else None
    y = host(dlr.dlr_scan(dev(w.u), params_dev(w.fwd), bwd_d, algo="tensor"))
    ref = oracle.dlr_layer(w.u, params_np(w.fwd), params_np(w.bwd) if bidir else None)
    assert oracle.rel_l2(y, ref) <= TOL
    # row by row as well: a wrong tile is a few rows among many
    err = np.linalg.norm(y - ref, axis=2) / np.maximum(np.linalg.norm(ref, axis=2), 1e-30)
    assert err.max() <= 1e-4, np.argwhere(err > 1e-4)[:8]
    check_status()


@pytest.mark.parametrize("B,H,N,L", [(8, 16, 64, 4096), (3, 2, 40, 3000), (1, 2, 64, 20000)])
def test_scan_prepare_apply_equals_scan(B, H, N, L):
    """dlr_scan_prepare + dlr_scan_apply (tables once, reused for several batches, both
    directions) give exactly what dlr_scan's tensor-core path gives, and match the oracle."""
    w = inputs.make_dlr(B, H, N, L, seed=3 * B + H + N + L, bidir=True, unit_channels=1)
    u = dev(w.u)
    fwd, bwd = params_dev(w.fwd), params_dev(w.bwd)
    ws_f = dlr.dlr_scan_prepare(fwd, B=B, L=L)
    ws_b = dlr.dlr_scan_prepare(bwd, B=B, L=L)
    for rep in range(2):  # the tables are only read: a second batch through them is the same
        y = dlr.dlr_scan_apply(u, ws_f, N)
        y = dlr.dlr_scan_apply(u, ws_b, N, out=y, reverse=True)
        y_ref = dlr.dlr_scan(u, fwd, bwd, algo="tensor")
        assert torch.equal(y, y_ref), rep
    ref = oracle.dlr_layer(w.u, params_np(w.fwd), params_np(w.bwd))
    assert oracle.rel_l2(host(y), ref) <= TOL
    check_status()


# pieces: 4 x 2 batch rows (TMA path); channel groups of a batch row (B < 4); channel groups
# with rows off the 64-step grid (plain-load path); one piece (L % 4 != 0)
@pytest.mark.parametrize("B,H,N,L", [(8, 16, 64, 4096), (2, 6, 16, 512), (1, 5, 8, 1000),
                                     (3, 2, 4, 33)])
def test_scan_host_buffers_match_oracle_and_device_path(B, H, N, L):
    """dlr_scan_host on pinned host buffers (pieces copied in, computed and copied out on three
    streams) matches the oracle and the device-buffer tensor-core path."""
    w = inputs.make_dlr(B, H, N, L, seed=5 * B + H + N + L, unit_channels=1)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    u_h = pin(w.u)
    p_h = tuple(pin(a) for a in (w.fwd.log_re, w.fwd.log_im, w.fwd.W))
    y_h = torch.zeros(u_h.shape, dtype=torch.float32).pin_memory()
    ws = torch.empty(dlr.dlr_scan_host_workspace_size(B, H, N, L), dtype=torch.uint8,
                     device="cuda")
    for rep in range(2):
        dlr.dlr_scan_host(u_h, p_h, y_h, ws)
        torch.cuda.current_stream().synchronize()
        ref = oracle.dlr_layer(w.u, params_np(w.fwd))
        assert oracle.rel_l2(y_h.numpy(), ref) <= TOL, rep
    y_dev = host(dlr.dlr_scan(dev(w.u), params_dev(w.fwd), algo="tensor"))
    assert oracle.rel_l2(y_h.numpy(), y_dev) <= 1e-6
    check_status()


# ------------------------------------------------------------------------------------------
# dlr_scan_backward_input (the layer's input gradient)

# rows off the 64-step grid (plain loads), the bank shape (TMA), rows longer than a tile
@pytest.mark.parametrize("B,H,N,L", [(2, 3, 5, 37), (8, 16, 64, 4096), (1, 2, 64, 20000),
                                     (3, 2, 40, 3000)])
def test_backward_input_matches_oracle(B, H, N, L):
    """du for an output gradient g: the layer run backwards on g with the same parameters,
    against the oracle's gradient of sum(g * y) with respect to u."""
    w = inputs.make_dlr(B, H, N, L, seed=11 * B + H + N + L, unit_channels=1)
    g = np.random.default_rng(B + L).standard_normal((B, H, L)).astype(np.float32)
    du = dlr.dlr_scan_backward_input(dev(g), params_dev(w.fwd))
    ref, _, _, _ = oracle.dlr_backward(w.u, g.astype(np.float64), *params_np(w.fwd))
    assert oracle.rel_l2(host(du), ref) <= TOL
    check_status()


# ------------------------------------------------------------------------------------------
# dlr_step (the recurrence advanced from a carried state)

def _step_pieces(u_d, ws, x, pieces):
    ys, t = [], 0
    for n in pieces:
        ys.append(dlr.dlr_step(u_d[:, :, t:t + n].contiguous(), ws, x))
        t += n
    assert t == u_d.shape[2]
    return torch.cat(ys, dim=2)


# states per lane 1, 2, 4, 8 with ragged last lanes; pieces of 1, across and on the 32-sample
# blocks, empty, and longer than several blocks
@pytest.mark.parametrize("B,H,N", [(2, 3, 5), (3, 2, 33), (8, 16, 64), (1, 4, 129), (2, 2, 256)])
def test_step_pieces_match_oracle(B, H, N):
    """Feeding a sequence in pieces through dlr_step, starting from zero, gives the oracle's
    outputs of the whole sequence and its final state."""
    pieces = [1, 1, 5, 31, 32, 33, 0, 100, 257]
    L = sum(pieces)
    w = inputs.make_dlr(B, H, N, L, seed=7 * B + H + N, unit_channels=1)
    ws = dlr.dlr_step_prepare(params_dev(w.fwd))
    x = torch.zeros((B, H, N, 2), dtype=torch.float32, device="cuda")
    y = _step_pieces(dev(w.u), ws, x, pieces)
    y_ref, x_ref = oracle.dlr_recurrence(w.u, *params_np(w.fwd), return_state=True)
    assert oracle.rel_l2(host(y), y_ref) <= TOL
    xs = host(x)
    assert oracle.rel_l2(xs, np.stack([x_ref.real, x_ref.imag], -1)) <= TOL  # (re, im) pairs
    check_status()


def test_step_from_a_given_state():
    """A nonzero carried state: y and the final state follow the oracle's recurrence from the
    same initial state."""
    B, H, N, L = 3, 5, 40, 300
    w = inputs.make_dlr(B, H, N, L, seed=41, unit_channels=1)
    rng = np.random.default_rng(42)
    x0 = (rng.standard_normal((B, H, N, 2)) * 3).astype(np.float32)
    ws = dlr.dlr_step_prepare(params_dev(w.fwd))
    x = dev(x0)
    y = dlr.dlr_step(dev(w.u), ws, x)
    x0c = x0[..., 0].astype(np.float64) + 1j * x0[..., 1]
    y_ref, x_ref = oracle.dlr_recurrence(w.u, *params_np(w.fwd), x0=x0c, return_state=True)
    assert oracle.rel_l2(host(y), y_ref) <= TOL
    xs = host(x)
    assert oracle.rel_l2(xs, np.stack([x_ref.real, x_ref.imag], -1)) <= TOL  # (re, im) pairs
    check_status()


def test_step_bank_and_long_unit_circle_stream():
    """The B=8 H=256 N=64 L=4096 bank fed in pieces of 512, and a stream of 16384 samples
    through 16 channels of which 8 sit at |lambda| = 1, fed in pieces of 4096: both against
    the oracle (the step path agrees with the chunked scan through it)."""
    w = inputs.make_workload("dlr_b8_h256_n64_l4096")
    ws = dlr.dlr_step_prepare(params_dev(w.fwd))
    x = torch.zeros((w.B, w.H, w.N, 2), dtype=torch.float32, device="cuda")
    y = _step_pieces(dev(w.u), ws, x, [512] * 8)
    assert oracle.rel_l2(host(y), oracle.dlr_layer(w.u, params_np(w.fwd))) <= TOL
    w = inputs.make_dlr(1, 16, 64, 16384, seed=43, unit_channels=8)
    ws = dlr.dlr_step_prepare(params_dev(w.fwd))
    x = torch.zeros((1, 16, 64, 2), dtype=torch.float32, device="cuda")
    y = _step_pieces(dev(w.u), ws, x, [4096] * 4)
    assert oracle.rel_l2(host(y), oracle.dlr_layer(w.u, params_np(w.fwd))) <= TOL
    check_status()


@pytest.mark.parametrize("bidir", [False, True])
def test_fft_and_scan_layers_agree_small(bidir):
    w = inputs.make_dlr(2, 4, 32, 3000, seed=77, bidir=bidir, unit_channels=1)
    bwd_d = params_dev(w.bwd) if bidir else None
    y_fft = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), bwd_d, path="fft"))
    y_scan = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), bwd_d, path="scan"))
    ref = oracle.dlr_layer(w.u, params_np(w.fwd), params_np(w.bwd) if bidir else None)
    assert oracle.rel_l2(y_fft, ref) <= TOL
    assert oracle.rel_l2(y_scan, ref) <= TOL
    assert oracle.rel_l2(y_fft, y_scan) <= TOL


# ------------------------------------------------------------------------------------------
# the named workloads at full size

@pytest.fixture(scope="module")
def wl_small():
    return inputs.make_workload("dlr_b1_h1_n16_l256")


@pytest.fixture(scope="module")
def wl_bank():
    return inputs.make_workload("dlr_b8_h256_n64_l4096")


def test_workload_single_channel(wl_small):
    w = wl_small
    ref = oracle.dlr_layer(w.u, params_np(w.fwd))
    for path in ("fft", "scan"):
        y = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), path=path))
        assert oracle.rel_l2(y, ref) <= TOL, path


def test_workload_bank_b8_h256_n64_l4096(wl_bank):
    w = wl_bank
    ref = oracle.dlr_layer(w.u, params_np(w.fwd))
    y_fft = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), path="fft"))
    y_scan = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), path="scan"))
    assert oracle.rel_l2(y_fft, ref) <= TOL
    assert oracle.rel_l2(y_scan, ref) <= TOL
    assert oracle.rel_l2(y_fft, y_scan) <= TOL
    check_status()


def sampled_channels(param_sets, count, seed):
    """A seeded subset of channels: the two whose slowest state is closest to |lambda| = 1
    (the smallest (log Lambda)_re^2 over the channel's states in any of the parameter sets,
    the hard case for long kernels) and count - 2 more drawn without replacement from the rest."""
    slowest = np.min([np.min(np.asarray(p.log_re, np.float64) ** 2, axis=1)
                      for p in param_sets], axis=0)
    near = np.argsort(slowest)[:2]
    rest = np.setdiff1d(np.arange(slowest.shape[0]), near)
    drawn = np.random.default_rng(seed).choice(rest, size=count - 2, replace=False)
    return np.sort(np.concatenate([near, drawn])).astype(np.int64)


def test_workload_prod_bidir_sampled_rows():
    """DLR-prod, bidirectional, B=4 H=128 N=1024 L=16384: the GPU runs the full layer; the
    oracle (direct O(L^2) Toeplitz sums) checks 8 seeded channels, including the two with
    the slowest-decaying states, on all 4 batch rows, together and one by one."""
    w = inputs.make_workload("dlrprod_bidir_b4_h128_n1024_l16384")
    y = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), params_dev(w.bwd), cast="re_im"))
    hs = sampled_channels([w.fwd, w.bwd], 8, 11)
    sub = lambda p: (p.log_re[hs], p.log_im[hs], p.W[hs])
    ref = oracle.dlr_prod_layer(np.ascontiguousarray(w.u[:, hs]), sub(w.fwd), sub(w.bwd))
    assert oracle.rel_l2(y[:, hs], ref) <= TOL
    for i in range(len(hs)):
        assert oracle.rel_l2(y[:, hs[i]], ref[:, i]) <= TOL
    assert np.all(np.isfinite(y))
    check_status()


def test_workload_long_unit_circle_scan():
    """B=1 H=256 N=64 L=65536, 8 channels at |lambda| = 1: chunked scan vs the oracle."""
    w = inputs.make_workload("dlr_b1_h256_n64_l65536_unit8")
    y = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), path="scan"))
    ref = oracle.dlr_layer(w.u, params_np(w.fwd))
    assert oracle.rel_l2(y, ref) <= TOL
    # the unit-circle channels alone (they dominate the norm, and are the hard case)
    assert oracle.rel_l2(y[:, :8], ref[:, :8]) <= TOL
    check_status()


def test_workload_long_unit_circle_fft_and_scan():
    """B=1 H=256 N=64 L=65536: the FFT path (2L = 131072, cluster transform) against the oracle,
    and FFT and scan paths against each other."""
    w = inputs.make_workload("dlr_b1_h256_n64_l65536_unit8")
    y_fft = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), path="fft"))
    y_scan = host(dlr.dlr_layer(dev(w.u), params_dev(w.fwd), path="scan"))
    ref = oracle.dlr_layer(w.u, params_np(w.fwd))
    assert oracle.rel_l2(y_fft, ref) <= TOL
    assert oracle.rel_l2(y_fft[:, :8], ref[:, :8]) <= TOL
    assert oracle.rel_l2(y_fft, y_scan) <= TOL
    check_status()


# ------------------------------------------------------------------------------------------
# S5

def s5_dev(p):
    return dev(p.lam), dev(p.log_delta), dev(p.Bt), dev(p.Ct), dev(p.D)


def s5_np(p):
    return p.lam, p.log_delta, p.Bt, p.Ct, p.D


@pytest.mark.parametrize("B,L,H,P", [(1, 1, 32, 32), (2, 63, 32, 32), (1, 200, 64, 32),
                                     (2, 1000, 96, 64)])
def test_s5_fp32_matches_oracle(B, L, H, P):
    w = inputs.make_s5(B, L, H, P, seed=B + L + H + P)
    y = host(dlr.s5_layer(dev(w.u), *s5_dev(w.params)))
    ref = oracle.s5_layer(w.u, *s5_np(w.params))
    assert oracle.rel_l2(y, ref) <= TOL
    check_status()


S5_ROWS = np.sort(np.random.default_rng(5).choice(8, size=2, replace=False))


def test_s5_workload_fp32_sampled_batch_row():
    """B=8 L=16384 H=512 P=256: the GPU runs the full layer; the oracle checks two seeded
    batch rows."""
    w = inputs.make_workload("s5_b8_l16384_h512_p256")
    y = host(dlr.s5_layer(dev(w.u), *s5_dev(w.params)))
    ref = oracle.s5_layer(np.ascontiguousarray(w.u[S5_ROWS]), *s5_np(w.params))
    assert oracle.rel_l2(y[S5_ROWS], ref) <= TOL
    for i, b in enumerate(S5_ROWS):
        assert oracle.rel_l2(y[b], ref[i]) <= TOL
    assert np.all(np.isfinite(y))
    check_status()


TOL_BF16 = 1e-2  # the bf16 tensor-core tier's bar


def state_part(y, u, D):
    """y - D (.) u in float64: the part the two projections and the scan produce (D (.) u is
    most of the norm of y on these inputs, so it would hide errors in that part)."""
    return np.asarray(y, np.float64) - np.asarray(u, np.float64) * np.asarray(D, np.float64)


# (3, 7000, 64, 32): 165 row tiles, more than there are SMs, so CTAs of the persistent GEMM
# take several tiles, the last one ragged. L a multiple of 64 takes the output projection with
# the scan's apply step fused in: (3, 64, 64, 32) has tiles spanning two batch rows and a
# ragged last tile, (2, 640, 96, 64) and (1, 192, 32, 32) several chunks per row; (1, 256, 64,
# 512) and (2, 128, 96, 1024) run the in-place apply over 16 and 32 blocks of states (P up to the
# limit of 1024).
@pytest.mark.parametrize("B,L,H,P", [(1, 1, 32, 32), (1, 200, 64, 32), (2, 1000, 96, 64),
                                     (1, 300, 512, 256), (3, 7000, 64, 32), (3, 64, 64, 32),
                                     (2, 640, 96, 64), (1, 192, 32, 32), (2, 4096, 512, 256),
                                     (1, 256, 64, 512), (2, 128, 96, 1024)])
def test_s5_bf16_tensor_cores_match_oracle(B, L, H, P):
    w = inputs.make_s5(B, L, H, P, seed=7 * B + L + H + P)
    y = host(dlr.s5_layer(dev(w.u), *s5_dev(w.params), prec="bf16"))
    ref = oracle.s5_layer(w.u, *s5_np(w.params))
    assert oracle.rel_l2(y, ref) <= TOL_BF16
    D = w.params.D
    assert oracle.rel_l2(state_part(y, w.u, D), state_part(ref, w.u, D)) <= TOL_BF16
    check_status()


def test_s5_workload_bf16_sampled_batch_row():
    w = inputs.make_workload("s5_b8_l16384_h512_p256")
    y = host(dlr.s5_layer(dev(w.u), *s5_dev(w.params), prec="bf16"))
    rows = np.sort(np.random.default_rng(6).choice(8, size=2, replace=False))
    u2, D = np.ascontiguousarray(w.u[rows]), w.params.D
    ref = oracle.s5_layer(u2, *s5_np(w.params))
    assert oracle.rel_l2(y[rows], ref) <= TOL_BF16
    assert oracle.rel_l2(state_part(y[rows], u2, D), state_part(ref, u2, D)) <= TOL_BF16
    assert np.all(np.isfinite(y))
    check_status()
