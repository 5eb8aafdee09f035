"""Thin Python binding over libdlr.so (include/dlr.h): argument marshalling only.

Every compute step runs in the library's CUDA kernels; this module passes device pointers,
sizes and the current torch CUDA stream, and turns non-zero status codes into exceptions.
There is no CPU fallback: if the library cannot be loaded, or a tensor is not a float32 CUDA
tensor, the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

DLR_OK, DLR_ERR_INVALID_ARG, DLR_ERR_UNSUPPORTED, DLR_ERR_CUDA, DLR_ERR_TIMEOUT, \
    DLR_ERR_WORKSPACE = range(6)
CAST = {"re": 0, "re_im": 1}
PREC = {"fp32": 0, "bf16": 1}

_lib = None


class DLRError(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = _load().dlr_status_string(status).decode() if _lib is not None else str(status)
        if status == DLR_ERR_CUDA and _lib is not None:
            name += " (" + _lib.dlr_last_cuda_error().decode() + ")"
        super().__init__(f"{fn} failed: {name}")
        self.status = status


def _checked() -> bool:
    """The bounds-checked library is loaded instead of the normal one when the environment
    variable DLR_BOUNDS_CHECK is 1 at the first call."""
    return os.environ.get("DLR_BOUNDS_CHECK", "0") == "1"


def _load():
    global _lib
    if _lib is None:
        path = _build.build(checked=_checked())
        lib = ctypes.CDLL(path)
        P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.dlr_kernel.argtypes = [P, P, P, i64, i64, i64, i32, P, P]
        lib.dlr_kernel.restype = i32
        lib.dlr_conv_workspace_size.argtypes = [i64, i64, i32]
        lib.dlr_conv_workspace_size.restype = sz
        lib.dlr_conv.argtypes = [P, P, P, i32, i64, i64, i64, P, P, sz, P]
        lib.dlr_conv.restype = i32
        lib.dlr_conv_spectrum.argtypes = [P, P, i32, i64, i64, P, sz, P]
        lib.dlr_conv_spectrum.restype = i32
        lib.dlr_conv_apply.argtypes = [P, i64, i64, i64, P, P, sz, P]
        lib.dlr_conv_spectrum_direct.argtypes = [P, P, P, P, P, P, i32, i64, i64, i64, P, sz, P]
        lib.dlr_conv_apply.restype = i32
        lib.dlr_scan_workspace_size.argtypes = [i64, i64, i64, i64]
        lib.dlr_scan_workspace_size.restype = sz
        lib.dlr_scan.argtypes = [P, P, P, P, P, P, P, i32, i64, i64, i64, i64, P, P, sz, P]
        lib.dlr_scan.restype = i32
        lib.dlr_scan_ex.argtypes = [P, P, P, P, P, P, P, i32, i64, i64, i64, i64, P, i32, P, sz,
                                    P]
        lib.dlr_scan_ex.restype = i32
        lib.dlr_scan_prepare.argtypes = [P, P, P, i64, i64, P, sz, P]
        lib.dlr_scan_prepare.restype = i32
        lib.dlr_scan_apply.argtypes = [P, i64, i64, i64, i64, i32, P, P, sz, P]
        lib.dlr_scan_apply.restype = i32
        lib.dlr_scan_host_workspace_size.argtypes = [i64, i64, i64, i64]
        lib.dlr_scan_host_workspace_size.restype = sz
        lib.dlr_scan_host.argtypes = [P, P, P, P, i64, i64, i64, i64, P, P, sz, P]
        lib.dlr_scan_host.restype = i32
        lib.dlr_scan_backward_input.argtypes = [P, P, P, P, i64, i64, i64, i64, P, P, sz, P]
        lib.dlr_scan_backward_params_workspace_size.argtypes = [i64, i64, i64, i64]
        lib.dlr_scan_backward_params_workspace_size.restype = sz
        lib.dlr_scan_backward_params.argtypes = [P, P, P, P, P, i64, i64, i64, i64, P, P, P, P,
                                                 sz, P]
        lib.dlr_scan_backward_params.restype = i32
        lib.dlr_layer_backward_workspace_size.argtypes = [i64, i64, i64, i64, i32, i32]
        lib.dlr_layer_backward_workspace_size.restype = sz
        lib.dlr_layer_backward.argtypes = [P] * 8 + [i32, i32] + [i64] * 4 + [P] * 8 + [sz, P]
        lib.dlr_layer_backward.restype = i32
        lib.dlr_scan_backward_input.restype = i32
        lib.dlr_step_workspace_size.argtypes = [i64, i64]
        lib.dlr_step_workspace_size.restype = sz
        lib.dlr_step_prepare.argtypes = [P, P, P, i64, i64, P, sz, P]
        lib.dlr_step_prepare.restype = i32
        lib.dlr_step.argtypes = [P, i64, i64, i64, i64, P, P, P, sz, P]
        lib.dlr_step.restype = i32
        lib.s5_workspace_size.argtypes = [i64, i64, i64, i64, i32]
        lib.s5_workspace_size.restype = sz
        lib.s5_layer.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64, i32, P, P, sz, P]
        lib.s5_layer_ex.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64, i32, i32, P, P, sz, P]
        lib.s5_layer_ex.restype = i32
        lib.s5_layer_tv_workspace_size.argtypes = [i64, i64, i64, i64]
        lib.s5_layer_tv_workspace_size.restype = sz
        lib.s5_layer_tv.argtypes = [P, P, P, P, P, P, P, i64, i64, i64, i64, P, P, sz, P]
        lib.s5_layer_tv.restype = i32
        lib.dlr_params_from_dss_exp.argtypes = [P, P, P, i64, i64, P, P, P, P]
        lib.dlr_params_from_dss_exp.restype = i32
        lib.dlr_log_re_from_reparam.argtypes = [P, i64, i32, ctypes.c_float, ctypes.c_float, P, P]
        lib.dlr_log_re_from_reparam.restype = i32
        lib.s5_layer.restype = i32
        lib.dlr_selftest_timeout.argtypes = [i32, P]
        lib.dlr_selftest_timeout.restype = i32
        lib.dlr_get_device_status.argtypes = [P]
        lib.dlr_get_device_status.restype = i32
        lib.dlr_status_string.argtypes = [i32]
        lib.dlr_status_string.restype = ctypes.c_char_p
        lib.dlr_abi_version.restype = i32
        lib.dlr_bounds_checked.restype = i32
        lib.dlr_bounds_site.restype = i32
        lib.dlr_selftest_bounds.argtypes = [P]
        lib.dlr_selftest_bounds.restype = i32
        lib.dlr_last_cuda_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def library_path() -> str:
    """Absolute path of the loaded library (loads it if needed)."""
    _load()
    return os.path.abspath(_build.LIB_CHECKED if _checked() else _build.LIB)


def bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(_load().dlr_bounds_checked())


def bounds_site() -> int:
    """Synchronise; return and clear the first failing site of the bounds-checked build
    (file number * 100000 + source line; 0 if none)."""
    return int(_load().dlr_bounds_site())


def selftest_bounds(stream=None) -> None:
    """Checked build: run the self-test whose one out-of-range read the check skips."""
    _ok("dlr_selftest_bounds", _load().dlr_selftest_bounds(_stream(stream)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_f32(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError("expected contiguous float32 CUDA tensors")


def _ok(fn: str, status: int):
    if status != DLR_OK:
        raise DLRError(fn, status)


def _params(p: Sequence[torch.Tensor]):
    log_re, log_im, W = p
    _check_f32(log_re, log_im, W)
    return log_re, log_im, W


def dlr_kernel(log_re, log_im, W, L: int, cast: str = "re", out=None, stream=None):
    """K[h, j] = Re (or Re*Im) of sum_n W[h,n] lambda[h,n]^j, j < L.  Returns [H, L]."""
    _check_f32(log_re, log_im, W)
    H, N = log_re.shape
    if out is None:
        out = torch.empty((H, L), dtype=torch.float32, device=log_re.device)
    _check_f32(out)
    _ok("dlr_kernel", _load().dlr_kernel(_ptr(log_re), _ptr(log_im), _ptr(W), H, N, L,
                                         CAST[cast], _ptr(out), _stream(stream)))
    return out


def dlr_conv_workspace_size(H: int, L: int, bidir: bool = False) -> int:
    """Bytes of device workspace dlr_conv / dlr_conv_spectrum need (twiddles and the H kernel
    spectra); 0 for unsupported sizes."""
    return int(_load().dlr_conv_workspace_size(H, L, 1 if bidir else 0))


def dlr_conv(u, K_fwd, K_bwd=None, out=None, workspace=None, stream=None):
    """y = causal (or, with K_bwd, bidirectional) Toeplitz product of u [B, H, L] with K."""
    _check_f32(u, K_fwd, K_bwd)
    B, H, L = u.shape
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    need = dlr_conv_workspace_size(H, L, K_bwd is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=u.device)
    _ok("dlr_conv", _load().dlr_conv(_ptr(u), _ptr(K_fwd), _ptr(K_bwd),
                                     1 if K_bwd is not None else 0, B, H, L, _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def dlr_conv_spectrum(K_fwd, K_bwd=None, workspace=None, stream=None):
    """Prepare the twiddle table and kernel spectra for dlr_conv_apply; returns the workspace."""
    _check_f32(K_fwd, K_bwd)
    H, L = K_fwd.shape
    need = dlr_conv_workspace_size(H, L, K_bwd is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=K_fwd.device)
    _ok("dlr_conv_spectrum", _load().dlr_conv_spectrum(
        _ptr(K_fwd), _ptr(K_bwd), 1 if K_bwd is not None else 0, H, L, _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return workspace


def dlr_conv_spectrum_direct(fwd, bwd=None, L=None, workspace=None, stream=None):
    """The spectra for dlr_conv_apply straight from the parameters (no kernel, no spectrum FFT):
    ``fwd`` / ``bwd`` = (log_re [H, N], log_im [H, N], W [H, N, 2]); returns the workspace."""
    lr, li, W = fwd
    _check_f32(lr, li, W)
    if bwd is not None:
        _check_f32(*bwd)
    H, N = lr.shape
    if L is None:
        raise ValueError("L (the sequence length) is required")
    need = dlr_conv_workspace_size(H, L, bwd is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=lr.device)
    b = bwd if bwd is not None else (None, None, None)
    _ok("dlr_conv_spectrum_direct", _load().dlr_conv_spectrum_direct(
        _ptr(lr), _ptr(li), _ptr(W), _ptr(b[0]), _ptr(b[1]), _ptr(b[2]),
        1 if bwd is not None else 0, H, N, L, _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return workspace


def dlr_conv_apply(u, workspace, out=None, stream=None):
    """y = FFT convolution of u [B, H, L] with the spectra prepared in ``workspace``."""
    _check_f32(u)
    B, H, L = u.shape
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    _ok("dlr_conv_apply", _load().dlr_conv_apply(_ptr(u), B, H, L, _ptr(out), _ptr(workspace),
                                                 workspace.numel(), _stream(stream)))
    return out


SCAN_ALGO = {"auto": 0, "fp32": 1, "tensor": 2}


def dlr_scan_workspace_size(B: int, H: int, N: int, L: int) -> int:
    """Bytes of workspace the tensor-core scan needs (0 when N > 64)."""
    return int(_load().dlr_scan_workspace_size(B, H, N, L))


def dlr_scan(u, fwd, bwd=None, out=None, stream=None, algo: str = "auto", workspace=None):
    """DLR recurrence (Re cast) as a chunked scan; ``fwd``/``bwd`` = (log_re, log_im, W).
    ``algo``: "fp32" (float32 FMA kernel), "tensor" (tensor-core contractions, N <= 64) or
    "auto" (tensor when N <= 64). The tensor path takes a uint8 device ``workspace`` of
    dlr_scan_workspace_size bytes (allocated here when not given)."""
    _check_f32(u)
    B, H, L = u.shape
    lr, li, W = _params(fwd)
    lr2 = li2 = W2 = None
    if bwd is not None:
        lr2, li2, W2 = _params(bwd)
    N = lr.shape[1]
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    need = dlr_scan_workspace_size(B, H, N, L) if algo != "fp32" else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=u.device)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _ok("dlr_scan", _load().dlr_scan_ex(_ptr(u), _ptr(lr), _ptr(li), _ptr(W), _ptr(lr2),
                                        _ptr(li2), _ptr(W2), 1 if bwd is not None else 0, B, H,
                                        N, L, _ptr(out), SCAN_ALGO[algo], _ptr(workspace),
                                        ws_bytes, _stream(stream)))
    return out


def dlr_scan_prepare(params, workspace=None, stream=None, B: int = 1, L: int = 64):
    """Channel tables of one parameter set (log_re, log_im, W) for dlr_scan_apply, into a uint8
    device ``workspace`` of dlr_scan_workspace_size bytes (allocated here when not given).
    Tensor-core path only (N <= 64)."""
    lr, li, W = _params(params)
    H, N = lr.shape
    need = dlr_scan_workspace_size(B, H, N, L)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=lr.device)
    _ok("dlr_scan_prepare", _load().dlr_scan_prepare(_ptr(lr), _ptr(li), _ptr(W), H, N,
                                                     _ptr(workspace), workspace.numel(),
                                                     _stream(stream)))
    return workspace


def dlr_scan_apply(u, workspace, N: int, out=None, reverse: bool = False, stream=None):
    """The tensor-core scan of u [B, H, L] with the tables dlr_scan_prepare left in
    ``workspace``: out = DLR(u), or (reverse) out += rev(DLR(rev(u)))."""
    _check_f32(u)
    B, H, L = u.shape
    if out is None:
        if reverse:
            raise ValueError("reverse=True adds into out: pass it")
        out = torch.empty_like(u)
    _check_f32(out)
    _ok("dlr_scan_apply", _load().dlr_scan_apply(_ptr(u), B, H, N, L, 1 if reverse else 0,
                                                 _ptr(out), _ptr(workspace), workspace.numel(),
                                                 _stream(stream)))
    return out


def dlr_scan_backward_params_workspace_size(B: int, H: int, N: int, L: int) -> int:
    """Bytes of device workspace dlr_scan_backward_params needs (0 for arguments out of range)."""
    return int(_load().dlr_scan_backward_params_workspace_size(B, H, N, L))


def dlr_scan_backward_params(u, g, params, workspace=None, stream=None):
    """Parameter gradients of the causal DLR layer (Re cast) for input u and output gradient g
    [B, H, L]: returns (d_log_re [H, N], d_log_im [H, N], dW [H, N, 2])."""
    _check_f32(u, g)
    lr, li, W = _params(params)
    B, H, L = u.shape
    N = lr.shape[1]
    if workspace is None:
        need = dlr_scan_backward_params_workspace_size(B, H, N, L)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=u.device)
    d_re = torch.empty_like(lr)
    d_im = torch.empty_like(li)
    dW = torch.empty_like(W)
    _ok("dlr_scan_backward_params",
        _load().dlr_scan_backward_params(_ptr(u), _ptr(g), _ptr(lr), _ptr(li), _ptr(W), B, H, N,
                                         L, _ptr(d_re), _ptr(d_im), _ptr(dW), _ptr(workspace),
                                         workspace.numel(), _stream(stream)))
    return d_re, d_im, dW


def dlr_layer_backward_workspace_size(B: int, H: int, N: int, L: int, bidir: bool = False,
                                      cast: str = "re") -> int:
    """Bytes of device workspace dlr_layer_backward needs (0 for arguments out of range)."""
    return int(_load().dlr_layer_backward_workspace_size(B, H, N, L, 1 if bidir else 0,
                                                         CAST[cast]))


def dlr_layer_backward(u, g, fwd, bwd=None, cast: str = "re", input_grad: bool = True,
                       workspace=None, stream=None):
    """Gradients of the DLR layer (causal, or bidirectional with the second parameter set
    `bwd`; Re or DLR-prod cast) for input u and output gradient g [B, H, L]. Returns
    (du or None, [(d_log_re, d_log_im, dW) per direction])."""
    _check_f32(u, g)
    lr, li, W = _params(fwd)
    B, H, L = u.shape
    N = lr.shape[1]
    if bwd is not None:
        lr2, li2, W2 = _params(bwd)
    else:
        lr2 = li2 = W2 = None
    if workspace is None:
        need = dlr_layer_backward_workspace_size(B, H, N, L, bwd is not None, cast)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=u.device)
    du = torch.empty_like(u) if input_grad else None
    outs = [(torch.empty_like(lr), torch.empty_like(li), torch.empty_like(W))]
    if bwd is not None:
        outs.append((torch.empty_like(lr2), torch.empty_like(li2), torch.empty_like(W2)))
    o2 = outs[1] if bwd is not None else (None, None, None)
    _ok("dlr_layer_backward",
        _load().dlr_layer_backward(_ptr(u), _ptr(g), _ptr(lr), _ptr(li), _ptr(W), _ptr(lr2),
                                   _ptr(li2), _ptr(W2), 1 if bwd is not None else 0, CAST[cast],
                                   B, H, N, L, _ptr(du), *[_ptr(t) for t in outs[0]],
                                   *[_ptr(t) for t in o2], _ptr(workspace), workspace.numel(),
                                   _stream(stream)))
    return du, outs


def dlr_scan_backward_input(g, params, workspace=None, out=None, stream=None):
    """Input gradient of the causal DLR layer for the output gradient g [B, H, L]: the layer
    run backwards in time on g with the same parameters (N <= 64). Returns du [B, H, L]."""
    _check_f32(g)
    lr, li, W = _params(params)
    B, H, L = g.shape
    N = lr.shape[1]
    if workspace is None:
        workspace = torch.empty(max(dlr_scan_workspace_size(B, H, N, L), 1), dtype=torch.uint8,
                                device=g.device)
    if out is None:
        out = torch.empty_like(g)
    _check_f32(out)
    _ok("dlr_scan_backward_input",
        _load().dlr_scan_backward_input(_ptr(g), _ptr(lr), _ptr(li), _ptr(W), B, H, N, L,
                                        _ptr(out), _ptr(workspace), workspace.numel(),
                                        _stream(stream)))
    return out


def dlr_step_workspace_size(H: int, N: int) -> int:
    """Bytes of device workspace dlr_step_prepare fills (24 per state); 0 when N > 256."""
    return int(_load().dlr_step_workspace_size(H, N))


def dlr_step_prepare(params, workspace=None, stream=None):
    """lambda (as a float pair) and W of one parameter set (log_re, log_im, W) for dlr_step,
    into a uint8 device ``workspace`` of dlr_step_workspace_size bytes (allocated here when not
    given)."""
    lr, li, W = _params(params)
    H, N = lr.shape
    need = dlr_step_workspace_size(H, N)
    if need == 0:
        raise ValueError(f"dlr_step: unsupported H={H}, N={N}")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=lr.device)
    _ok("dlr_step_prepare", _load().dlr_step_prepare(_ptr(lr), _ptr(li), _ptr(W), H, N,
                                                     _ptr(workspace), workspace.numel(),
                                                     _stream(stream)))
    return workspace


def dlr_step(u, workspace, state, out=None, stream=None):
    """Advance the causal DLR layer over u [B, H, T] from ``state`` [B, H, N, 2] (float32,
    updated in place: on return it holds the state after the last sample), with the tables of
    dlr_step_prepare in ``workspace``. Returns y [B, H, T]."""
    _check_f32(u, state)
    B, H, T = u.shape
    if state.dim() != 4 or tuple(state.shape[:2]) != (B, H) or state.shape[3] != 2:
        raise ValueError("state must be [B, H, N, 2]")
    N = state.shape[2]
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    _ok("dlr_step", _load().dlr_step(_ptr(u), B, H, N, T, _ptr(state), _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def dlr_scan_host_workspace_size(B: int, H: int, N: int, L: int) -> int:
    """Bytes of device workspace dlr_scan_host needs (device copies of u, y and the
    parameters, and the scan's channel tables)."""
    return int(_load().dlr_scan_host_workspace_size(B, H, N, L))


def dlr_scan_host(u, params, out, workspace, stream=None):
    """The causal DLR layer on host buffers: u, out [B, H, L] and the parameters are CPU float32
    tensors (pinned for overlap); ``workspace`` is a uint8 device tensor of
    dlr_scan_host_workspace_size bytes. Enqueued on ``stream``; synchronise it before reading
    ``out``."""
    lr, li, W = params
    for t in (u, out, lr, li, W):
        if t.device.type != "cpu" or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("dlr_scan_host takes contiguous float32 host tensors")
    B, H, L = u.shape
    N = lr.shape[1]
    if tuple(out.shape) != (B, H, L):
        raise ValueError("out must have the shape of u")
    _ok("dlr_scan_host", _load().dlr_scan_host(_ptr(u), _ptr(lr), _ptr(li), _ptr(W), B, H, N, L,
                                               _ptr(out), _ptr(workspace), workspace.numel(),
                                               _stream(stream)))
    return out


def s5_workspace_size(B: int, L: int, H: int, P: int, prec: str = "fp32") -> int:
    """Bytes of device workspace s5_layer needs at this size and precision tier."""
    return int(_load().s5_workspace_size(B, L, H, P, PREC[prec]))


def s5_layer(u, lam, log_delta, Bt, Ct, D, prec: str = "fp32", out=None, workspace=None,
             stream=None):
    """S5 SSM outputs for u [B, L, H]; parameters as in include/dlr.h. ``prec``: "fp32" (float32
    results: projections as three tf32 tensor-core products, float32 scan) or "bf16" (bf16
    projection operands and intermediates, float32 accumulation and scan)."""
    _check_f32(u, lam, log_delta, Bt, Ct, D)
    B, L, H = u.shape
    P = lam.shape[0]
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    need = s5_workspace_size(B, L, H, P, prec)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=u.device)
    _ok("s5_layer", _load().s5_layer(_ptr(u), _ptr(lam), _ptr(log_delta), _ptr(Bt), _ptr(Ct),
                                     _ptr(D), B, L, H, P, PREC[prec], _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


DISC = {"zoh": 0, "bilinear": 1}
REPARAM = {"exp": 0, "softplus": 1, "best": 2}


def s5_layer_ex(u, lam, log_delta, Bt, Ct, D, prec: str = "fp32", disc: str = "zoh",
                out=None, workspace=None, stream=None):
    """s5_layer with the discretisation chosen: 'zoh' or 'bilinear'."""
    _check_f32(u, lam, log_delta, Bt, Ct, D)
    B, L, H = u.shape
    P = lam.shape[0]
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    need = s5_workspace_size(B, L, H, P, prec)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=u.device)
    _ok("s5_layer_ex", _load().s5_layer_ex(_ptr(u), _ptr(lam), _ptr(log_delta), _ptr(Bt),
                                           _ptr(Ct), _ptr(D), B, L, H, P, PREC[prec],
                                           DISC[disc], _ptr(out), _ptr(workspace),
                                           workspace.numel(), _stream(stream)))
    return out


def s5_layer_tv(u, dt, lam, log_delta, Bt, Ct, D, out=None, workspace=None, stream=None):
    """S5 with per-step gaps dt [B, L] (irregular sampling); float32 tier."""
    _check_f32(u, dt, lam, log_delta, Bt, Ct, D)
    B, L, H = u.shape
    P = lam.shape[0]
    if out is None:
        out = torch.empty_like(u)
    _check_f32(out)
    need = _load().s5_layer_tv_workspace_size(B, L, H, P)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=u.device)
    _ok("s5_layer_tv", _load().s5_layer_tv(_ptr(u), _ptr(dt), _ptr(lam), _ptr(log_delta),
                                           _ptr(Bt), _ptr(Ct), _ptr(D), B, L, H, P, _ptr(out),
                                           _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def dlr_params_from_dss_exp(Lam, log_delta, W, stream=None):
    """DSS_exp parameters (Lam [H, N, 2], log_delta [H], W [H, N, 2]) as the DLR's
    (log_re, log_im, W')."""
    _check_f32(Lam, log_delta, W)
    H, N = Lam.shape[0], Lam.shape[1]
    lr = torch.empty((H, N), dtype=torch.float32, device=Lam.device)
    li = torch.empty_like(lr)
    Wo = torch.empty_like(W)
    _ok("dlr_params_from_dss_exp",
        _load().dlr_params_from_dss_exp(_ptr(Lam), _ptr(log_delta), _ptr(W), H, N, _ptr(lr),
                                        _ptr(li), _ptr(Wo), _stream(stream)))
    return lr, li, Wo


def dlr_log_re_from_reparam(w, kind: str, a: float = 1.0, b: float = 1.0, stream=None):
    """(log Lambda)_re = sqrt(f(w)) for the decay-rate maps 'exp', 'softplus', 'best'."""
    _check_f32(w)
    out = torch.empty_like(w)
    _ok("dlr_log_re_from_reparam",
        _load().dlr_log_re_from_reparam(_ptr(w), w.numel(), REPARAM[kind], float(a), float(b),
                                        _ptr(out), _stream(stream)))
    return out


def selftest_timeout(limit_ms: int = 50, stream=None) -> None:
    """Launch the bounded-wait self-test (see include/dlr.h); read the result with
    device_status()."""
    _ok("dlr_selftest_timeout", _load().dlr_selftest_timeout(limit_ms, _stream(stream)))


def device_status(stream=None) -> int:
    """Synchronise and return (then clear) the library's device status word."""
    return int(_load().dlr_get_device_status(_stream(stream)))


def dlr_layer(u, fwd, bwd=None, cast: str = "re", path: str = "fft", workspace=None,
              stream=None, out=None):
    """The whole DLR layer u -> y: kernel generation + FFT convolution (path='fft') or the
    chunked scan (path='scan', Re cast only)."""
    L = u.shape[-1]
    if path == "scan":
        if cast != "re":
            raise ValueError("the scan path exists only for the Re cast")
        return dlr_scan(u, fwd, bwd, out=out, stream=stream, workspace=workspace)
    K1 = dlr_kernel(*fwd, L, cast, stream=stream)
    K2 = dlr_kernel(*bwd, L, cast, stream=stream) if bwd is not None else None
    return dlr_conv(u, K1, K2, out=out, workspace=workspace, stream=stream)
