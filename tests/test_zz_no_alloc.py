"""dlr_conv_noalloc: the allocation-free variant of dlr_conv, for callers whose device memory
is owned by a host application's fixed plan or who cannot afford a cudaMalloc on their path.

Called through the C ABI (ctypes) and compared with dlr_conv on two calls in a row (the two
calls share the library's fixed scratch array, so the second must not see the first's
leftovers). This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_gb300 import dlr

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _lib():
    lib = dlr._load()
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.dlr_conv_noalloc.argtypes = [P, P, P, ctypes.c_int, i64, i64, i64, P, P]
    lib.dlr_conv_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(u, K1, K2):
    B, H, L = u.shape
    y = torch.empty_like(u)
    st = _lib().dlr_conv_noalloc(
        ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(K1.data_ptr()),
        ctypes.c_void_p(K2.data_ptr()) if K2 is not None else None, 1 if K2 is not None else 0,
        B, H, L, ctypes.c_void_p(y.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, dlr._load().dlr_status_string(st)
    return y


def _case(seed, B, H, L, bidir):
    rng = np.random.default_rng(seed)
    u = torch.from_numpy(rng.standard_normal((B, H, L)).astype(np.float32)).cuda()
    K1 = torch.from_numpy((rng.standard_normal((H, L)) * np.exp(-np.arange(L) / 400.0))
                          .astype(np.float32)).cuda()
    K2 = (torch.from_numpy((rng.standard_normal((H, L)) * np.exp(-np.arange(L) / 700.0))
                           .astype(np.float32)).cuda() if bidir else None)
    return u, K1, K2


def test_noalloc_matches_dlr_conv_on_two_calls_in_a_row():
    cases = [(1, 4, 256, 4096, True), (2, 3, 16, 1000, False)]
    for seed, B, H, L, bidir in cases:
        u, K1, K2 = _case(seed, B, H, L, bidir)
        y_ref = dlr.dlr_conv(u, K1, K2)
        y = _noalloc(u, K1, K2)
        torch.cuda.synchronize()
        assert oracle.rel_l2(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL
    assert dlr.device_status() == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    u, K1, _ = _case(3, 1, 512, 4096, False)   # needs ~16.8 MB of spectra > 16 MiB
    y = torch.empty_like(u)
    st = _lib().dlr_conv_noalloc(ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(K1.data_ptr()),
                                 None, 0, 1, 512, 4096, ctypes.c_void_p(y.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == dlr.DLR_ERR_WORKSPACE
