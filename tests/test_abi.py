"""C-ABI checks that need no GPU: libdlr.so builds, loads, exports every function declared in
include/dlr.h, and rejects invalid arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from state_space_sequence_gb300 import build as dlr_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dlr.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b([a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def lib():
    path = dlr_build.build()
    lib = ctypes.CDLL(path)
    return lib


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["dlr_kernel", "dlr_conv", "dlr_conv_workspace_size", "dlr_scan", "s5_layer",
                 "s5_workspace_size", "dlr_get_device_status", "dlr_status_string",
                 "dlr_abi_version", "dlr_step_prepare", "dlr_step", "dlr_step_workspace_size",
                 "dlr_conv_spectrum_direct", "dlr_scan_backward_params", "s5_layer_ex",
                 "s5_layer_tv", "dlr_params_from_dss_exp", "dlr_log_re_from_reparam",
                 "dlr_bounds_checked", "dlr_bounds_site", "dlr_selftest_bounds"]:
        assert must in names, must


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libdlr.so does not export {name}"


def test_status_strings_and_version(lib):
    lib.dlr_status_string.restype = ctypes.c_char_p
    assert lib.dlr_status_string(0) == b"DLR_OK"
    assert lib.dlr_status_string(4) == b"DLR_ERR_TIMEOUT"
    assert lib.dlr_status_string(6) == b"DLR_ERR_BOUNDS"
    assert lib.dlr_abi_version() == 12


def test_normal_build_has_no_bounds_checks(lib):
    """The normal library reports itself unchecked and refuses the bounds self-test without
    launching anything (its guards compile to nothing, so the planted read must not run)."""
    assert lib.dlr_bounds_checked() == 0
    lib.dlr_selftest_bounds.argtypes = [ctypes.c_void_p]
    assert lib.dlr_selftest_bounds(None) == 2  # DLR_ERR_UNSUPPORTED


def test_host_validation_rejects_bad_arguments(lib):
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.dlr_kernel.argtypes = [P, P, P, i64, i64, i64, ctypes.c_int, P, P]
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    # non-positive sizes
    assert lib.dlr_kernel(fake, fake, fake, 0, 4, 8, 0, fake, None) == 1
    assert lib.dlr_kernel(fake, fake, fake, 2, 4, -1, 0, fake, None) == 1
    # NULL and misaligned pointers
    assert lib.dlr_kernel(None, fake, fake, 2, 4, 8, 0, fake, None) == 1
    assert lib.dlr_kernel(ctypes.c_void_p(0x1004), fake, fake, 2, 4, 8, 0, fake, None) == 1
    # bad cast enum
    assert lib.dlr_kernel(fake, fake, fake, 2, 4, 8, 7, fake, None) == 1
    sz = ctypes.c_size_t
    lib.dlr_scan.argtypes = [P] * 7 + [ctypes.c_int, i64, i64, i64, i64, P, P, sz, P]
    # N above the scan's limit -> unsupported
    assert lib.dlr_scan(fake, fake, fake, fake, None, None, None, 0, 1, 1, 129, 8,
                        ctypes.c_void_p(0x9000), None, 0, None) == 2
    # bidirectional without second parameter set
    assert lib.dlr_scan(fake, fake, fake, fake, None, None, None, 1, 1, 1, 4, 8,
                        ctypes.c_void_p(0x9000), None, 0, None) == 1
    # overlapping u and y
    assert lib.dlr_scan(fake, fake, fake, fake, None, None, None, 0, 1, 1, 4, 64,
                        ctypes.c_void_p(0x1010), None, 0, None) == 1
    # tensor-core path (N <= 64) without its workspace
    assert lib.dlr_scan(fake, fake, fake, fake, None, None, None, 0, 1, 1, 4, 64,
                        ctypes.c_void_p(0x9000), None, 0, None) == 5
    lib.dlr_scan_ex.argtypes = [P] * 7 + [ctypes.c_int, i64, i64, i64, i64, P, ctypes.c_int, P,
                                          sz, P]
    # tensor-core path forced above 64 states -> unsupported; unknown algorithm -> invalid
    assert lib.dlr_scan_ex(fake, fake, fake, fake, None, None, None, 0, 1, 1, 65, 64,
                           ctypes.c_void_p(0x9000), 2, fake, 1 << 30, None) == 2
    assert lib.dlr_scan_ex(fake, fake, fake, fake, None, None, None, 0, 1, 1, 4, 64,
                           ctypes.c_void_p(0x9000), 7, None, 0, None) == 1
    # the float32 kernel needs no workspace (validation passes up to the launch, which is not
    # reached here: N above 128 keeps the call on the host)
    assert lib.dlr_scan_ex(fake, fake, fake, fake, None, None, None, 0, 1, 1, 129, 64,
                           ctypes.c_void_p(0x9000), 1, None, 0, None) == 2
    lib.dlr_scan_prepare.argtypes = [P, P, P, i64, i64, P, sz, P]
    lib.dlr_scan_apply.argtypes = [P, i64, i64, i64, i64, ctypes.c_int, P, P, sz, P]
    # tables for N above 64 -> unsupported; missing workspace; unknown direction flag
    assert lib.dlr_scan_prepare(fake, fake, fake, 4, 65, fake, 1 << 30, None) == 2
    assert lib.dlr_scan_prepare(fake, fake, fake, 4, 64, None, 0, None) == 5
    assert lib.dlr_scan_apply(fake, 1, 1, 4, 64, 2, ctypes.c_void_p(0x9000), fake, 1 << 20,
                              None) == 1
    assert lib.dlr_scan_apply(fake, 1, 1, 4, 64, 0, ctypes.c_void_p(0x9000), None, 0,
                              None) == 5
    # host-buffer entry point: the workspace holds u, y, the parameters and the tables
    lib.dlr_scan_host_workspace_size.argtypes = [i64, i64, i64, i64]
    lib.dlr_scan_host_workspace_size.restype = sz
    lib.dlr_scan_host.argtypes = [P, P, P, P, i64, i64, i64, i64, P, P, sz, P]
    need = lib.dlr_scan_host_workspace_size(8, 256, 64, 4096)
    assert need >= 2 * 8 * 256 * 4096 * 4 + 256 * 83968
    assert lib.dlr_scan_host_workspace_size(0, 1, 1, 1) == 0
    y = ctypes.c_void_p(0x9000)
    assert lib.dlr_scan_host(fake, fake, fake, fake, 0, 1, 4, 64, y, fake, 1 << 30, None) == 1
    assert lib.dlr_scan_host(None, fake, fake, fake, 1, 1, 4, 64, y, fake, 1 << 30, None) == 1
    assert lib.dlr_scan_host(fake, fake, fake, fake, 1, 1, 65, 64, y, fake, 1 << 30, None) == 2
    assert lib.dlr_scan_host(fake, fake, fake, fake, 1, 1, 4, 64, y, None, 0, None) == 5
    assert lib.dlr_scan_host(fake, fake, fake, fake, 1, 1, 4, 64, y, fake, 16, None) == 5
    lib.dlr_conv.argtypes = [P, P, P, ctypes.c_int, i64, i64, i64, P, P, ctypes.c_size_t, P]
    # missing workspace
    assert lib.dlr_conv(fake, fake, None, 0, 1, 1, 16, ctypes.c_void_p(0x9000), None, 0,
                        None) == 5
    # causal call given a backward kernel
    assert lib.dlr_conv(fake, fake, fake, 0, 1, 1, 16, ctypes.c_void_p(0x9000), fake, 1 << 20,
                        None) == 1
    lib.s5_layer.argtypes = [P] * 6 + [i64] * 4 + [ctypes.c_int, P, P, ctypes.c_size_t, P]
    # H not a multiple of 32
    assert lib.s5_layer(fake, fake, fake, fake, fake, fake, 1, 16, 48, 32, 0,
                        ctypes.c_void_p(0x90000), fake, 1 << 30, None) == 2


def test_workspace_queries(lib):
    lib.dlr_conv_workspace_size.restype = ctypes.c_size_t
    lib.dlr_conv_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    # L = 4096 -> n = 4096: twiddle tables of n and 2n points + spectra H*(n+1) complex
    assert lib.dlr_conv_workspace_size(256, 4096, 0) == 4096 * 8 + 8192 * 8 + 256 * 4097 * 8
    assert lib.dlr_conv_workspace_size(0, 4096, 0) == 0
    lib.dlr_scan_workspace_size.restype = ctypes.c_size_t
    lib.dlr_scan_workspace_size.argtypes = [ctypes.c_int64] * 4
    # one table blob of 83968 bytes per channel for the tensor-core scan; none above 64 states
    assert lib.dlr_scan_workspace_size(8, 256, 64, 4096) == 256 * 83968
    assert lib.dlr_scan_workspace_size(8, 256, 65, 4096) == 0
    lib.s5_workspace_size.restype = ctypes.c_size_t
    lib.s5_workspace_size.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int]
    assert lib.s5_workspace_size(8, 16384, 512, 256, 0) >= 8 * 16384 * 512 * 4


def test_step_validation(lib):
    """dlr_step_prepare / dlr_step: sizes, limits, workspace and overlap are checked on the
    host before anything is launched."""
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.dlr_step_workspace_size.restype = sz
    lib.dlr_step_workspace_size.argtypes = [i64, i64]
    assert lib.dlr_step_workspace_size(256, 64) == 256 * 64 * 24
    assert lib.dlr_step_workspace_size(4, 257) == 0
    lib.dlr_step_prepare.argtypes = [P, P, P, i64, i64, P, sz, P]
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x100000)
    assert lib.dlr_step_prepare(fake, fake, fake, 0, 4, ws, 1 << 20, None) == 1
    assert lib.dlr_step_prepare(fake, fake, fake, 2, 300, ws, 1 << 20, None) == 2
    assert lib.dlr_step_prepare(fake, fake, fake, 2, 4, ws, 10, None) == 5
    lib.dlr_step.argtypes = [P, i64, i64, i64, i64, P, P, P, sz, P]
    u, x, y = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    # negative T, too many states, missing workspace
    assert lib.dlr_step(u, 1, 2, 4, -1, x, y, ws, 1 << 20, None) == 1
    assert lib.dlr_step(u, 1, 2, 300, 8, x, y, ws, 1 << 20, None) == 2
    assert lib.dlr_step(u, 1, 2, 4, 8, x, y, None, 0, None) == 5
    # T = 0 launches nothing and succeeds; u and y overlapping; x overlapping y
    assert lib.dlr_step(None, 1, 2, 4, 0, x, None, ws, 1 << 20, None) == 0
    assert lib.dlr_step(u, 1, 2, 4, 8, x, ctypes.c_void_p(0x10010), ws, 1 << 20, None) == 1
    assert lib.dlr_step(u, 1, 2, 4, 8, x, ctypes.c_void_p(0x20010), ws, 1 << 20, None) == 1


def test_backward_input_validation(lib):
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.dlr_scan_backward_input.argtypes = [P, P, P, P, i64, i64, i64, i64, P, P, sz, P]
    fake = ctypes.c_void_p(0x1000)
    g, du, ws = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x100000)
    assert lib.dlr_scan_backward_input(g, fake, fake, fake, 1, 2, 4, 0, du, ws, 1 << 20,
                                       None) == 1
    assert lib.dlr_scan_backward_input(g, fake, fake, fake, 1, 2, 65, 8, du, ws, 1 << 20,
                                       None) == 2
    assert lib.dlr_scan_backward_input(g, fake, fake, fake, 1, 2, 4, 8, du, None, 0, None) == 5
    assert lib.dlr_scan_backward_input(g, fake, fake, fake, 1, 2, 4, 8, ctypes.c_void_p(0x10010),
                                       ws, 1 << 20, None) == 1


def test_conv_and_s5_validation(lib):
    """dlr_conv_spectrum / dlr_conv_apply / dlr_conv_noalloc / s5_layer reject invalid sizes,
    enums, pointers, overlaps, limits and short workspaces on the host, before any launch."""
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    k, k2 = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000)
    # far apart, so that only the intended check fails
    u, y, ws = (ctypes.c_void_p(0x10000000), ctypes.c_void_p(0x20000000),
                ctypes.c_void_p(0x30000000))
    big = 1 << 40
    lib.dlr_conv_spectrum.argtypes = [P, P, i32, i64, i64, P, sz, P]
    assert lib.dlr_conv_spectrum(k, None, 0, 0, 64, ws, big, None) == 1       # H < 1
    assert lib.dlr_conv_spectrum(k, None, 5, 2, 64, ws, big, None) == 1       # bad direction
    assert lib.dlr_conv_spectrum(ctypes.c_void_p(0x1004), None, 0, 2, 64, ws, big, None) == 1
    assert lib.dlr_conv_spectrum(k, k2, 0, 2, 64, ws, big, None) == 1         # causal + K_bwd
    assert lib.dlr_conv_spectrum(k, None, 1, 2, 64, ws, big, None) == 1       # bidir, no K_bwd
    assert lib.dlr_conv_spectrum(k, None, 0, 2, 70000, ws, big, None) == 2    # L > 65536
    assert lib.dlr_conv_spectrum(k, None, 0, 2, 64, ws, 16, None) == 5        # short workspace
    lib.dlr_conv_apply.argtypes = [P, i64, i64, i64, P, P, sz, P]
    assert lib.dlr_conv_apply(u, 0, 2, 64, y, ws, big, None) == 1
    assert lib.dlr_conv_apply(u, 1, 2, 64, ctypes.c_void_p(0x10000100), ws, big, None) == 1
    assert lib.dlr_conv_apply(u, 1, 2, 70000, y, ws, big, None) == 2
    assert lib.dlr_conv_apply(u, 1, 2, 64, y, None, 0, None) == 5
    lib.dlr_conv_noalloc.argtypes = [P, P, P, i32, i64, i64, i64, P, P]
    assert lib.dlr_conv_noalloc(u, k, None, 0, 1, 2, 20000, y, None) == 2     # L > 16384
    far = ctypes.c_void_p(1 << 46)  # the 64 GB rows of this call overlap nothing
    assert lib.dlr_conv_noalloc(u, k, None, 0, 1, 1 << 20, 16384, far, None) == 5  # > scratch
    assert lib.dlr_conv_noalloc(u, k, k2, 0, 1, 2, 64, y, None) == 1
    lib.s5_layer.argtypes = [P] * 6 + [i64] * 4 + [i32, P, P, sz, P]
    p = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(5)]
    assert lib.s5_layer(u, *p, 1, 64, 32, 32, 7, y, ws, big, None) == 1       # bad precision
    assert lib.s5_layer(u, None, *p[1:], 1, 64, 32, 32, 0, y, ws, big, None) == 1
    assert lib.s5_layer(u, *p, 1, 64, 32, 48, 0, y, ws, big, None) == 2       # P % 32
    assert lib.s5_layer(u, *p, 1, 64, 32, 2048, 0, y, ws, big, None) == 2     # P > 1024
    assert lib.s5_layer(u, *p, 1, 64, 32, 32, 0, ctypes.c_void_p(0x10000010), ws, big, None) == 1
    assert lib.s5_layer(u, *p, 1, 64, 32, 32, 0, y, ws, 16, None) == 5        # short workspace


def test_direct_spectrum_validation(lib):
    """dlr_conv_spectrum_direct: sizes, direction and second parameter set, the 8-byte W
    alignment, limits and the workspace are checked on the host before any launch."""
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.dlr_conv_spectrum_direct.argtypes = [P] * 6 + [ctypes.c_int, i64, i64, i64, P, sz, P]
    lib.dlr_conv_workspace_size.argtypes = [i64, i64, ctypes.c_int]
    lib.dlr_conv_workspace_size.restype = sz
    f = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x8000)
    need = lib.dlr_conv_workspace_size(4, 100, 0)
    call = lib.dlr_conv_spectrum_direct
    assert call(f, f, f, None, None, None, 0, 0, 8, 100, ws, need, None) == 1   # H = 0
    assert call(f, f, f, None, None, None, 0, 4, 0, 100, ws, need, None) == 1   # N = 0
    assert call(None, f, f, None, None, None, 0, 4, 8, 100, ws, need, None) == 1
    assert call(f, f, ctypes.c_void_p(0x1004), None, None, None, 0, 4, 8, 100, ws, need,
                None) == 1                                                      # W misaligned
    assert call(f, f, f, None, None, None, 3, 4, 8, 100, ws, need, None) == 1   # direction
    assert call(f, f, f, None, None, None, 1, 4, 8, 100, ws, need, None) == 1   # no 2nd set
    assert call(f, f, f, f, f, f, 0, 4, 8, 100, ws, need, None) == 1           # extra set
    assert call(f, f, f, None, None, None, 0, 4, 257, 100, ws, need, None) == 2  # N > 256
    assert call(f, f, f, None, None, None, 0, 4, 8, 65537, ws, need, None) == 2  # L
    assert call(f, f, f, None, None, None, 0, 4, 8, 100, None, 0, None) == 5
    assert call(f, f, f, None, None, None, 0, 4, 8, 100, ws, need - 1, None) == 5


def test_backward_params_validation(lib):
    """dlr_scan_backward_params: sizes, pointers and alignment, outputs that overlap the
    parameters or each other, limits and the workspace are checked on the host."""
    P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.dlr_scan_backward_params.argtypes = [P] * 5 + [i64] * 4 + [P] * 4 + [sz, P]
    lib.dlr_scan_backward_params_workspace_size.argtypes = [i64] * 4
    lib.dlr_scan_backward_params_workspace_size.restype = sz
    wsz = lib.dlr_scan_backward_params_workspace_size
    # correlation route (N >= 16, L <= 8192): the M-point twiddle table (M = 2^ceil(log2(2L-1)))
    # and c [H, L]; otherwise 16 bytes per (b, h, n); each part rounded up to 256 bytes
    assert wsz(8, 256, 64, 4096) == 8 * 8192 + 4 * 256 * 4096
    assert wsz(2, 3, 16, 5) == 256 + 256                         # M = 16; c of 60 bytes
    assert wsz(8, 256, 8, 4096) == 16 * 8 * 256 * 8              # few states
    # rows longer than 8192: two dlr_conv workspaces for the B * H rows, one for the H
    # channels, the impulse rows and c; rows longer than 65536: the recurrences
    lib.dlr_conv_workspace_size.argtypes = [i64, i64, ctypes.c_int]
    lib.dlr_conv_workspace_size.restype = sz
    r256 = lambda b: (b + 255) // 256 * 256
    cw = lib.dlr_conv_workspace_size
    assert wsz(8, 256, 64, 8193) == (2 * r256(cw(8 * 256, 8193, 0)) + r256(cw(256, 8193, 0)) +
                                     2 * r256(4 * 256 * 8193))
    assert wsz(8, 256, 64, 65537) == 16 * 8 * 256 * 64
    assert wsz(0, 1, 1, 1) == 0
    assert wsz(1, 1, 1, 0) == 0
    assert wsz(1, 1, 1, 1 << 24) == 0
    u, g = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    lr, li, W = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x310000), ctypes.c_void_p(0x320000)
    dr, di, dW = ctypes.c_void_p(0x400000), ctypes.c_void_p(0x410000), ctypes.c_void_p(0x420000)
    ws = ctypes.c_void_p(0x500000)
    need = wsz(2, 3, 4, 10)
    call = lib.dlr_scan_backward_params
    assert call(u, g, lr, li, W, 0, 3, 4, 10, dr, di, dW, ws, need, None) == 1
    assert call(None, g, lr, li, W, 2, 3, 4, 10, dr, di, dW, ws, need, None) == 1
    assert call(u, g, lr, li, W, 2, 3, 4, 10, dr, di, ctypes.c_void_p(0x420004), ws, need,
                None) == 1                                                   # dW misaligned
    assert call(u, g, lr, li, W, 2, 3, 4, 10, lr, di, dW, ws, need, None) == 1   # overlap
    assert call(u, g, lr, li, W, 2, 3, 4, 10, dr, dr, dW, ws, need, None) == 1   # overlap
    assert call(u, g, lr, li, W, 2, 3, 4, 1 << 24, dr, di, dW, ws, need, None) == 2
    assert call(u, g, lr, li, W, 2, 3, 4, 10, dr, di, dW, None, 0, None) == 5
    assert call(u, g, lr, li, W, 2, 3, 4, 10, dr, di, dW, ws, need - 16, None) == 5


def test_layer_backward_validation(lib):
    """dlr_layer_backward: directions and casts, the second parameter set given exactly when
    bidirectional, output alignment and overlaps, the DLR-prod cast's row limit and the
    workspace are checked on the host; the workspace size is the gradients' part, two kernel
    buffers and the convolution workspace."""
    P, i64, sz, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    lib.dlr_layer_backward_workspace_size.argtypes = [i64] * 4 + [i32, i32]
    lib.dlr_layer_backward_workspace_size.restype = sz
    lib.dlr_conv_workspace_size.argtypes = [i64, i64, i32]
    lib.dlr_conv_workspace_size.restype = sz
    lib.dlr_layer_backward.argtypes = [P] * 8 + [i32, i32] + [i64] * 4 + [P] * 8 + [sz, P]
    wsz = lib.dlr_layer_backward_workspace_size
    conv = lib.dlr_conv_workspace_size(256, 4096, 0)
    # causal Re, correlation route: table 64 KB + c 4 MB; kernels 2 x 4 MB; convolution
    assert wsz(8, 256, 64, 4096, 0, 0) == 8 * 8192 + 4 * 256 * 4096 + 2 * 4 * 256 * 4096 + conv
    # bidirectional DLR-prod: + c2 4 MB + two complex kernels of 8 MB
    assert wsz(8, 256, 64, 4096, 1, 1) == (8 * 8192 + 2 * 4 * 256 * 4096 + 2 * 8 * 256 * 4096 +
                                          2 * 4 * 256 * 4096 + conv)
    assert wsz(8, 256, 64, 65537, 0, 1) == 0
    assert wsz(1, 1, 1, 65537, 0, 0) == 0
    assert wsz(1, 1, 1, 8, 2, 0) == 0
    assert wsz(1, 1, 1, 8, 0, 2) == 0
    u, g = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    a = [ctypes.c_void_p(0x300000 + 0x10000 * i) for i in range(6)]   # two parameter sets
    o = [ctypes.c_void_p(0x400000 + 0x10000 * i) for i in range(6)]   # their gradients
    du, ws = ctypes.c_void_p(0x500000), ctypes.c_void_p(0x1000000)
    call = lib.dlr_layer_backward
    need = wsz(2, 3, 20, 100, 1, 0)
    assert need > 0
    ok = (u, g, *a, 1, 0, 2, 3, 20, 100, du, *o, ws, need, None)
    assert call(*ok[:8], 2, *ok[9:]) == 1                                      # direction
    assert call(*ok[:9], 2, *ok[10:]) == 1                                     # cast
    assert call(u, g, *a[:3], None, None, None, *ok[8:]) == 1                  # bidir: set 2
    assert call(u, g, *a[:3], None, None, None, 0, 0, 2, 3, 20, 100, du, *o[:3], *o[:3], ws,
                need, None) == 1                                               # causal: no set 2
    assert call(*ok[:14], ctypes.c_void_p(0x500004), *ok[15:]) == 1           # du alignment
    assert call(*ok[:15], a[0], *ok[16:]) == 1                                 # output on input
    assert call(*ok[:15], o[0], o[0], *ok[17:]) == 1                          # outputs overlap
    assert call(*ok[:14], u, *ok[15:]) == 1                                    # du on u
    assert call(*ok[:9], 1, 2, 3, 20, 65537, *ok[14:]) == 2                    # rows too long
    assert call(*ok[:-3], None, 0, None) == 5
    assert call(*ok[:-2], need - 16, None) == 5


def test_variant_entry_points_validation(lib):
    """s5_layer_ex, s5_layer_tv, dlr_params_from_dss_exp and dlr_log_re_from_reparam check their
    arguments on the host before any launch."""
    P, i64, sz, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int, \
        ctypes.c_float
    f = ctypes.c_void_p(0x100000)
    y = ctypes.c_void_p(0x900000)
    ws = ctypes.c_void_p(0xa00000)
    lib.s5_layer_ex.argtypes = [P] * 6 + [i64] * 4 + [i32, i32, P, P, sz, P]
    assert lib.s5_layer_ex(f, f, f, f, f, f, 1, 8, 32, 32, 0, 2, y, ws, 1 << 30, None) == 1
    assert lib.s5_layer_ex(f, f, f, f, f, f, 1, 8, 33, 32, 0, 1, y, ws, 1 << 30, None) == 2
    assert lib.s5_layer_ex(f, f, f, f, f, f, 1, 8, 32, 32, 0, 1, y, None, 0, None) == 5
    lib.s5_layer_tv.argtypes = [P] * 7 + [i64] * 4 + [P, P, sz, P]
    lib.s5_layer_tv_workspace_size.argtypes = [i64] * 4
    lib.s5_layer_tv_workspace_size.restype = sz
    assert lib.s5_layer_tv_workspace_size(0, 1, 32, 32) == 0
    assert lib.s5_layer_tv(f, None, f, f, f, f, f, 1, 8, 32, 32, y, ws, 1 << 30, None) == 1
    assert lib.s5_layer_tv(f, y, f, f, f, f, f, 1, 8, 32, 32, y, ws, 1 << 30, None) == 1
    assert lib.s5_layer_tv(f, f, f, f, f, f, f, 1, 8, 32, 48, y, ws, 1 << 30, None) == 2
    assert lib.s5_layer_tv(f, f, f, f, f, f, f, 1, 8, 32, 32, y, ws, 16, None) == 5
    lib.dlr_params_from_dss_exp.argtypes = [P, P, P, i64, i64, P, P, P, P]
    a, b, c = ctypes.c_void_p(0x200000), ctypes.c_void_p(0x210000), ctypes.c_void_p(0x220000)
    o1, o2, o3 = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x310000), ctypes.c_void_p(0x320000)
    assert lib.dlr_params_from_dss_exp(a, b, c, 0, 4, o1, o2, o3, None) == 1
    assert lib.dlr_params_from_dss_exp(ctypes.c_void_p(0x200004), b, c, 2, 4, o1, o2, o3,
                                       None) == 1
    assert lib.dlr_params_from_dss_exp(a, b, c, 2, 4, a, o2, o3, None) == 1    # overlap
    lib.dlr_log_re_from_reparam.argtypes = [P, i64, i32, f32, f32, P, P]
    assert lib.dlr_log_re_from_reparam(a, 10, 3, 1.0, 1.0, o1, None) == 1      # kind
    assert lib.dlr_log_re_from_reparam(a, 10, 2, 1.0, 0.0, o1, None) == 1      # b <= 0
    assert lib.dlr_log_re_from_reparam(a, 10, 2, -1.0, 1.0, o1, None) == 1     # a < 0
    assert lib.dlr_log_re_from_reparam(a, 0, 0, 1.0, 1.0, o1, None) == 1
