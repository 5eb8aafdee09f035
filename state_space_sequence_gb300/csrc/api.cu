// api.cu -- the extern "C" entry points declared in include/dlr.h: argument validation,
// workspace carving and kernel dispatch on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "dlr.h"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 1;
cudaError_t launch_dlr_kernel(const float* log_re, const float* log_im, const float* W, int H,
                              int N, int L, bool re_im, float* K, int* status, cudaStream_t s);
int conv_log2_size(int64_t L);
size_t conv_workspace_bytes(int64_t H, int64_t L);
cudaError_t launch_dlr_conv_spectrum(const float* K1, const float* K2, int H, int L, void* ws,
                                     cudaStream_t s);
cudaError_t launch_dlr_conv_apply(const float* u, int B, int H, int L, float* y, const void* ws,
                                  cudaStream_t s);
cudaError_t launch_dlr_scan(const float* u, const float* lr, const float* li, const float* W,
                            const float* lr2, const float* li2, const float* W2, bool bidir,
                            int B, int H, int N, int L, float* y, cudaStream_t s);
size_t scan_tc_workspace_bytes(int64_t H);
cudaError_t launch_scan_tc_tables(const float* lr, const float* li, const float* W, int H, int N,
                                  void* ws, cudaStream_t s);
cudaError_t launch_scan_tc_apply(const float* u, int B, int H, int L, bool reverse, float* y,
                                 const void* ws, int* status, cudaStream_t s, bool after_tables);
cudaError_t launch_dlr_scan_tc(const float* u, const float* lr, const float* li, const float* W,
                               const float* lr2, const float* li2, const float* W2, bool bidir,
                               int B, int H, int N, int L, float* y, void* ws, int* status,
                               cudaStream_t s);
size_t s5_workspace_bytes(int64_t B, int64_t L, int64_t H, int64_t P, bool bf16);
cudaError_t launch_s5(const float* u, const float* lambda, const float* log_delta,
                      const float* Bt, const float* Ct, const float* D, int B, int L, int H, int P,
                      bool bf16, bool bilinear, float* y, void* ws, int* status,
                      cudaStream_t s);
cudaError_t launch_dss_exp_map(const float* Lam, const float* log_delta, const float* W,
                               int64_t H, int64_t N, float* log_re, float* log_im, float* Wout,
                               int* status, cudaStream_t s);
cudaError_t launch_reparam_map(const float* w, int64_t count, int kind, float a, float b,
                               float* log_re, cudaStream_t s);
cudaError_t launch_s5_tv(const float* u, const float* dt, const float* lambda,
                         const float* log_delta, const float* Bt, const float* Ct,
                         const float* D, int B, int L, int H, int P, float* y, void* ws,
                         int* status, cudaStream_t s);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s);
cudaError_t launch_selftest_bounds(cudaStream_t s);
size_t grad_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t L);
size_t grads_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t L, bool bidir, bool prod);
cudaError_t launch_dlr_grads(const float* u, const float* g, const float* lr1, const float* li1,
                             const float* W1, const float* lr2, const float* li2,
                             const float* W2, int B, int H, int N, int L, bool prod,
                             float* dr1, float* di1, float* dW1, float* dr2, float* di2,
                             float* dW2, void* ws, int* status, cudaStream_t s, float* kap1,
                             float* kap2);
cudaError_t launch_dlr_grad_params(const float* u, const float* g, const float* log_re,
                                   const float* log_im, const float* W, int B, int H, int N,
                                   int L, float* d_log_re, float* d_log_im, float* dW, void* ws,
                                   int* status, cudaStream_t s);
cudaError_t launch_spectrum_direct(const float* lr1, const float* li1, const float* W1,
                                   const float* lr2, const float* li2, const float* W2, int H,
                                   int N, int L, void* ws, cudaStream_t s);
size_t step_workspace_bytes(int64_t H, int64_t N);
cudaError_t launch_step_tables(const float* lr, const float* li, const float* W, int64_t H,
                               int64_t N, void* ws, cudaStream_t s);
cudaError_t launch_step(const float* u, int64_t B, int64_t H, int64_t N, int64_t T,
                        const void* ws, float* x, float* y, cudaStream_t s);
}  // namespace dlr

// The library's device status word (one per device that loads the library), and the first
// failing site of the bounds-checked build.
__device__ int g_dlr_device_status = 0;
__device__ int g_dlr_bounds_site = 0;

namespace {
// The last CUDA error a call of this thread turned into DLR_ERR_CUDA (for diagnostics).
thread_local const char* t_last_cuda_error_msg = "no error";
}  // namespace

namespace dlr {
// Every entry point maps a CUDA error through here, so dlr_last_cuda_error() names it.
dlr_status status_from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DLR_OK;
  t_last_cuda_error_msg = cudaGetErrorString(e);
  return DLR_ERR_CUDA;
}
}  // namespace dlr

namespace {

constexpr int64_t kMaxL = (int64_t(1) << 24) - 1;
constexpr int64_t kMaxGrid = 2147483647;

// Device address of the status word on the current device (kernels with bounded waits write it).
int* status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dlr_device_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dlr_status from_cuda(cudaError_t e) { return dlr::status_from_cuda(e); }

// Three non-blocking streams per device for the host-buffer entry point: copies in, compute,
// copies out. Created on first use and kept for the life of the process.
constexpr int kMaxDevices = 64;
cudaStream_t g_pipe[kMaxDevices][3];
std::once_flag g_pipe_once[kMaxDevices];
cudaError_t g_pipe_err[kMaxDevices];

cudaError_t pipe_streams(cudaStream_t (&st)[3]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_pipe_once[dev], [dev] {
    g_pipe_err[dev] = cudaSuccess;
    for (int i = 0; i < 3 && g_pipe_err[dev] == cudaSuccess; ++i)
      g_pipe_err[dev] = cudaStreamCreateWithFlags(&g_pipe[dev][i], cudaStreamNonBlocking);
  });
  if (g_pipe_err[dev] != cudaSuccess) return g_pipe_err[dev];
  for (int i = 0; i < 3; ++i) st[i] = g_pipe[dev][i];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
  uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

dlr_status check_params(const float* log_re, const float* log_im, const float* W) {
  if (!log_re || !log_im || !W) return DLR_ERR_INVALID_ARG;
  if (!aligned16(log_re) || !aligned16(log_im) || !aligned16(W)) return DLR_ERR_INVALID_ARG;
  return DLR_OK;
}

}  // namespace

extern "C" {

int dlr_abi_version(void) { return 12; }

const char* dlr_last_cuda_error(void) { return t_last_cuda_error_msg; }

const char* dlr_status_string(dlr_status s) {
  switch (s) {
    case DLR_OK: return "DLR_OK";
    case DLR_ERR_INVALID_ARG: return "DLR_ERR_INVALID_ARG";
    case DLR_ERR_UNSUPPORTED: return "DLR_ERR_UNSUPPORTED";
    case DLR_ERR_CUDA: return "DLR_ERR_CUDA";
    case DLR_ERR_TIMEOUT: return "DLR_ERR_TIMEOUT";
    case DLR_ERR_WORKSPACE: return "DLR_ERR_WORKSPACE";
    case DLR_ERR_BOUNDS: return "DLR_ERR_BOUNDS";
  }
  return "DLR_ERR_UNKNOWN";
}

dlr_status dlr_kernel(const float* log_re, const float* log_im, const float* W, int64_t H,
                      int64_t N, int64_t L, dlr_cast cast, float* K, dlr_stream_t stream) {
  if (H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (cast != DLR_CAST_RE && cast != DLR_CAST_RE_IM) return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  if (!K || !aligned16(K)) return DLR_ERR_INVALID_ARG;
  if (L > kMaxL || H > 65535 || N > (int64_t(1) << 24)) return DLR_ERR_UNSUPPORTED;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_dlr_kernel(log_re, log_im, W, (int)H, (int)N, (int)L,
                                          cast == DLR_CAST_RE_IM, K, status,
                                          (cudaStream_t)stream));
}

size_t dlr_conv_workspace_size(int64_t H, int64_t L, dlr_dir dir) {
  (void)dir;
  if (H < 1 || L < 1 || L > 65536) return 0;
  return dlr::conv_workspace_bytes(H, L);
}

static dlr_status check_conv_ws(int64_t H, int64_t L, const void* ws, size_t bytes) {
  if (!ws || !aligned16(ws) || bytes < dlr::conv_workspace_bytes(H, L)) return DLR_ERR_WORKSPACE;
  return DLR_OK;
}

dlr_status dlr_conv_spectrum(const float* K_fwd, const float* K_bwd, dlr_dir dir, int64_t H,
                             int64_t L, void* workspace, size_t workspace_bytes,
                             dlr_stream_t stream) {
  if (H < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return DLR_ERR_INVALID_ARG;
  if (!K_fwd || !aligned16(K_fwd)) return DLR_ERR_INVALID_ARG;
  if (dir == DLR_BIDIR && (!K_bwd || !aligned16(K_bwd))) return DLR_ERR_INVALID_ARG;
  if (dir == DLR_CAUSAL && K_bwd) return DLR_ERR_INVALID_ARG;
  if (L > 65536 || H > kMaxGrid / 8) return DLR_ERR_UNSUPPORTED;
  dlr_status st = check_conv_ws(H, L, workspace, workspace_bytes);
  if (st != DLR_OK) return st;
  return from_cuda(dlr::launch_dlr_conv_spectrum(K_fwd, dir == DLR_BIDIR ? K_bwd : nullptr,
                                                 (int)H, (int)L, workspace,
                                                 (cudaStream_t)stream));
}

dlr_status dlr_conv_spectrum_direct(const float* log_re, const float* log_im, const float* W,
                                    const float* log_re2, const float* log_im2,
                                    const float* W2, dlr_dir dir, int64_t H, int64_t N,
                                    int64_t L, void* workspace, size_t workspace_bytes,
                                    dlr_stream_t stream) {
  if (H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return DLR_ERR_INVALID_ARG;
  auto al8 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; };
  if (!log_re || !log_im || !W || !al8(W)) return DLR_ERR_INVALID_ARG;
  const bool two = dir == DLR_BIDIR;
  if (two && (!log_re2 || !log_im2 || !W2 || !al8(W2))) return DLR_ERR_INVALID_ARG;
  if (!two && (log_re2 || log_im2 || W2)) return DLR_ERR_INVALID_ARG;
  if (N > 256 || L > 65536 || H > 65535) return DLR_ERR_UNSUPPORTED;
  dlr_status st = check_conv_ws(H, L, workspace, workspace_bytes);
  if (st != DLR_OK) return st;
  return from_cuda(dlr::launch_spectrum_direct(log_re, log_im, W, two ? log_re2 : nullptr,
                                               two ? log_im2 : nullptr, two ? W2 : nullptr,
                                               (int)H, (int)N, (int)L, workspace,
                                               (cudaStream_t)stream));
}

dlr_status dlr_conv_apply(const float* u, int64_t B, int64_t H, int64_t L, float* y,
                          const void* workspace, size_t workspace_bytes, dlr_stream_t stream) {
  if (B < 1 || H < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (!u || !y || !aligned16(u) || !aligned16(y)) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  if (ranges_overlap(u, bytes, y, bytes)) return DLR_ERR_INVALID_ARG;
  if (L > 65536 || B * H > kMaxGrid / 8) return DLR_ERR_UNSUPPORTED;
  dlr_status st = check_conv_ws(H, L, workspace, workspace_bytes);
  if (st != DLR_OK) return st;
  return from_cuda(dlr::launch_dlr_conv_apply(u, (int)B, (int)H, (int)L, y, workspace,
                                              (cudaStream_t)stream));
}

dlr_status dlr_conv(const float* u, const float* K_fwd, const float* K_bwd, dlr_dir dir,
                    int64_t B, int64_t H, int64_t L, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream) {
  if (B < 1 || H < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (!u || !y || !aligned16(u) || !aligned16(y)) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  if (ranges_overlap(u, bytes, y, bytes)) return DLR_ERR_INVALID_ARG;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return DLR_ERR_INVALID_ARG;
  if (!K_fwd || !aligned16(K_fwd)) return DLR_ERR_INVALID_ARG;
  if (dir == DLR_BIDIR && (!K_bwd || !aligned16(K_bwd))) return DLR_ERR_INVALID_ARG;
  if (dir == DLR_CAUSAL && K_bwd) return DLR_ERR_INVALID_ARG;
  if (L > 65536 || B * H > kMaxGrid / 8) return DLR_ERR_UNSUPPORTED;
  dlr_status st = check_conv_ws(H, L, workspace, workspace_bytes);
  if (st != DLR_OK) return st;
  st = dlr_conv_spectrum(K_fwd, K_bwd, dir, H, L, workspace, workspace_bytes, stream);
  if (st != DLR_OK) return st;
  return dlr_conv_apply(u, B, H, L, y, workspace, workspace_bytes, stream);
}

size_t dlr_scan_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L) {
  if (B < 1 || H < 1 || N < 1 || L < 1 || N > 64) return 0;
  return dlr::scan_tc_workspace_bytes(H);
}

dlr_status dlr_scan(const float* u, const float* log_re, const float* log_im, const float* W,
                    const float* log_re2, const float* log_im2, const float* W2, dlr_dir dir,
                    int64_t B, int64_t H, int64_t N, int64_t L, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream) {
  return dlr_scan_ex(u, log_re, log_im, W, log_re2, log_im2, W2, dir, B, H, N, L, y,
                     DLR_SCAN_AUTO, workspace, workspace_bytes, stream);
}

dlr_status dlr_scan_ex(const float* u, const float* log_re, const float* log_im, const float* W,
                       const float* log_re2, const float* log_im2, const float* W2, dlr_dir dir,
                       int64_t B, int64_t H, int64_t N, int64_t L, float* y,
                       dlr_scan_algo algo, void* workspace, size_t workspace_bytes,
                       dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (algo != DLR_SCAN_AUTO && algo != DLR_SCAN_FP32 && algo != DLR_SCAN_TENSOR)
    return DLR_ERR_INVALID_ARG;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return DLR_ERR_INVALID_ARG;
  if (!u || !y || !aligned16(u) || !aligned16(y)) return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  if (dir == DLR_BIDIR) {
    st = check_params(log_re2, log_im2, W2);
    if (st != DLR_OK) return st;
  }
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  if (ranges_overlap(u, bytes, y, bytes)) return DLR_ERR_INVALID_ARG;
  if (N > 128 || L > kMaxL || B * H > kMaxGrid) return DLR_ERR_UNSUPPORTED;
  if (algo == DLR_SCAN_TENSOR && N > 64) return DLR_ERR_UNSUPPORTED;
  const bool tensor = algo == DLR_SCAN_TENSOR || (algo == DLR_SCAN_AUTO && N <= 64);
  if (tensor) {
    const size_t need = dlr::scan_tc_workspace_bytes(H);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
    if (ranges_overlap(workspace, need, u, bytes) || ranges_overlap(workspace, need, y, bytes))
      return DLR_ERR_INVALID_ARG;
    return from_cuda(dlr::launch_dlr_scan_tc(u, log_re, log_im, W, log_re2, log_im2, W2,
                                             dir == DLR_BIDIR, (int)B, (int)H, (int)N, (int)L,
                                             y, workspace, status_word(), (cudaStream_t)stream));
  }
  return from_cuda(dlr::launch_dlr_scan(u, log_re, log_im, W, log_re2, log_im2, W2,
                                        dir == DLR_BIDIR, (int)B, (int)H, (int)N, (int)L, y,
                                        (cudaStream_t)stream));
}

dlr_status dlr_scan_prepare(const float* log_re, const float* log_im, const float* W, int64_t H,
                            int64_t N, void* workspace, size_t workspace_bytes,
                            dlr_stream_t stream) {
  if (H < 1 || N < 1) return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  if (N > 64 || H > kMaxGrid) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr::scan_tc_workspace_bytes(H);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  return from_cuda(dlr::launch_scan_tc_tables(log_re, log_im, W, (int)H, (int)N, workspace,
                                              (cudaStream_t)stream));
}

dlr_status dlr_scan_apply(const float* u, int64_t B, int64_t H, int64_t N, int64_t L,
                          int reverse, float* y, const void* workspace, size_t workspace_bytes,
                          dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (reverse != 0 && reverse != 1) return DLR_ERR_INVALID_ARG;
  if (!u || !y || !aligned16(u) || !aligned16(y)) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  if (ranges_overlap(u, bytes, y, bytes)) return DLR_ERR_INVALID_ARG;
  if (N > 64 || L > kMaxL || B * H > kMaxGrid) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr::scan_tc_workspace_bytes(H);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  if (ranges_overlap(workspace, need, u, bytes) || ranges_overlap(workspace, need, y, bytes))
    return DLR_ERR_INVALID_ARG;
  return from_cuda(dlr::launch_scan_tc_apply(u, (int)B, (int)H, (int)L, reverse != 0, y,
                                             workspace, status_word(), (cudaStream_t)stream,
                                             false));
}

size_t dlr_scan_backward_params_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L) {
  if (B < 1 || H < 1 || N < 1 || L < 1 || L > kMaxL) return 0;
  return dlr::grad_workspace_bytes(B, H, N, L);
}

dlr_status dlr_scan_backward_params(const float* u, const float* g, const float* log_re,
                                    const float* log_im, const float* W, int64_t B, int64_t H,
                                    int64_t N, int64_t L, float* d_log_re, float* d_log_im,
                                    float* dW, void* workspace, size_t workspace_bytes,
                                    dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (!u || !g || !d_log_re || !d_log_im || !dW) return DLR_ERR_INVALID_ARG;
  auto al4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  auto al8 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; };
  if (!al4(u) || !al4(g) || !al4(d_log_re) || !al4(d_log_im) || !al8(dW))
    return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  const size_t pn = sizeof(float) * (size_t)H * (size_t)N;
  // the outputs must not overlap the parameters or each other
  const void* outs[3] = {d_log_re, d_log_im, dW};
  const size_t osz[3] = {pn, pn, 2 * pn};
  const void* ins[3] = {log_re, log_im, W};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j)
      if (ranges_overlap(outs[i], osz[i], ins[j], osz[j])) return DLR_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (ranges_overlap(outs[i], osz[i], outs[j], osz[j])) return DLR_ERR_INVALID_ARG;
  }
  if (L > kMaxL || B * H > kMaxGrid / 64 || N > 65536) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr::grad_workspace_bytes(B, H, N, L);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  return from_cuda(dlr::launch_dlr_grad_params(u, g, log_re, log_im, W, (int)B, (int)H, (int)N,
                                               (int)L, d_log_re, d_log_im, dW, workspace,
                                               status_word(), (cudaStream_t)stream));
}

// Workspace of dlr_layer_backward: the gradients' part, then the two kernels of the input
// gradient's convolution and the convolution workspace, each rounded up to 256 bytes.
namespace {
size_t round256(size_t b) { return (b + 255) & ~size_t(255); }
size_t layer_bwd_grads_bytes(int64_t B, int64_t H, int64_t N, int64_t L, bool bidir, bool prod) {
  return round256(dlr::grads_workspace_bytes(B, H, N, L, bidir, prod));
}
}  // namespace

size_t dlr_layer_backward_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L,
                                         dlr_dir dir, dlr_cast cast) {
  if (B < 1 || H < 1 || N < 1 || L < 1 || L > 65536) return 0;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return 0;
  if (cast != DLR_CAST_RE && cast != DLR_CAST_RE_IM) return 0;
  const size_t hl = sizeof(float) * (size_t)H * (size_t)L;
  return layer_bwd_grads_bytes(B, H, N, L, dir == DLR_BIDIR, cast == DLR_CAST_RE_IM) +
         2 * round256(hl) + dlr::conv_workspace_bytes(H, L);
}

dlr_status dlr_layer_backward(const float* u, const float* g, const float* log_re,
                              const float* log_im, const float* W, const float* log_re2,
                              const float* log_im2, const float* W2, dlr_dir dir, dlr_cast cast,
                              int64_t B, int64_t H, int64_t N, int64_t L, float* du,
                              float* d_log_re, float* d_log_im, float* dW, float* d_log_re2,
                              float* d_log_im2, float* dW2, void* workspace,
                              size_t workspace_bytes, dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return DLR_ERR_INVALID_ARG;
  if (cast != DLR_CAST_RE && cast != DLR_CAST_RE_IM) return DLR_ERR_INVALID_ARG;
  const bool bidir = dir == DLR_BIDIR, prod = cast == DLR_CAST_RE_IM;
  if (!u || !g || !aligned16(u) || !aligned16(g)) return DLR_ERR_INVALID_ARG;
  if (du && !aligned16(du)) return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  if (bidir) {
    st = check_params(log_re2, log_im2, W2);
    if (st != DLR_OK) return st;
  } else if (log_re2 || log_im2 || W2 || d_log_re2 || d_log_im2 || dW2) {
    return DLR_ERR_INVALID_ARG;
  }
  auto al4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  auto al8 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; };
  const int sets = bidir ? 2 : 1;
  float* outs[6] = {d_log_re, d_log_im, dW, d_log_re2, d_log_im2, dW2};
  const float* ins[6] = {log_re, log_im, W, log_re2, log_im2, W2};
  const size_t pn = sizeof(float) * (size_t)H * (size_t)N;
  const size_t sz[6] = {pn, pn, 2 * pn, pn, pn, 2 * pn};
  for (int i = 0; i < 3 * sets; ++i) {
    if (!outs[i] || !al4(outs[i]) || (i % 3 == 2 && !al8(outs[i]))) return DLR_ERR_INVALID_ARG;
    for (int j = 0; j < 3 * sets; ++j)
      if (ranges_overlap(outs[i], sz[i], ins[j], sz[j])) return DLR_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3 * sets; ++j)
      if (ranges_overlap(outs[i], sz[i], outs[j], sz[j])) return DLR_ERR_INVALID_ARG;
  }
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  if (du) {
    if (ranges_overlap(du, bytes, u, bytes) || ranges_overlap(du, bytes, g, bytes))
      return DLR_ERR_INVALID_ARG;
    for (int i = 0; i < 3 * sets; ++i)
      if (ranges_overlap(du, bytes, outs[i], sz[i])) return DLR_ERR_INVALID_ARG;
  }
  if (L > 65536 || N > 65536 || B * H > kMaxGrid / 64) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr_layer_backward_workspace_size(B, H, N, L, dir, cast);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  if (ranges_overlap(workspace, need, u, bytes) || ranges_overlap(workspace, need, g, bytes) ||
      (du && ranges_overlap(workspace, need, du, bytes)))
    return DLR_ERR_INVALID_ARG;
  for (int i = 0; i < 3 * sets; ++i)
    if (ranges_overlap(workspace, need, outs[i], sz[i])) return DLR_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = status_word();
  // du's kernels: kappa1 of the first direction, kappa2 of the second (zero for a causal
  // layer); with the DLR-prod cast the gradients' complex kernels give them
  const size_t hl = sizeof(float) * (size_t)H * (size_t)L;
  uint8_t* p = ws + layer_bwd_grads_bytes(B, H, N, L, bidir, prod);
  float* kap1 = reinterpret_cast<float*>(p);
  float* kap2 = reinterpret_cast<float*>(p + round256(hl));
  void* cws = p + 2 * round256(hl);
  cudaError_t e = dlr::launch_dlr_grads(u, g, log_re, log_im, W, log_re2, log_im2, W2, (int)B,
                                        (int)H, (int)N, (int)L, prod, d_log_re, d_log_im, dW,
                                        d_log_re2, d_log_im2, dW2, ws, status, s,
                                        du && prod ? kap1 : nullptr,
                                        du && prod ? kap2 : nullptr);
  if (e != cudaSuccess || !du) return from_cuda(e);
  // du: the convolution of g whose causal kernel is the second direction's and whose
  // anti-causal kernel is the first's (the adjoint swaps the directions)
  if (!prod) {
    if ((e = dlr::launch_dlr_kernel(log_re, log_im, W, (int)H, (int)N, (int)L, false, kap1,
                                    status, s)) != cudaSuccess)
      return from_cuda(e);
    if (bidir &&
        (e = dlr::launch_dlr_kernel(log_re2, log_im2, W2, (int)H, (int)N, (int)L, false, kap2,
                                    status, s)) != cudaSuccess)
      return from_cuda(e);
  }
  if (!bidir && (e = cudaMemsetAsync(kap2, 0, hl, s)) != cudaSuccess) return from_cuda(e);
  if ((e = dlr::launch_dlr_conv_spectrum(kap2, kap1, (int)H, (int)L, cws, s)) != cudaSuccess)
    return from_cuda(e);
  return from_cuda(dlr::launch_dlr_conv_apply(g, (int)B, (int)H, (int)L, du, cws, s));
}

dlr_status dlr_scan_backward_input(const float* g, const float* log_re, const float* log_im,
                                   const float* W, int64_t B, int64_t H, int64_t N, int64_t L,
                                   float* du, void* workspace, size_t workspace_bytes,
                                   dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (!g || !du || !aligned16(g) || !aligned16(du)) return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  if (ranges_overlap(g, bytes, du, bytes)) return DLR_ERR_INVALID_ARG;
  if (N > 64 || L > kMaxL || B * H > kMaxGrid) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr::scan_tc_workspace_bytes(H);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  if (ranges_overlap(workspace, need, g, bytes) || ranges_overlap(workspace, need, du, bytes))
    return DLR_ERR_INVALID_ARG;
  // du = rev(DLR(rev(g))) with the same parameters: the reversed pass adds into du
  cudaError_t e = cudaMemsetAsync(du, 0, bytes, (cudaStream_t)stream);
  if (e == cudaSuccess)
    e = dlr::launch_scan_tc_tables(log_re, log_im, W, (int)H, (int)N, workspace,
                                   (cudaStream_t)stream);
  if (e == cudaSuccess)
    e = dlr::launch_scan_tc_apply(g, (int)B, (int)H, (int)L, true, du, workspace, status_word(),
                                  (cudaStream_t)stream, true);
  return from_cuda(e);
}

size_t dlr_step_workspace_size(int64_t H, int64_t N) {
  if (H < 1 || N < 1 || N > 256 || H > (int64_t(1) << 31)) return 0;
  return dlr::step_workspace_bytes(H, N);
}

dlr_status dlr_step_prepare(const float* log_re, const float* log_im, const float* W, int64_t H,
                            int64_t N, void* workspace, size_t workspace_bytes,
                            dlr_stream_t stream) {
  if (H < 1 || N < 1) return DLR_ERR_INVALID_ARG;
  dlr_status st = check_params(log_re, log_im, W);
  if (st != DLR_OK) return st;
  if (N > 256 || H > (int64_t(1) << 31)) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr::step_workspace_bytes(H, N);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  return from_cuda(dlr::launch_step_tables(log_re, log_im, W, H, N, workspace,
                                           (cudaStream_t)stream));
}

dlr_status dlr_step(const float* u, int64_t B, int64_t H, int64_t N, int64_t T, float* x,
                    float* y, const void* workspace, size_t workspace_bytes,
                    dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || T < 0) return DLR_ERR_INVALID_ARG;
  if (N > 256 || T > kMaxL || B * H > kMaxGrid) return DLR_ERR_UNSUPPORTED;
  if (!x || !aligned16(x)) return DLR_ERR_INVALID_ARG;
  const size_t need = dlr::step_workspace_bytes(H, N);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  const size_t xbytes = 2 * sizeof(float) * (size_t)B * (size_t)H * (size_t)N;
  if (ranges_overlap(workspace, need, x, xbytes)) return DLR_ERR_INVALID_ARG;
  if (T == 0) return DLR_OK;
  if (!u || !y || !aligned16(u) || !aligned16(y)) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)T;
  if (ranges_overlap(u, bytes, y, bytes) || ranges_overlap(x, xbytes, u, bytes) ||
      ranges_overlap(x, xbytes, y, bytes) || ranges_overlap(workspace, need, u, bytes) ||
      ranges_overlap(workspace, need, y, bytes))
    return DLR_ERR_INVALID_ARG;
  return from_cuda(dlr::launch_step(u, B, H, N, T, workspace, x, y, (cudaStream_t)stream));
}

size_t s5_workspace_size(int64_t B, int64_t L, int64_t H, int64_t P, dlr_prec prec) {
  if (B < 1 || L < 1 || H < 1 || P < 1) return 0;
  return dlr::s5_workspace_bytes(B, L, H, P, prec == DLR_BF16_TC);
}

static dlr_status s5_common(const float* u, const float* lambda, const float* log_delta,
                            const float* Bt, const float* Ct, const float* D, int64_t B,
                            int64_t L, int64_t H, int64_t P, dlr_prec prec, dlr_disc disc,
                            float* y, void* workspace, size_t workspace_bytes,
                            dlr_stream_t stream) {
  if (B < 1 || L < 1 || H < 1 || P < 1) return DLR_ERR_INVALID_ARG;
  if (prec != DLR_FP32 && prec != DLR_BF16_TC) return DLR_ERR_INVALID_ARG;
  if (disc != DLR_DISC_ZOH && disc != DLR_DISC_BILINEAR) return DLR_ERR_INVALID_ARG;
  const void* ptrs[] = {u, lambda, log_delta, Bt, Ct, D, y};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)L * (size_t)H;
  if (ranges_overlap(u, bytes, y, bytes)) return DLR_ERR_INVALID_ARG;
  if (H % 32 || P % 32 || H > 1024 || P > 1024) return DLR_ERR_UNSUPPORTED;
  if (B > 65535 || (L + 63) / 64 > 65535 || B * L > kMaxGrid / 4) return DLR_ERR_UNSUPPORTED;
  const bool bf16 = prec == DLR_BF16_TC;
  const size_t need = dlr::s5_workspace_bytes(B, L, H, P, bf16);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_s5(u, lambda, log_delta, Bt, Ct, D, (int)B, (int)L, (int)H,
                                  (int)P, bf16, disc == DLR_DISC_BILINEAR, y, workspace, status,
                                  (cudaStream_t)stream));
}

dlr_status s5_layer(const float* u, const float* lambda, const float* log_delta,
                    const float* Bt, const float* Ct, const float* D, int64_t B, int64_t L,
                    int64_t H, int64_t P, dlr_prec prec, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream) {
  return s5_common(u, lambda, log_delta, Bt, Ct, D, B, L, H, P, prec, DLR_DISC_ZOH, y, workspace,
                   workspace_bytes, stream);
}

dlr_status s5_layer_ex(const float* u, const float* lambda, const float* log_delta,
                       const float* Bt, const float* Ct, const float* D, int64_t B, int64_t L,
                       int64_t H, int64_t P, dlr_prec prec, dlr_disc disc, float* y,
                       void* workspace, size_t workspace_bytes, dlr_stream_t stream) {
  return s5_common(u, lambda, log_delta, Bt, Ct, D, B, L, H, P, prec, disc, y, workspace,
                   workspace_bytes, stream);
}

size_t s5_layer_tv_workspace_size(int64_t B, int64_t L, int64_t H, int64_t P) {
  if (B < 1 || L < 1 || H < 1 || P < 1) return 0;
  return dlr::s5_workspace_bytes(B, L, H, P, false);
}

dlr_status s5_layer_tv(const float* u, const float* dt, const float* lambda,
                       const float* log_delta, const float* Bt, const float* Ct, const float* D,
                       int64_t B, int64_t L, int64_t H, int64_t P, float* y, void* workspace,
                       size_t workspace_bytes, dlr_stream_t stream) {
  if (B < 1 || L < 1 || H < 1 || P < 1) return DLR_ERR_INVALID_ARG;
  const void* ptrs[] = {u, dt, lambda, log_delta, Bt, Ct, D, y};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)L * (size_t)H;
  if (ranges_overlap(u, bytes, y, bytes) ||
      ranges_overlap(dt, sizeof(float) * (size_t)B * (size_t)L, y, bytes))
    return DLR_ERR_INVALID_ARG;
  if (H % 32 || P % 32 || H > 1024 || P > 1024) return DLR_ERR_UNSUPPORTED;
  if (B > 65535 || (L + 63) / 64 > 65535 || B * L > kMaxGrid / 4) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr::s5_workspace_bytes(B, L, H, P, false);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_s5_tv(u, dt, lambda, log_delta, Bt, Ct, D, (int)B, (int)L, (int)H,
                                     (int)P, y, workspace, status, (cudaStream_t)stream));
}

dlr_status dlr_params_from_dss_exp(const float* Lambda, const float* log_delta, const float* W,
                                   int64_t H, int64_t N, float* log_re, float* log_im,
                                   float* W_out, dlr_stream_t stream) {
  if (H < 1 || N < 1) return DLR_ERR_INVALID_ARG;
  auto al8 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; };
  auto al4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!Lambda || !log_delta || !W || !log_re || !log_im || !W_out) return DLR_ERR_INVALID_ARG;
  if (!al8(Lambda) || !al8(W) || !al8(W_out) || !al4(log_delta) || !al4(log_re) || !al4(log_im))
    return DLR_ERR_INVALID_ARG;
  const size_t pn = sizeof(float) * (size_t)H * (size_t)N;
  const void* outs[3] = {log_re, log_im, W_out};
  const size_t osz[3] = {pn, pn, 2 * pn};
  const void* ins[3] = {Lambda, log_delta, W};
  const size_t isz[3] = {2 * pn, sizeof(float) * (size_t)H, 2 * pn};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j)
      if (ranges_overlap(outs[i], osz[i], ins[j], isz[j])) return DLR_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (ranges_overlap(outs[i], osz[i], outs[j], osz[j])) return DLR_ERR_INVALID_ARG;
  }
  if ((int64_t)H * N > kMaxGrid * 64) return DLR_ERR_UNSUPPORTED;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_dss_exp_map(Lambda, log_delta, W, H, N, log_re, log_im, W_out,
                                           status, (cudaStream_t)stream));
}

dlr_status dlr_log_re_from_reparam(const float* w, int64_t count, dlr_reparam kind, float a,
                                   float b, float* log_re, dlr_stream_t stream) {
  if (count < 1 || !w || !log_re) return DLR_ERR_INVALID_ARG;
  auto al4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(w) || !al4(log_re)) return DLR_ERR_INVALID_ARG;
  if (kind != DLR_REPARAM_EXP && kind != DLR_REPARAM_SOFTPLUS && kind != DLR_REPARAM_BEST)
    return DLR_ERR_INVALID_ARG;
  if (kind == DLR_REPARAM_BEST && !(a >= 0.f && b > 0.f)) return DLR_ERR_INVALID_ARG;
  if (count > kMaxGrid * 64) return DLR_ERR_UNSUPPORTED;
  return from_cuda(dlr::launch_reparam_map(w, count, (int)kind, a, b, log_re,
                                           (cudaStream_t)stream));
}

size_t dlr_scan_host_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return 0;
  const size_t data = align256(sizeof(float) * (size_t)B * (size_t)H * (size_t)L);
  const size_t par = align256(sizeof(float) * (size_t)H * (size_t)N);
  return 2 * data + 4 * par + dlr::scan_tc_workspace_bytes(H);
}

dlr_status dlr_scan_host(const float* u, const float* log_re, const float* log_im,
                         const float* W, int64_t B, int64_t H, int64_t N, int64_t L, float* y,
                         void* workspace, size_t workspace_bytes, dlr_stream_t stream) {
  if (B < 1 || H < 1 || N < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (!u || !y || !log_re || !log_im || !W) return DLR_ERR_INVALID_ARG;
  const size_t rows = (size_t)B * (size_t)H;
  const size_t bytes = sizeof(float) * rows * (size_t)L;
  if (ranges_overlap(u, bytes, y, bytes)) return DLR_ERR_INVALID_ARG;
  if (N > 64 || L > kMaxL || B * H > kMaxGrid) return DLR_ERR_UNSUPPORTED;
  const size_t need = dlr_scan_host_workspace_size(B, H, N, L);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return DLR_ERR_WORKSPACE;
  char* base = static_cast<char*>(workspace);
  const size_t data = align256(bytes), par = align256(sizeof(float) * (size_t)H * (size_t)N);
  float* ud = reinterpret_cast<float*>(base);
  float* yd = reinterpret_cast<float*>(base + data);
  float* lrd = reinterpret_cast<float*>(base + 2 * data);
  float* lid = reinterpret_cast<float*>(base + 2 * data + par);
  float* Wd = reinterpret_cast<float*>(base + 2 * data + 2 * par);
  char* tables = base + 2 * data + 4 * par;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;

  cudaStream_t st[3];
  cudaError_t e = pipe_streams(st);
  if (e != cudaSuccess) return from_cuda(e);
  // pieces: groups of whole batch rows when B >= 4, else channel groups of each batch row, so
  // that a piece is one contiguous [B', H', L] block whose tables start at channel h0
  // (one piece when L % 4 != 0: piece starts must stay 16-byte aligned)
  const int64_t kTarget = L % 4 ? 1 : 4;
  const int64_t per_b = B >= kTarget ? (B + kTarget - 1) / kTarget : 1;
  const int64_t groups = B >= kTarget ? 1 : std::min<int64_t>(H, (kTarget + B - 1) / B);
  const int64_t per_h = (H + groups - 1) / groups;
  const size_t table_bytes = dlr::scan_tc_workspace_bytes(1);

  cudaEvent_t ev_start, ev_par, ev_end;
  auto mk = [](cudaEvent_t* ev) { return cudaEventCreateWithFlags(ev, cudaEventDisableTiming); };
  if ((e = mk(&ev_start)) != cudaSuccess) return from_cuda(e);
  if ((e = mk(&ev_par)) != cudaSuccess || (e = mk(&ev_end)) != cudaSuccess) {
    cudaEventDestroy(ev_start);
    return from_cuda(e);
  }
  auto run = [&]() -> cudaError_t {
    cudaError_t r;
    // the caller's earlier work on `stream` comes first
    if ((r = cudaEventRecord(ev_start, (cudaStream_t)stream)) != cudaSuccess) return r;
    for (int i = 0; i < 3; ++i)
      if ((r = cudaStreamWaitEvent(st[i], ev_start, 0)) != cudaSuccess) return r;
    const size_t pb = sizeof(float) * (size_t)H * (size_t)N;
    if ((r = cudaMemcpyAsync(lrd, log_re, pb, cudaMemcpyHostToDevice, st[0])) != cudaSuccess ||
        (r = cudaMemcpyAsync(lid, log_im, pb, cudaMemcpyHostToDevice, st[0])) != cudaSuccess ||
        (r = cudaMemcpyAsync(Wd, W, 2 * pb, cudaMemcpyHostToDevice, st[0])) != cudaSuccess)
      return r;
    if ((r = cudaEventRecord(ev_par, st[0])) != cudaSuccess) return r;
    if ((r = cudaStreamWaitEvent(st[1], ev_par, 0)) != cudaSuccess) return r;
    if ((r = dlr::launch_scan_tc_tables(lrd, lid, Wd, (int)H, (int)N, tables, st[1])) !=
        cudaSuccess)
      return r;
    // the first and last groups of rows are halved: nothing overlaps the first piece's copy in
    // or the last piece's compute and copy out, so smaller end pieces shorten both
    for (int64_t b0 = 0, nb = 0; b0 < B; b0 += nb) {
      nb = std::min(per_b, B - b0);
      if (b0 == 0 && nb > 1 && B > per_b) nb /= 2;
      if (b0 + nb == B && nb > 1) nb /= 2;
      for (int64_t h0 = 0; h0 < H; h0 += per_h) {
        const int64_t nh = std::min(per_h, H - h0);
        // a piece is contiguous: whole batch rows (nh == H) or channels of one batch row
        const size_t off = ((size_t)b0 * (size_t)H + (size_t)h0) * (size_t)L;
        const size_t pbytes = sizeof(float) * (size_t)nb * (size_t)nh * (size_t)L;
        cudaEvent_t in, done;
        if ((r = mk(&in)) != cudaSuccess) return r;
        if ((r = mk(&done)) != cudaSuccess) {
          cudaEventDestroy(in);
          return r;
        }
        r = cudaMemcpyAsync(ud + off, u + off, pbytes, cudaMemcpyHostToDevice, st[0]);
        if (r == cudaSuccess) r = cudaEventRecord(in, st[0]);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(st[1], in, 0);
        if (r == cudaSuccess)
          r = dlr::launch_scan_tc_apply(ud + off, (int)nb, (int)nh, (int)L, false, yd + off,
                                        tables + (size_t)h0 * table_bytes, status, st[1],
                                        false);
        if (r == cudaSuccess) r = cudaEventRecord(done, st[1]);
        if (r == cudaSuccess) r = cudaStreamWaitEvent(st[2], done, 0);
        if (r == cudaSuccess)
          r = cudaMemcpyAsync(y + off, yd + off, pbytes, cudaMemcpyDeviceToHost, st[2]);
        cudaEventDestroy(in);  // released once recorded work completes
        cudaEventDestroy(done);
        if (r != cudaSuccess) return r;
      }
    }
    // the caller's later work on `stream` waits for the last copy out (which follows every
    // piece's compute, itself after the tables)
    if ((r = cudaEventRecord(ev_end, st[2])) != cudaSuccess) return r;
    return cudaStreamWaitEvent((cudaStream_t)stream, ev_end, 0);
  };
  e = run();
  if (e != cudaSuccess) {
    // Some pieces may already be queued on the internal streams, reading the caller's host
    // buffers and workspace: let them finish before the error returns, so that the caller may
    // free or reuse those buffers at once.
    for (int i = 0; i < 3; ++i) cudaStreamSynchronize(st[i]);
  }
  cudaEventDestroy(ev_start);
  cudaEventDestroy(ev_par);
  cudaEventDestroy(ev_end);
  return from_cuda(e);
}

dlr_status dlr_selftest_timeout(int limit_ms, dlr_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 2000) return DLR_ERR_INVALID_ARG;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_selftest_timeout((uint64_t)limit_ms * 1000000ull, status,
                                                (cudaStream_t)stream));
}

int dlr_bounds_checked(void) {
#ifdef DLR_BOUNDS_CHECK
  return 1;
#else
  return 0;
#endif
}

int dlr_bounds_site(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dlr_bounds_site, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dlr_bounds_site, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

dlr_status dlr_selftest_bounds(dlr_stream_t stream) {
#ifdef DLR_BOUNDS_CHECK
  return from_cuda(dlr::launch_selftest_bounds((cudaStream_t)stream));
#else
  (void)stream;
  return DLR_ERR_UNSUPPORTED;
#endif
}

dlr_status dlr_get_device_status(dlr_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DLR_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dlr_device_status, sizeof(int)) != cudaSuccess)
    return DLR_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_dlr_device_status, &zero, sizeof(int)) != cudaSuccess)
      return DLR_ERR_CUDA;
  }
  return (dlr_status)v;
}

}  // extern "C"
