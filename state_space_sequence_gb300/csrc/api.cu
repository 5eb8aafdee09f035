// api.cu -- the extern "C" entry points declared in include/dlr.h: argument validation,
// workspace carving and kernel dispatch on the caller's stream.
#include <cuda_runtime.h>

#include "dlr.h"

namespace dlr {
cudaError_t launch_dlr_kernel(const float* log_re, const float* log_im, const float* W, int H,
                              int N, int L, bool re_im, float* K, cudaStream_t s);
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
                      bool bf16, float* y, void* ws, int* status, cudaStream_t s);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s);
}  // namespace dlr

// The library's device status word (one per device that loads the library).
__device__ int g_dlr_device_status = 0;

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

// The last CUDA error a call of this thread turned into DLR_ERR_CUDA (for diagnostics).
thread_local const char* t_last_cuda_error = "no error";

dlr_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DLR_OK;
  t_last_cuda_error = cudaGetErrorString(e);
  return DLR_ERR_CUDA;
}

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

int dlr_abi_version(void) { return 3; }

const char* dlr_last_cuda_error(void) { return t_last_cuda_error; }

const char* dlr_status_string(dlr_status s) {
  switch (s) {
    case DLR_OK: return "DLR_OK";
    case DLR_ERR_INVALID_ARG: return "DLR_ERR_INVALID_ARG";
    case DLR_ERR_UNSUPPORTED: return "DLR_ERR_UNSUPPORTED";
    case DLR_ERR_CUDA: return "DLR_ERR_CUDA";
    case DLR_ERR_TIMEOUT: return "DLR_ERR_TIMEOUT";
    case DLR_ERR_WORKSPACE: return "DLR_ERR_WORKSPACE";
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
  return from_cuda(dlr::launch_dlr_kernel(log_re, log_im, W, (int)H, (int)N, (int)L,
                                          cast == DLR_CAST_RE_IM, K, (cudaStream_t)stream));
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

size_t s5_workspace_size(int64_t B, int64_t L, int64_t H, int64_t P, dlr_prec prec) {
  if (B < 1 || L < 1 || H < 1 || P < 1) return 0;
  return dlr::s5_workspace_bytes(B, L, H, P, prec == DLR_BF16_TC);
}

dlr_status s5_layer(const float* u, const float* lambda, const float* log_delta,
                    const float* Bt, const float* Ct, const float* D, int64_t B, int64_t L,
                    int64_t H, int64_t P, dlr_prec prec, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream) {
  if (B < 1 || L < 1 || H < 1 || P < 1) return DLR_ERR_INVALID_ARG;
  if (prec != DLR_FP32 && prec != DLR_BF16_TC) return DLR_ERR_INVALID_ARG;
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
  int* status = bf16 ? status_word() : nullptr;
  if (bf16 && !status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_s5(u, lambda, log_delta, Bt, Ct, D, (int)B, (int)L, (int)H,
                                  (int)P, bf16, y, workspace, status, (cudaStream_t)stream));
}

dlr_status dlr_selftest_timeout(int limit_ms, dlr_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 2000) return DLR_ERR_INVALID_ARG;
  int* status = status_word();
  if (!status) return DLR_ERR_CUDA;
  return from_cuda(dlr::launch_selftest_timeout((uint64_t)limit_ms * 1000000ull, status,
                                                (cudaStream_t)stream));
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
