// dlr_backward.cu -- gradients of the causal DLR layer (Re cast) with respect to its parameters
// ("Simplifying and Understanding State Space Models with Diagonal Linear RNNs", section 2:
// y_k = sum_{j<=k} Re K_j u_{k-j}, K_j = sum_n W_n lambda_n^j, and the gradient analysis there,
// d K_j / d lambda_n = W_n j lambda_n^{j-1}, d K_j / d W_n = lambda_n^j; section 2.2:
// lambda = exp(-a^2 + i theta), a = (log Lambda)_re, theta = (log Lambda)_im).
//
// For a loss with gradient g [B, H, L] with respect to y, let c_j = sum_b sum_k g_{b,k} u_{b,k-j}.
// Then, with S0 = sum_j c_j lambda^j and S1 = sum_j j c_j lambda^j,
//     dW = (Re S0, -Im S0),   d a = -2 a Re(W S1),   d theta = -Im(W S1).
// Both sums are sums over the steps of g against states of the forward recurrence driven by u:
//     S0 = sum_b sum_k g_{b,k} x_k,          x_k = lambda x_{k-1} + u_k
//     S1 = sum_b sum_k g_{b,k} D_k,          D_k = sum_j j lambda^j u_{k-j} = lambda (D_{k-1} + x_{k-1})
// (the second recurrence is lambda times the derivative of x with respect to lambda), so the
// gradients need neither the kernel nor the correlation c.
//
// dlr_grad_rows: one thread per (b, h, n) runs both recurrences over the row. lambda is the
// float pair hi + lo of its double-precision value (as in the recurrent mode), so its rounding
// does not compound over the row. A warp holds 32 states of one (b, h) row: lane j loads
// u_{k0+j} and g_{k0+j}, the steps take them by shuffles. The products are summed in float
// over each block of 32 steps, the blocks into the running sums. Each thread leaves its
// row's (S0, S1) in the workspace; dlr_grad_finish adds the B rows of each (h, n) and forms
// the three gradients.
#include <cuda_runtime.h>

#include <cstdint>

#include "dlr_common.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 2;

namespace {

constexpr int kGradWarps = 4;  // warps per block

__global__ void __launch_bounds__(kGradWarps * 32)
    dlr_grad_rows(const float* __restrict__ u, const float* __restrict__ g,
                  const float* __restrict__ log_re, const float* __restrict__ log_im, int B,
                  int H, int N, int L, int warps_per_row, float4* __restrict__ part) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * kGradWarps + (threadIdx.x >> 5);
  const int64_t row = wid / warps_per_row;  // (b, h)
  if (row >= (int64_t)B * H) return;        // whole warps only
  const int n = (int)(wid - row * warps_per_row) * 32 + lane;
  const int h = (int)(row % H);
  const bool on = n < N;
  // lambda as a float pair
  float lhr = 0.f, lhi = 0.f, llr = 0.f, lli = 0.f;
  if (on) {
    const double a = log_re[(size_t)h * N + n], th = log_im[(size_t)h * N + n];
    const double mag = exp(-a * a);
    double s, c;
    sincos(th, &s, &c);
    const double re = mag * c, im = mag * s;
    lhr = (float)re;
    lhi = (float)im;
    llr = (float)(re - (double)lhr);
    lli = (float)(im - (double)lhi);
  }
  const float* ur = u + row * (int64_t)L;
  const float* gr = g + row * (int64_t)L;
  float xr = 0.f, xi = 0.f, dr = 0.f, di = 0.f;
  float s0r = 0.f, s0i = 0.f, s1r = 0.f, s1i = 0.f;
#pragma unroll 1
  for (int k0 = 0; k0 < L; k0 += 32) {
    const int k = k0 + lane;
    const float uk = k < L ? __ldg(ur + k) : 0.f;
    const float gk = k < L ? __ldg(gr + k) : 0.f;
    const int steps = min(32, L - k0);
    float p0r = 0.f, p0i = 0.f, p1r = 0.f, p1i = 0.f;
#pragma unroll 8
    for (int t = 0; t < steps; ++t) {
      const float ut = __shfl_sync(0xffffffffu, uk, t);
      const float gt = __shfl_sync(0xffffffffu, gk, t);
      // D_k = lambda (D_{k-1} + x_{k-1}), then x_k = lambda x_{k-1} + u_k (lambda = hi + lo,
      // the lo products first)
      const float er = dr + xr, ei = di + xi;
      dr = fmaf(lhr, er, fmaf(-lhi, ei, fmaf(llr, er, -lli * ei)));
      di = fmaf(lhr, ei, fmaf(lhi, er, fmaf(llr, ei, lli * er)));
      const float nr = fmaf(lhr, xr, fmaf(-lhi, xi, fmaf(llr, xr, fmaf(-lli, xi, ut))));
      const float ni = fmaf(lhr, xi, fmaf(lhi, xr, fmaf(llr, xi, lli * xr)));
      xr = nr;
      xi = ni;
      p0r = fmaf(gt, xr, p0r);
      p0i = fmaf(gt, xi, p0i);
      p1r = fmaf(gt, dr, p1r);
      p1i = fmaf(gt, di, p1i);
    }
    s0r += p0r;
    s0i += p0i;
    s1r += p1r;
    s1i += p1i;
  }
  if (on && DLR_IN(row * (int64_t)N + n, (int64_t)B * H * N))
    part[row * (int64_t)N + n] = make_float4(s0r, s0i, s1r, s1i);
}

// Sum over the batch rows and the gradients: dW = (Re S0, -Im S0), d log_re = -2 a Re(W S1),
// d log_im = -Im(W S1).
__global__ void dlr_grad_finish(const float4* __restrict__ part, const float* __restrict__ log_re,
                                const float2* __restrict__ W, int B, int H, int N,
                                float* __restrict__ d_log_re, float* __restrict__ d_log_im,
                                float2* __restrict__ dW) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (h, n)
  if (i >= (int64_t)H * N) return;
  const int64_t hn = i;
  double s0r = 0.0, s0i = 0.0, s1r = 0.0, s1i = 0.0;
  for (int b = 0; b < B; ++b) {
    const float4 p = DLR_IN((int64_t)b * H * N + hn, (int64_t)B * H * N)
                         ? part[(int64_t)b * H * N + hn]
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    s0r += p.x;
    s0i += p.y;
    s1r += p.z;
    s1i += p.w;
  }
  const float2 w = W[hn];
  const double ws1r = (double)w.x * s1r - (double)w.y * s1i;
  const double ws1i = (double)w.x * s1i + (double)w.y * s1r;
  dW[hn] = make_float2((float)s0r, (float)-s0i);
  d_log_re[hn] = (float)(-2.0 * (double)log_re[hn] * ws1r);
  d_log_im[hn] = (float)(-ws1i);
}

}  // namespace

size_t grad_workspace_bytes(int64_t B, int64_t H, int64_t N) {
  return sizeof(float4) * (size_t)B * (size_t)H * (size_t)N;
}

cudaError_t launch_dlr_grad_params(const float* u, const float* g, const float* log_re,
                                   const float* log_im, const float* W, int B, int H, int N,
                                   int L, float* d_log_re, float* d_log_im, float* dW, void* ws,
                                   cudaStream_t s) {
  float4* part = static_cast<float4*>(ws);
  const int wpr = (N + 31) / 32;
  const int64_t warps = (int64_t)B * H * wpr;
  const int64_t blocks = (warps + kGradWarps - 1) / kGradWarps;
  dlr_grad_rows<<<(unsigned)blocks, kGradWarps * 32, 0, s>>>(u, g, log_re, log_im, B, H, N, L,
                                                              wpr, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t hn = (int64_t)H * N;
  dlr_grad_finish<<<(unsigned)((hn + 255) / 256), 256, 0, s>>>(
      part, log_re, reinterpret_cast<const float2*>(W), B, H, N, d_log_re, d_log_im,
      reinterpret_cast<float2*>(dW));
  return cudaGetLastError();
}

}  // namespace dlr
