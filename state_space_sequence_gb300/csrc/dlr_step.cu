// dlr_step.cu -- the DLR layer advanced from a carried state: the recurrent ("RNN") mode of a
// diagonal SSM layer, whose hidden state is kept between calls so that a sequence can be fed
// a few samples at a time ("The Annotated S4", part 1 "An SSM Neural Network": the layer's
// RNN mode with its state cache; part 3 "Sampling and Caching": the discretised recurrence is
// computed once per layer, then the cached state is advanced sample by sample). The recurrence
// and read-out are those of "Simplifying and Understanding State Space Models with Diagonal
// Linear RNNs", section 2, Eq. 1 with the Re cast:
//     x_{n,t} = lambda_n x_{n,t-1} + u_t,      y_t = sum_n Re(W_n x_{n,t}),
// with x_{n,-1} the state the caller passes in (zero for a fresh sequence).
//
// dlr_step_tables evaluates lambda_n = exp(-(log_re)^2) e^{i log_im} once per parameter set in
// double precision and keeps it as a float pair (hi + lo, |lo| <= ulp(hi) / 2), with W, in a
// workspace. Each step multiplies by both halves, so the float rounding of lambda does not
// compound coherently over a long stream: over k steps it would move a contribution by about
// k * 6e-8 of itself.
//
// dlr_step_kernel: one warp per (b, h) row, lane l owning states n = l + 32 i (i < kPer) in
// registers. The T samples go in blocks of 32: lane j loads u_{t0+j}, every step takes its
// sample by a shuffle, and each lane keeps its partial read-out of the 32 steps; a
// reduce-scatter over the warp (16 + 8 + 4 + 2 + 1 shuffles) leaves the whole sum of step
// t0 + j in lane j, which stores y coalesced. A block of one sample (decoding one step at a
// time) takes a plain warp sum instead. The state goes back to x at the end.
#include <cuda_runtime.h>

#include "dlr_common.cuh"

#include <cstdint>

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 12;

namespace {

constexpr int kStepWarps = 8;  // rows per block

// lambda as (hi.re, hi.im, lo.re, lo.im) and W, per (h, n)
__global__ void dlr_step_tables(const float* __restrict__ log_re, const float* __restrict__ log_im,
                                const float2* __restrict__ W, int64_t HN, float4* __restrict__ lam,
                                float2* __restrict__ w) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < HN;
       i += (int64_t)gridDim.x * blockDim.x) {
    const double a = log_re[i], th = log_im[i];
    const double mag = exp(-a * a);
    double s, c;
    sincos(th, &s, &c);
    const double re = mag * c, im = mag * s;
    const float rh = (float)re, ih = (float)im;
    lam[i] = make_float4(rh, ih, (float)(re - (double)rh), (float)(im - (double)ih));
    w[i] = W[i];
  }
}

template <int kPer>
__global__ void __launch_bounds__(kStepWarps * 32)
dlr_step_kernel(const float* __restrict__ u, const float4* __restrict__ lam,
                const float2* __restrict__ wt, int64_t rows, int H, int N, int T,
                float2* __restrict__ x, float* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kStepWarps + (threadIdx.x >> 5);
  if (row >= rows) return;  // whole warps only
  const int h = (int)(row % H);
  float4 lm[kPer];
  float2 wv[kPer], xs[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = lane + 32 * i;
    if (n < N) {
      lm[i] = __ldg(&lam[(int64_t)h * N + n]);
      wv[i] = __ldg(&wt[(int64_t)h * N + n]);
      xs[i] = x[row * N + n];
    } else {  // padding states: lambda = W = 0 keep them at zero and out of y
      lm[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      wv[i] = make_float2(0.f, 0.f);
      xs[i] = make_float2(0.f, 0.f);
    }
  }
  const float* ur = u + row * T;
  float* yr = y + row * T;
  // one sample: x = lambda x + u_t and its read-out, summed over the warp
  auto advance = [&](float ut) {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const float xr = xs[i].x, xi = xs[i].y;
      // (hi + lo) * x + u, the lo products first
      const float cr = fmaf(lm[i].z, xr, fmaf(-lm[i].w, xi, ut));
      const float ci = fmaf(lm[i].z, xi, lm[i].w * xr);
      const float nr = fmaf(lm[i].x, xr, fmaf(-lm[i].y, xi, cr));
      const float ni = fmaf(lm[i].x, xi, fmaf(lm[i].y, xr, ci));
      xs[i] = make_float2(nr, ni);
      acc = fmaf(wv[i].x, nr, fmaf(-wv[i].y, ni, acc));
    }
    return acc;
  };
  for (int t0 = 0; t0 < T; t0 += 32) {
    const int nt = min(32, T - t0);  // warp-uniform
    const float uv = lane < nt ? ur[t0 + lane] : 0.f;
    if (nt == 1) {  // a single sample (decoding): a plain warp sum
      float acc = advance(__shfl_sync(0xffffffffu, uv, 0));  // u_t is in lane 0
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0 && DLR_IN(t0, T)) yr[t0] = acc;
      continue;
    }
    float p[32];
    if (nt == 32) {  // a whole block: no per-step branch, so the steps can overlap
#pragma unroll
      for (int j = 0; j < 32; ++j) p[j] = advance(__shfl_sync(0xffffffffu, uv, j));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float ut = __shfl_sync(0xffffffffu, uv, j);
        p[j] = (j < nt) ? advance(ut) : 0.f;
      }
    }
    // reduce-scatter: after the round with offset o, lane l holds in p[0 .. o-1] the partial
    // sums (over the lanes that agree with l above bit log2(o)) of the steps whose bits above
    // log2(o) match l's; at the end p[0] of lane l is the whole sum of step t0 + l
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < o; ++k) {
        const float send = upper ? p[k] : p[k + o];
        const float keep = upper ? p[k + o] : p[k];
        p[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    if (lane < nt && DLR_IN(t0 + lane, T)) yr[t0 + lane] = p[0];
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = lane + 32 * i;
    if (n < N) x[row * N + n] = xs[i];
  }
}

template <int kPer>
cudaError_t launch_step(const float* u, const float4* lam, const float2* w, int64_t rows, int H,
                        int N, int T, float2* x, float* y, cudaStream_t s) {
  const int64_t blocks = (rows + kStepWarps - 1) / kStepWarps;
  dlr_step_kernel<kPer><<<(unsigned)blocks, kStepWarps * 32, 0, s>>>(u, lam, w, rows, H, N, T, x,
                                                                     y);
  return cudaGetLastError();
}

}  // namespace

// Workspace: [H * N] float4 lambda, then [H * N] float2 W.
size_t step_workspace_bytes(int64_t H, int64_t N) {
  return (size_t)H * (size_t)N * (sizeof(float4) + sizeof(float2));
}

cudaError_t launch_step_tables(const float* lr, const float* li, const float* W, int64_t H,
                               int64_t N, void* ws, cudaStream_t s) {
  const int64_t HN = H * N;
  float4* lam = static_cast<float4*>(ws);
  float2* w = reinterpret_cast<float2*>(lam + HN);
  const int64_t blocks = (HN + 255) / 256;
  dlr_step_tables<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(
      lr, li, reinterpret_cast<const float2*>(W), HN, lam, w);
  return cudaGetLastError();
}

// x: [B, H, N] complex (float pairs), read and written; u, y: [B, H, T]. N <= 256.
cudaError_t launch_step(const float* u, int64_t B, int64_t H, int64_t N, int64_t T,
                        const void* ws, float* x, float* y, cudaStream_t s) {
  const float4* lam = static_cast<const float4*>(ws);
  const float2* w = reinterpret_cast<const float2*>(lam + H * N);
  const int64_t rows = B * H;
  float2* xs = reinterpret_cast<float2*>(x);
  if (N <= 32) return launch_step<1>(u, lam, w, rows, (int)H, (int)N, (int)T, xs, y, s);
  if (N <= 64) return launch_step<2>(u, lam, w, rows, (int)H, (int)N, (int)T, xs, y, s);
  if (N <= 128) return launch_step<4>(u, lam, w, rows, (int)H, (int)N, (int)T, xs, y, s);
  return launch_step<8>(u, lam, w, rows, (int)H, (int)N, (int)T, xs, y, s);
}

}  // namespace dlr
