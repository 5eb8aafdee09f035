// dlr_backward.cu -- gradients of the DLR layer with respect to its parameters
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
// The bidirectional layer (section 2.1: y = DLR1(u) + rev(DLR2(rev(u)))) adds the gradients of
// the causal layer on the reversed rows with the second parameter set: its correlation is c at
// negative lags, c_{-j} = sum_b sum_k g_{b,k} u_{b,k+j}. The DLR-prod cast (section 2.1:
// kappa_j = Re K_j Im K_j) changes only the weights: d kappa_j = Im(K_j dK_j), so with
// w_j = c_j K_j (K complex), S0 = sum_j w_j lambda^j, S1 = sum_j j w_j lambda^j:
//     dW = (Im S0, Re S0),   d a = -2 a Im(W S1),   d theta = Re(W S1).
//
// Two routes compute S0 and S1.
//
// Lag correlation (N >= 16 or the DLR-prod cast, which needs c itself; L <= 65536): c is
// formed first, then the two power sums per state. Rows of up to 8192 take grad_corr below;
// longer rows take the FFT convolution's own spectrum and apply kernels (grad_cross).
//  - grad_corr: one CTA per channel h. For each batch row, z = u + i g (zero-padded to
//    M = 2^lg >= 2L - 1 points, so the circular correlation equals the linear one for lags
//    0 .. L-1) is transformed once; the two real spectra come out as U_f = (Z_f + conj
//    Z_{M-f}) / 2 and G_f = (Z_f - conj Z_{M-f}) / 2i, and A_f += G_f conj(U_f) is summed
//    over the batch for f = 0 .. M/2 (A is Hermitian: c is real). One inverse transform then
//    gives c_j = (1/M) sum_f A_f e^{2 pi i f j / M}.
//  - the power sums: for 64 states or more on the tensor cores (dlr_moments_tc.cu); else
//    grad_moments: one warp per four states of a channel, lanes along the lag (the block's
//    eight warps share one channel and stage its weights in shared memory, 1024 lags at a
//    time, the next tile's loads in flight during the current one): lane t sums
//    c_{32m+t} lambda^{32m} and (32m+t) c_{32m+t} lambda^{32m} over the blocks m, each
//    lambda^{32m} evaluated directly from the parameters (a batch of 32 by the 32 lanes, read
//    back from a per-warp shared table), then multiplies by its own lambda^t; the warp adds
//    the lanes and lane 0 forms the three gradients.
// Per input element this is one complex FFT point per row and a few flops per (state, lag)
// instead of the recurrences' two complex updates per (state, step, row). For the DLR-prod
// cast the complex kernel comes from the generators' complex mode, and the input gradient's
// Re K Im K kernels are formed from it (prod_cast).
//
// Recurrences (fewer states, or longer rows):
// dlr_grad_rows: one thread per (b, h, n) runs both recurrences over the row, in blocks of 32
// steps. A warp holds 32 states of one (b, h) row: lane j loads u_{k0+j} and g_{k0+j}, the steps
// take them by shuffles. Within a block both recurrences start from zero in float (lambda a
// float, at most 32 products deep) and, with t the step within the block, the state carried in
// (X at the block's start, DX = lambda dX/d lambda) adds lambda^{t+1} X to x and
// (t+1) lambda^{t+1} X + lambda^{t+1} DX to D; so the block adds
//     to S0:  sum g x_loc + Gam X,              Gam  = sum_t g_t lambda^{t+1},
//     to S1:  sum g D_loc + Gam DX + Gam1 X,    Gam1 = sum_t (t+1) g_t lambda^{t+1},
// and the carries move on as X <- mu X + x_loc, DX <- 32 mu X + mu DX + D_loc (mu = lambda^32,
// from double). X, DX, S0 and S1 are two-float complex numbers, so no rounding accumulates
// along the row: a plain float recurrence drifts as sqrt(L) rounding errors on unit-circle
// states (2e-5 relative at L = 9000). Each thread leaves its row's (S0, S1) in the workspace;
// dlr_grad_finish adds the B rows of each (h, n) and forms the three gradients.
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "fft_rows.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 2;

cudaError_t launch_twiddle_table(float2* tw, int logn, cudaStream_t s);
// the FFT convolution (dlr_conv.cu), for the correlation of rows longer than 8192
int conv_log2_size(int64_t L);
size_t conv_workspace_bytes(int64_t H, int64_t L);
float2* conv_spectra(void* ws, int64_t L);
cudaError_t launch_dlr_conv_spectrum(const float* K1, const float* K2, int H, int L, void* ws,
                                     cudaStream_t s);
cudaError_t launch_twiddles(int lg, void* ws, cudaStream_t s);
cudaError_t launch_dlr_conv_apply(const float* u, int B, int H, int L, float* y, const void* ws,
                                  cudaStream_t s);

namespace {

using fft::padded;

constexpr int kGradWarps = 4;  // warps per block

__device__ __forceinline__ ff split_double(double v) {
  const float hi = (float)v;
  return {hi, (float)(v - (double)hi)};
}
__device__ __forceinline__ cff cff_of(cf a) { return {{a.re, 0.f}, {a.im, 0.f}}; }
__device__ __forceinline__ cff cff_add(cff a, cff b) {
  return {ff_add(a.re, b.re), ff_add(a.im, b.im)};
}

__global__ void __launch_bounds__(kGradWarps * 32)
    dlr_grad_rows(const float* __restrict__ u, const float* __restrict__ g,
                  const float* __restrict__ log_re, const float* __restrict__ log_im, int B,
                  int H, int N, int L, int warps_per_row, int rev, float4* __restrict__ part) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * kGradWarps + (threadIdx.x >> 5);
  const int64_t row = wid / warps_per_row;  // (b, h)
  if (row >= (int64_t)B * H) return;        // whole warps only
  const int n = (int)(wid - row * warps_per_row) * 32 + lane;
  const int h = (int)(row % H);
  const bool on = n < N;
  // lambda (float) and mu = lambda^32 (two-float), from double
  cf lam = {0.f, 0.f};
  cff mu = {{0.f, 0.f}, {0.f, 0.f}};
  if (on) {
    const double a = log_re[(size_t)h * N + n], th = log_im[(size_t)h * N + n];
    double s, c;
    sincos(th, &s, &c);
    const double mag = exp(-a * a);
    lam = {(float)(mag * c), (float)(mag * s)};
    sincos(32.0 * th, &s, &c);
    const double mag32 = exp(-32.0 * a * a);
    mu = {split_double(mag32 * c), split_double(mag32 * s)};
  }
  const float* ur = u + row * (int64_t)L;
  const float* gr = g + row * (int64_t)L;
  const cff zero = {{0.f, 0.f}, {0.f, 0.f}};
  cff X = zero, DX = zero, S0 = zero, S1 = zero;
#pragma unroll 1
  for (int k0 = 0; k0 < L; k0 += 32) {
    const int k = k0 + lane;
    const int kk = rev ? L - 1 - k : k;  // rev: the reversed row (the second direction)
    const float uk = k < L ? __ldg(ur + kk) : 0.f;
    const float gk = k < L ? __ldg(gr + kk) : 0.f;
    const int steps = min(32, L - k0);
    float xr = 0.f, xi = 0.f, dr = 0.f, di = 0.f;     // block-local x, D
    float rr = lam.re, ri = lam.im;                   // lambda^{t+1}
    float p0r = 0.f, p0i = 0.f, p1r = 0.f, p1i = 0.f;  // sum g x_loc, sum g D_loc
    float g0r = 0.f, g0i = 0.f, g1r = 0.f, g1i = 0.f;  // Gam, Gam1
#pragma unroll 8
    for (int t = 0; t < steps; ++t) {
      const float ut = __shfl_sync(0xffffffffu, uk, t);
      const float gt = __shfl_sync(0xffffffffu, gk, t);
      // D_loc <- lambda (D_loc + x_loc), then x_loc <- lambda x_loc + u_t
      const float er = dr + xr, ei = di + xi;
      dr = fmaf(lam.re, er, -lam.im * ei);
      di = fmaf(lam.re, ei, lam.im * er);
      const float nr = fmaf(lam.re, xr, fmaf(-lam.im, xi, ut));
      const float ni = fmaf(lam.re, xi, lam.im * xr);
      xr = nr;
      xi = ni;
      p0r = fmaf(gt, xr, p0r);
      p0i = fmaf(gt, xi, p0i);
      p1r = fmaf(gt, dr, p1r);
      p1i = fmaf(gt, di, p1i);
      const float gw = (float)(t + 1) * gt;
      g0r = fmaf(gt, rr, g0r);
      g0i = fmaf(gt, ri, g0i);
      g1r = fmaf(gw, rr, g1r);
      g1i = fmaf(gw, ri, g1i);
      const float qr = fmaf(lam.re, rr, -lam.im * ri);
      ri = fmaf(lam.re, ri, lam.im * rr);
      rr = qr;
    }
    const cff gam = cff_of({g0r, g0i}), gam1 = cff_of({g1r, g1i});
    S0 = cff_fma(gam, X, cff_add(S0, cff_of({p0r, p0i})));
    S1 = cff_fma(gam1, X, cff_fma(gam, DX, cff_add(S1, cff_of({p1r, p1i}))));
    if (steps == 32) {
      // DX <- 32 mu X + mu DX + D_loc (32 mu X exact: a power of two), X <- mu X + x_loc
      const cff muX = cff_fma(mu, X, zero);
      const cff mu32X = {{32.f * muX.re.hi, 32.f * muX.re.lo}, {32.f * muX.im.hi, 32.f * muX.im.lo}};
      DX = cff_fma(mu, DX, cff_add(mu32X, cff_of({dr, di})));
      X = cff_add(muX, cff_of({xr, xi}));
    }
  }
  if (on && DLR_IN(row * (int64_t)N + n, (int64_t)B * H * N))
    part[row * (int64_t)N + n] = make_float4(S0.re.hi + S0.re.lo, S0.im.hi + S0.im.lo,
                                             S1.re.hi + S1.re.lo, S1.im.hi + S1.im.lo);
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

// ---- lag correlation route ----

// One CTA per channel h: c[h, j] = sum_b sum_k g_{b,h,k} u_{b,h,k-j}, j < L, by transforms of
// M = 2^kLog >= 2L - 1 points. Shared memory: the transform buffer (padded) and A_f, f <= M/2.
template <int kLog>
__global__ void __launch_bounds__(fftr::Plan<kLog>::T, kLog <= 13 ? 2 : 1)
    grad_corr(const float* __restrict__ u, const float* __restrict__ g, int B, int H, int L,
              const float2* __restrict__ tw, float* __restrict__ c, float* __restrict__ c2) {
  using P = fftr::Plan<kLog>;
  constexpr int M = P::n, T = P::T, kHalf = M / 2;
  constexpr int PER = (M + T - 1) / T;
  constexpr bool kDup = P::R0 == 2 && P::n16 > 0;  // the first pass is radix 2 (see below)
  extern __shared__ float2 smem[];
  float2* buf = smem;
  float2* acc = smem + P::buf_elems;
  const int tid = threadIdx.x;
  const int h = blockIdx.x;
  for (int f = tid; f <= kHalf; f += T)
    if (DLR_IN(f, kHalf + 1)) acc[f] = make_float2(0.f, 0.f);
#pragma unroll 1
  for (int b = 0; b < B; ++b) {
    const float* ur = u + ((size_t)b * H + h) * (size_t)L;
    const float* gr = g + ((size_t)b * H + h) * (size_t)L;
    if constexpr (kDup) {
      // a radix-2 first pass over z (zero above M/2 > L - 1) leaves z_m at 2m and 2m + 1:
      // written here directly, and the transform starts at its second pass
      constexpr int PH = (kHalf + T - 1) / T;
      float2 z[PH];
#pragma unroll
      for (int q = 0; q < PH; ++q) {
        const int m = tid + q * T;
        z[q] = m < L ? make_float2(__ldg(ur + m), __ldg(gr + m)) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < PH; ++q) {
        const int m = tid + q * T;
        if (m < kHalf && DLR_IN(padded(2 * m) + 1, P::buf_elems)) {
          buf[padded(2 * m)] = z[q];  // 2m and 2m + 1 share a padding group (2m even)
          buf[padded(2 * m) + 1] = z[q];
        }
      }
      __syncthreads();
      fftr::local_fft<kLog, false, true>(buf, tw);  // ends with a barrier
    } else {
      // every load of the row before the first store
      float2 z[PER];
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int m = tid + q * T;
        z[q] = m < L ? make_float2(__ldg(ur + m), __ldg(gr + m)) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int m = tid + q * T;
        if (m < M && DLR_IN(padded(m), P::buf_elems)) buf[padded(m)] = z[q];
      }
      __syncthreads();
      fftr::local_fft<kLog, false>(buf, tw);  // ends with a barrier
    }
    for (int f = tid; f <= kHalf; f += T) {
      const int fm = (M - f) & (M - 1);
      if (!DLR_IN(padded(f), P::buf_elems) || !DLR_IN(padded(fm), P::buf_elems) ||
          !DLR_IN(f, kHalf + 1))
        continue;
      const float2 za = buf[padded(f)], zb = buf[padded(fm)];
      // U_f = (Z_f + conj Z_{M-f}) / 2, G_f = (Z_f - conj Z_{M-f}) / 2i
      const float ur_ = 0.5f * (za.x + zb.x), ui = 0.5f * (za.y - zb.y);
      const float gr_ = 0.5f * (za.y + zb.y), gi = 0.5f * (zb.x - za.x);
      float2 a = acc[f];
      a.x = fmaf(gr_, ur_, fmaf(gi, ui, a.x));  // Re G conj(U)
      a.y = fmaf(gi, ur_, fmaf(-gr_, ui, a.y));  // Im G conj(U)
      acc[f] = a;
    }
    __syncthreads();  // the next row overwrites the buffer
  }
  // the Hermitian spectrum of the real correlation, then its inverse transform
  for (int f = tid; f <= kHalf; f += T) {
    if (!DLR_IN(f, kHalf + 1) || !DLR_IN(padded(f), P::buf_elems)) continue;
    const float2 a = acc[f];
    buf[padded(f)] = a;
    if (f > 0 && f < kHalf && DLR_IN(padded(M - f), P::buf_elems))
      buf[padded(M - f)] = make_float2(a.x, -a.y);
  }
  __syncthreads();
  fftr::local_fft<kLog, true>(buf, tw);
  const float inv = 1.0f / (float)M;
  float* ch = c + (size_t)h * (size_t)L;
  for (int j = tid; j < L; j += T)
    if (DLR_IN(padded(j), P::buf_elems)) ch[j] = buf[padded(j)].x * inv;
  if (c2) {  // the negative lags: c2_j = sum_b sum_k g_{b,k} u_{b,k+j}, at M - j (j > 0)
    float* c2h = c2 + (size_t)h * (size_t)L;
    for (int j = tid; j < L; j += T) {
      const int m = (M - j) & (M - 1);
      if (DLR_IN(padded(m), P::buf_elems)) c2h[j] = buf[padded(m)].x * inv;
    }
  }
}

// ---- lag correlation of rows longer than 8192, through the FFT convolution's kernels ----
// The convolution's spectrum kernel, run on the rows of u and of g as if they were kernel
// columns, stores their zero-padded spectra as X/(4n) (n + 1 bins of the 2n-point real
// transform); A = (4n) sum_b G conj(U) is then stored as the spectrum of the real column c
// (c_j at j, c_{-j} at 2n - j), and the convolution's apply kernel on an impulse returns that
// column's first L entries: c. With conj(A) it returns the negative lags.
__global__ void grad_cross(const float2* __restrict__ su, const float2* __restrict__ sg, int B,
                           int H, int nb, float scale, float2* __restrict__ a) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // h * nb + f
  if (i >= (int64_t)H * nb) return;
  const int64_t h = i / nb, f = i - h * nb;
  float ar = 0.f, ai = 0.f;
  for (int b = 0; b < B; ++b) {
    const int64_t o = ((int64_t)b * H + h) * nb + f;
    const float2 x = su[o], y = sg[o];
    ar = fmaf(y.x, x.x, fmaf(y.y, x.y, ar));   // Re G conj(U)
    ai = fmaf(y.y, x.x, fmaf(-y.x, x.y, ai));  // Im G conj(U)
  }
  if (DLR_IN(i, (int64_t)H * nb)) a[i] = make_float2(ar * scale, ai * scale);
}
// kappa_j = Re K_j Im K_j from the complex kernel (the DLR-prod cast, as the generators form it)
__global__ void prod_cast(const float2* __restrict__ K, float* __restrict__ kap, int64_t count) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) {
    const float2 k = K[i];
    kap[i] = k.x * k.y;
  }
}
__global__ void conj_spectra(float2* __restrict__ a, int64_t count) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) a[i].y = -a[i].y;
}
__global__ void impulse_rows(float* __restrict__ d, int H, int L) {  // d zeroed before
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < H && DLR_IN((int64_t)h * L, (int64_t)H * L)) d[(size_t)h * L] = 1.f;
}

constexpr int kMomWarps = 8;   // warps per block
constexpr int kMomStates = 4;  // states per warp

// S0 = sum_j w_j lambda^j and S1 = sum_j j w_j lambda^j for kMomStates states of channel h per
// warp, then the gradients of those states. Re cast: w_j = c_j, dW = (Re S0, -Im S0),
// d log_re = -2a Re(W S1), d log_im = -Im(W S1). DLR-prod cast (kappa_j = Re K_j Im K_j, so
// d kappa_j = Im(K_j dK_j)): w_j = c_j K_j with the complex kernel Kc, dW = (Im S0, Re S0),
// d log_re = -2a Im(W S1), d log_im = Re(W S1).
constexpr int kLagTile = 1024;  // lags staged in shared memory at a time (32 blocks of 32)

template <bool kProd>
__global__ void __launch_bounds__(kMomWarps * 32)
    grad_moments(const float* __restrict__ c, const float2* __restrict__ Kc,
                 const float* __restrict__ log_re, const float* __restrict__ log_im,
                 const float2* __restrict__ W, int H, int N, int L, int blocks_per_h,
                 float* __restrict__ d_log_re, float* __restrict__ d_log_im,
                 float2* __restrict__ dW) {
  // the weights of a lag: (w_j, j w_j), real (Re cast: float2) or complex (DLR-prod: float4)
  using WT = typename std::conditional<kProd, float4, float2>::type;
  constexpr int kPer = kLagTile / (kMomWarps * 32);  // lags a thread stages per tile
  __shared__ WT sw[2][kLagTile];
  __shared__ float2 spw[kMomWarps][kMomStates][32];  // each warp's lambda^{32 m} of a tile
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x / blocks_per_h;  // every warp of the block takes channel h
  const int n0 = ((blockIdx.x - h * blocks_per_h) * kMomWarps + warp) * kMomStates;
  const bool active = n0 < N;  // idle warps still stage weights and meet at the barriers
  const float* ch = c + (size_t)h * (size_t)L;
  const float2* kh = kProd ? Kc + (size_t)h * (size_t)L : nullptr;
  lam_param p[kMomStates];
#pragma unroll
  for (int s = 0; s < kMomStates; ++s) {
    const int n = min(n0 + s, N - 1);
    p[s] = make_lam_param(log_re[(size_t)h * N + n], log_im[(size_t)h * N + n]);
  }
  cf a0[kMomStates], a1[kMomStates];
#pragma unroll
  for (int s = 0; s < kMomStates; ++s) a0[s] = a1[s] = {0.f, 0.f};
  WT reg[kPer];
  auto load_tile = [&](int t) {  // the next tile's weights into registers (loads in flight)
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int j = t * kLagTile + q * (kMomWarps * 32) + tid;
      const float cj = j < L ? __ldg(ch + j) : 0.f;
      if constexpr (!kProd) {
        reg[q] = make_float2(cj, (float)j * cj);
      } else {
        const float2 kj = j < L ? __ldg(kh + j) : make_float2(0.f, 0.f);
        const float tr = cj * kj.x, ti = cj * kj.y;
        reg[q] = make_float4(tr, ti, (float)j * tr, (float)j * ti);
      }
    }
  };
  auto store_tile = [&](int buf) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) sw[buf][q * (kMomWarps * 32) + tid] = reg[q];
  };
  const int ntiles = (L + kLagTile - 1) / kLagTile;
  load_tile(0);
  store_tile(0);
  __syncthreads();
#pragma unroll 1
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles) load_tile(t + 1);
    if (active) {
      // lambda^{32 m} for the tile's block m = 32 t + lane, into the warp's table (read back
      // as one broadcast per state and block)
#pragma unroll
      for (int s = 0; s < kMomStates; ++s) {
        const cf pw = lam_pow(p[s], 32 * (32 * t + lane));
        spw[warp][s][lane] = make_float2(pw.re, pw.im);
      }
      __syncwarp();
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const WT wv = sw[buf][32 * i + lane];  // lag j = 1024 t + 32 i + lane
#pragma unroll
        for (int s = 0; s < kMomStates; ++s) {
          const float2 pf = spw[warp][s][i];
          const cf w = {pf.x, pf.y};
          if constexpr (!kProd) {
            a0[s].re = fmaf(wv.x, w.re, a0[s].re);
            a0[s].im = fmaf(wv.x, w.im, a0[s].im);
            a1[s].re = fmaf(wv.y, w.re, a1[s].re);
            a1[s].im = fmaf(wv.y, w.im, a1[s].im);
          } else {
            a0[s] = cfma({wv.x, wv.y}, w, a0[s]);
            a1[s] = cfma({wv.z, wv.w}, w, a1[s]);
          }
        }
      }
      __syncwarp();  // the table is rewritten at the next tile
    }
    if (t + 1 < ntiles) store_tile(buf ^ 1);  // that buffer was last read before the barrier
    __syncthreads();
  }
  if (!active) return;
#pragma unroll
  for (int s = 0; s < kMomStates; ++s) {
    const cf lt = lam_pow(p[s], lane);
    cf s0 = cmul(a0[s], lt), s1 = cmul(a1[s], lt);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s0.re += __shfl_xor_sync(0xffffffffu, s0.re, o);
      s0.im += __shfl_xor_sync(0xffffffffu, s0.im, o);
      s1.re += __shfl_xor_sync(0xffffffffu, s1.re, o);
      s1.im += __shfl_xor_sync(0xffffffffu, s1.im, o);
    }
    const int n = n0 + s;
    if (lane == 0 && n < N) {
      const size_t hn = (size_t)h * N + n;
      const float2 w = W[hn];
      const double ws1r = (double)w.x * s1.re - (double)w.y * s1.im;
      const double ws1i = (double)w.x * s1.im + (double)w.y * s1.re;
      if constexpr (!kProd) {
        dW[hn] = make_float2(s0.re, -s0.im);
        d_log_re[hn] = (float)(-2.0 * (double)log_re[hn] * ws1r);
        d_log_im[hn] = (float)(-ws1i);
      } else {
        dW[hn] = make_float2(s0.im, s0.re);
        d_log_re[hn] = (float)(-2.0 * (double)log_re[hn] * ws1i);
        d_log_im[hn] = (float)ws1r;
      }
    }
  }
}

template <int kLog>
cudaError_t launch_corr(const float* u, const float* g, int B, int H, int L, const float2* tw,
                        float* c, float* c2, cudaStream_t s) {
  using P = fftr::Plan<kLog>;
  const size_t smem = (P::buf_elems + (size_t)(P::n / 2 + 1)) * sizeof(float2);
  cudaError_t e = max_smem_once<grad_corr<kLog>>(smem);
  if (e != cudaSuccess) return e;
  grad_corr<kLog><<<(unsigned)H, P::T, smem, s>>>(u, g, B, H, L, tw, c, c2);
  return cudaGetLastError();
}

// M = 2^lg >= 2L - 1 points
int corr_log2_size(int64_t L) {
  int lg = 0;
  while ((int64_t(1) << lg) < 2 * L - 1) ++lg;
  return lg;
}

// Correlation routes: one CTA per channel (L <= 8192) or through the convolution's kernels
// (L <= 65536); otherwise the blocked recurrences (Re cast only).
bool corr_route(int64_t N, int64_t L, bool prod) { return (prod || N >= 16) && L <= 65536; }
bool corr_long(int64_t L) { return L > 8192; }

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Workspace of the gradients. Correlation route: the M-point twiddle table, c [H, L], with a
// second direction the negative lags c2 [H, L], with the DLR-prod cast the complex kernel of
// each direction [H, L] float2. Recurrence route: the per-row sums [B, H, N] float4, reused
// by the second direction.
struct GradWs {
  float2* tw;
  float *c, *c2;
  float2 *k1, *k2;
  float4* part;
  void *su, *sg, *sa;  // long rows: convolution workspaces of the u rows, g rows, channels
  float* imp;          // long rows: the impulse rows [H, L]
};
GradWs carve_grads(void* ws, int64_t B, int64_t H, int64_t N, int64_t L, bool bidir, bool prod,
                   size_t* total) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  GradWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* q = p ? p + off : nullptr;
    off += align256(bytes);
    return q;
  };
  if (corr_route(N, L, prod)) {
    const size_t hl = (size_t)H * (size_t)L;
    if (corr_long(L)) {
      w.su = take(conv_workspace_bytes(B * H, L));
      w.sg = take(conv_workspace_bytes(B * H, L));
      w.sa = take(conv_workspace_bytes(H, L));
      w.imp = reinterpret_cast<float*>(take(sizeof(float) * hl));
    } else {
      w.tw = reinterpret_cast<float2*>(take(sizeof(float2) << corr_log2_size(L)));
    }
    w.c = reinterpret_cast<float*>(take(sizeof(float) * hl));
    if (bidir) w.c2 = reinterpret_cast<float*>(take(sizeof(float) * hl));
    if (prod) w.k1 = reinterpret_cast<float2*>(take(sizeof(float2) * hl));
    if (prod && bidir) w.k2 = reinterpret_cast<float2*>(take(sizeof(float2) * hl));
  } else {
    w.part = reinterpret_cast<float4*>(take(sizeof(float4) * (size_t)B * H * N));
  }
  if (total) *total = off;
  return w;
}

}  // namespace
cudaError_t launch_moments_tc(const float* c, const float2* Kc, bool prod, const float* log_re,
                              const float* log_im, const float* W, int H, int N, int L,
                              float* d_log_re, float* d_log_im, float* dW, int* status,
                              cudaStream_t s);
namespace {

// The moments of one parameter set from its weights (c, and the complex kernel for DLR-prod):
// on the tensor cores (dlr_moments_tc.cu) for 64 states or more, else on FFMA.
cudaError_t launch_moments(const float* c, const float2* Kc, bool prod, const float* log_re,
                           const float* log_im, const float* W, int H, int N, int L,
                           float* d_log_re, float* d_log_im, float* dW, int* status,
                           cudaStream_t s) {
  if (N >= 64)
    return launch_moments_tc(c, Kc, prod, log_re, log_im, W, H, N, L, d_log_re, d_log_im, dW,
                             status, s);
  const int bph = (N + kMomWarps * kMomStates - 1) / (kMomWarps * kMomStates);
  const unsigned grid = (unsigned)((int64_t)H * bph);
  const float2* Wc = reinterpret_cast<const float2*>(W);
  float2* dWc = reinterpret_cast<float2*>(dW);
  if (prod)
    grad_moments<true><<<grid, kMomWarps * 32, 0, s>>>(c, Kc, log_re, log_im, Wc, H, N, L, bph,
                                                        d_log_re, d_log_im, dWc);
  else
    grad_moments<false><<<grid, kMomWarps * 32, 0, s>>>(c, Kc, log_re, log_im, Wc, H, N, L, bph,
                                                         d_log_re, d_log_im, dWc);
  return cudaGetLastError();
}

// The recurrence route for one parameter set (rev: on the reversed rows).
cudaError_t launch_rows(const float* u, const float* g, const float* log_re, const float* log_im,
                        const float* W, int B, int H, int N, int L, bool rev, float4* part,
                        float* d_log_re, float* d_log_im, float* dW, cudaStream_t s) {
  const int wpr = (N + 31) / 32;
  const int64_t warps = (int64_t)B * H * wpr;
  const int64_t blocks = (warps + kGradWarps - 1) / kGradWarps;
  dlr_grad_rows<<<(unsigned)blocks, kGradWarps * 32, 0, s>>>(u, g, log_re, log_im, B, H, N, L,
                                                              wpr, rev ? 1 : 0, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t hn = (int64_t)H * N;
  dlr_grad_finish<<<(unsigned)((hn + 255) / 256), 256, 0, s>>>(
      part, log_re, reinterpret_cast<const float2*>(W), B, H, N, d_log_re, d_log_im,
      reinterpret_cast<float2*>(dW));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dlr_kernel_complex(const float* log_re, const float* log_im, const float* W,
                                      int H, int N, int L, float2* K, int* status,
                                      cudaStream_t s);

size_t grads_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t L, bool bidir, bool prod) {
  size_t total = 0;
  carve_grads(nullptr, B, H, N, L, bidir, prod, &total);
  return total;
}

size_t grad_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t L) {
  return grads_workspace_bytes(B, H, N, L, false, false);
}

// The parameter gradients of the causal (lr2 == nullptr) or bidirectional layer in either
// cast. The second direction is the causal layer on the reversed rows with the second
// parameter set: its correlation is c at negative lags, its recurrences run on reversed rows.
// The DLR-prod cast takes the correlation route (L <= 8192).
cudaError_t launch_dlr_grads(const float* u, const float* g, const float* lr1, const float* li1,
                             const float* W1, const float* lr2, const float* li2,
                             const float* W2, int B, int H, int N, int L, bool prod,
                             float* dr1, float* di1, float* dW1, float* dr2, float* di2,
                             float* dW2, void* ws, int* status, cudaStream_t s, float* kap1,
                             float* kap2) {
  const bool bidir = lr2 != nullptr;
  const GradWs w = carve_grads(ws, B, H, N, L, bidir, prod, nullptr);
  cudaError_t e;
  if (!corr_route(N, L, prod)) {
    if ((e = launch_rows(u, g, lr1, li1, W1, B, H, N, L, false, w.part, dr1, di1, dW1, s)) !=
        cudaSuccess)
      return e;
    if (bidir)
      return launch_rows(u, g, lr2, li2, W2, B, H, N, L, true, w.part, dr2, di2, dW2, s);
    return cudaSuccess;
  }
  if (L > 65536) return cudaErrorInvalidValue;
  if (corr_long(L)) {
    const int n = 1 << conv_log2_size(L);
    const int nb = n + 1;
    if ((e = launch_dlr_conv_spectrum(u, nullptr, B * H, L, w.su, s)) != cudaSuccess) return e;
    if ((e = launch_dlr_conv_spectrum(g, nullptr, B * H, L, w.sg, s)) != cudaSuccess) return e;
    float2* a = conv_spectra(w.sa, L);
    const int64_t bins = (int64_t)H * nb;
    grad_cross<<<(unsigned)((bins + 255) / 256), 256, 0, s>>>(
        conv_spectra(w.su, L), conv_spectra(w.sg, L), B, H, nb, 4.0f * (float)n, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_twiddles(conv_log2_size(L), w.sa, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(w.imp, 0, sizeof(float) * (size_t)H * L, s)) != cudaSuccess)
      return e;
    impulse_rows<<<(H + 255) / 256, 256, 0, s>>>(w.imp, H, L);
    if ((e = launch_dlr_conv_apply(w.imp, 1, H, L, w.c, w.sa, s)) != cudaSuccess) return e;
    if (bidir) {
      conj_spectra<<<(unsigned)((bins + 255) / 256), 256, 0, s>>>(a, bins);
      if ((e = launch_dlr_conv_apply(w.imp, 1, H, L, w.c2, w.sa, s)) != cudaSuccess) return e;
    }
  } else {
    const int lg = corr_log2_size(L);
    if ((e = launch_twiddle_table(w.tw, lg, s)) != cudaSuccess) return e;
    switch (lg) {
#define CORR_CASE(G) \
  case G: e = launch_corr<G>(u, g, B, H, L, w.tw, w.c, w.c2, s); break;
      CORR_CASE(0) CORR_CASE(1) CORR_CASE(2) CORR_CASE(3) CORR_CASE(4) CORR_CASE(5)
      CORR_CASE(6) CORR_CASE(7) CORR_CASE(8) CORR_CASE(9) CORR_CASE(10) CORR_CASE(11)
      CORR_CASE(12) CORR_CASE(13) CORR_CASE(14)
#undef CORR_CASE
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  if (prod) {
    if ((e = launch_dlr_kernel_complex(lr1, li1, W1, H, N, L, w.k1, status, s)) != cudaSuccess)
      return e;
    if (bidir &&
        (e = launch_dlr_kernel_complex(lr2, li2, W2, H, N, L, w.k2, status, s)) != cudaSuccess)
      return e;
    // the cast kernels of the input gradient's convolution, when asked for
    const int64_t hl = (int64_t)H * L;
    const unsigned gb = (unsigned)((hl + 255) / 256);
    if (kap1) prod_cast<<<gb, 256, 0, s>>>(w.k1, kap1, hl);
    if (kap2 && bidir) prod_cast<<<gb, 256, 0, s>>>(w.k2, kap2, hl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = launch_moments(w.c, w.k1, prod, lr1, li1, W1, H, N, L, dr1, di1, dW1, status, s)) !=
      cudaSuccess)
    return e;
  if (bidir)
    return launch_moments(w.c2, w.k2, prod, lr2, li2, W2, H, N, L, dr2, di2, dW2, status, s);
  return cudaSuccess;
}

cudaError_t launch_dlr_grad_params(const float* u, const float* g, const float* log_re,
                                   const float* log_im, const float* W, int B, int H, int N,
                                   int L, float* d_log_re, float* d_log_im, float* dW, void* ws,
                                   int* status, cudaStream_t s) {
  return launch_dlr_grads(u, g, log_re, log_im, W, nullptr, nullptr, nullptr, B, H, N, L, false,
                          d_log_re, d_log_im, dW, nullptr, nullptr, nullptr, ws, status, s,
                          nullptr, nullptr);
}

}  // namespace dlr
