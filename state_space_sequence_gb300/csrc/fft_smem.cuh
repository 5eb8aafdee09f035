// fft_smem.cuh -- complex FFT of a power-of-two size held in one CTA's shared memory.
//
// Stockham auto-sort formulation (natural order in, natural order out, no bit reversal), as
// described for GPUs by Govindaraju et al., "High Performance Discrete Fourier Transforms on
// Graphics Processors" (SC'08): pass s with sub-transform size ns combines R sub-transforms,
//   for j in [0, n/R):  k = j mod ns
//     v_r = x[j + r n/R] * w_{ns R}^{r k}        (r = 0..R-1)
//     v   = DFT_R(v)
//     x'[(j - k) R + k + r ns] = v_r
// Each pass loads every point into registers, synchronises, then stores (in place).
// Shared memory is padded by one element per 16 so that the stride-R stores of the first
// pass and the unit-stride loads are both free of bank conflicts.
#pragma once

#include "dlr_common.cuh"

namespace dlr {
namespace fft {

__host__ __device__ constexpr int padded(int i) { return i + (i >> 4); }
__host__ __device__ constexpr int padded_size(int n) { return n + (n >> 4) + 1; }

// Multiply by -i (forward) or +i (inverse).
template <bool kInv>
__device__ __forceinline__ cf rot90(cf a) {
  return kInv ? cf{-a.im, a.re} : cf{a.im, -a.re};
}

template <bool kInv>
__device__ __forceinline__ void dft2(cf& a, cf& b) {
  cf t = a;
  a = cadd(t, b);
  b = {t.re - b.re, t.im - b.im};
}

// In-place DFT of size 4: x0..x3 -> X0..X3 in natural order.
template <bool kInv>
__device__ __forceinline__ void dft4(cf& x0, cf& x1, cf& x2, cf& x3) {
  cf t0 = cadd(x0, x2), t1 = {x0.re - x2.re, x0.im - x2.im};
  cf t2 = cadd(x1, x3), t3 = rot90<kInv>({x1.re - x3.re, x1.im - x3.im});
  x0 = cadd(t0, t2);
  x2 = {t0.re - t2.re, t0.im - t2.im};
  x1 = cadd(t1, t3);
  x3 = {t1.re - t3.re, t1.im - t3.im};
}

// Mathematical constants cos(pi/8), sin(pi/8), sqrt(2)/2.
constexpr float kC8 = 0.92387953251128675613f;
constexpr float kS8 = 0.38268343236508977173f;
constexpr float kR2 = 0.70710678118654752440f;

// w_16^e for e in {1, 2, 3} (forward sign e^{-2 pi i e/16}; inverse conjugates).
template <bool kInv, int e>
__device__ __forceinline__ cf w16(cf a) {
  constexpr float sg = kInv ? 1.f : -1.f;
  if (e == 1) return cmul(a, {kC8, sg * kS8});
  if (e == 2) return cmul(a, {kR2, sg * kR2});
  if (e == 3) return cmul(a, {kS8, sg * kC8});
  return a;
}

template <int R, bool kInv>
__device__ __forceinline__ void dft(cf (&v)[R]);

template <>
__device__ __forceinline__ void dft<1, false>(cf (&)[1]) {}
template <>
__device__ __forceinline__ void dft<1, true>(cf (&)[1]) {}
template <>
__device__ __forceinline__ void dft<2, false>(cf (&v)[2]) { dft2<false>(v[0], v[1]); }
template <>
__device__ __forceinline__ void dft<2, true>(cf (&v)[2]) { dft2<true>(v[0], v[1]); }
template <>
__device__ __forceinline__ void dft<4, false>(cf (&v)[4]) { dft4<false>(v[0], v[1], v[2], v[3]); }
template <>
__device__ __forceinline__ void dft<4, true>(cf (&v)[4]) { dft4<true>(v[0], v[1], v[2], v[3]); }

// Size 8 = 2 x 4: DFT2 over (r, r+4), twiddle w8^{r q}, DFT4 over r; X[q + 2 s].
template <bool kInv>
__device__ __forceinline__ void dft8_impl(cf (&v)[8]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) dft2<kInv>(v[r], v[r + 4]);
  // v[r] = a[r][0], v[r+4] = a[r][1]; twiddle a[r][1] *= w8^r = w16^{2r}
  v[5] = w16<kInv, 2>(v[5]);
  v[6] = rot90<kInv>(v[6]);
  v[7] = rot90<kInv>(w16<kInv, 2>(v[7]));
  dft4<kInv>(v[0], v[1], v[2], v[3]);  // q = 0 -> X[0], X[2], X[4], X[6]
  dft4<kInv>(v[4], v[5], v[6], v[7]);  // q = 1 -> X[1], X[3], X[5], X[7]
  cf o[8];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    o[2 * s] = v[s];
    o[2 * s + 1] = v[4 + s];
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = o[i];
}
template <>
__device__ __forceinline__ void dft<8, false>(cf (&v)[8]) { dft8_impl<false>(v); }
template <>
__device__ __forceinline__ void dft<8, true>(cf (&v)[8]) { dft8_impl<true>(v); }

// Size 16 = 4 x 4: DFT4 over (r, r+4, r+8, r+12), twiddle w16^{r q}, DFT4 over r; X[q + 4 s].
template <bool kInv>
__device__ __forceinline__ void dft16_impl(cf (&v)[16]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) dft4<kInv>(v[r], v[r + 4], v[r + 8], v[r + 12]);
  // a[r][q] sits in v[r + 4q]; twiddle by w16^{r q}
  v[5] = w16<kInv, 1>(v[5]);
  v[6] = w16<kInv, 2>(v[6]);
  v[7] = w16<kInv, 3>(v[7]);
  v[9] = w16<kInv, 2>(v[9]);
  v[10] = rot90<kInv>(v[10]);
  v[11] = rot90<kInv>(w16<kInv, 2>(v[11]));
  v[13] = w16<kInv, 3>(v[13]);
  v[14] = rot90<kInv>(w16<kInv, 2>(v[14]));
  {  // w16^9 = -w16^1
    cf t = w16<kInv, 1>(v[15]);
    v[15] = {-t.re, -t.im};
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) dft4<kInv>(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  cf o[16];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int s = 0; s < 4; ++s) o[q + 4 * s] = v[4 * q + s];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = o[i];
}
template <>
__device__ __forceinline__ void dft<16, false>(cf (&v)[16]) { dft16_impl<false>(v); }
template <>
__device__ __forceinline__ void dft<16, true>(cf (&v)[16]) { dft16_impl<true>(v); }

// DFT of size 16 whose inputs 8..15 are zero (the zero-padded half of a row): the first
// stage's DFT4s see (x_r, x_{r+4}, 0, 0).
template <bool kInv>
__device__ __forceinline__ void dft16_lowhalf(cf (&v)[16]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const cf a = v[r], b = v[r + 4], rb = rot90<kInv>(v[r + 4]);
    v[r] = cadd(a, b);
    v[r + 8] = {a.re - b.re, a.im - b.im};
    v[r + 4] = cadd(a, rb);
    v[r + 12] = {a.re - rb.re, a.im - rb.im};
  }
  v[5] = w16<kInv, 1>(v[5]);
  v[6] = w16<kInv, 2>(v[6]);
  v[7] = w16<kInv, 3>(v[7]);
  v[9] = w16<kInv, 2>(v[9]);
  v[10] = rot90<kInv>(v[10]);
  v[11] = rot90<kInv>(w16<kInv, 2>(v[11]));
  v[13] = w16<kInv, 3>(v[13]);
  v[14] = rot90<kInv>(w16<kInv, 2>(v[14]));
  {
    cf t = w16<kInv, 1>(v[15]);
    v[15] = {-t.re, -t.im};
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) dft4<kInv>(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  cf o[16];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int s = 0; s < 4; ++s) o[q + 4 * s] = v[4 * q + s];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = o[i];
}

// One Stockham pass of radix R over n = 2^kLog points with kThreads threads.
// tw[m] = exp(-2 pi i m / n), m < n.
template <int kLog, int R, bool kInv, int kThreads>
__device__ __forceinline__ void stockham_pass(float2* buf, int ns, const float2* __restrict__ tw) {
  constexpr int n = 1 << kLog;
  constexpr int NB = n / R;
  constexpr int PER = (NB + kThreads - 1) / kThreads;
  cf v[PER][R];
  int dst[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int j = threadIdx.x + q * kThreads;
    dst[q] = -1;
    if (NB % kThreads == 0 || j < NB) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float2 f = buf[padded(j + r * NB)];
        v[q][r] = {f.x, f.y};
      }
      const int k = j & (ns - 1);
      if (ns > 1) {
        const int e = k * (n / (ns * R));
#pragma unroll
        for (int r = 1; r < R; ++r) {
          float2 w = __ldg(&tw[r * e]);
          v[q][r] = cmul(v[q][r], {w.x, kInv ? -w.y : w.y});
        }
      }
      dft<R, kInv>(v[q]);
      dst[q] = (j - k) * R + k;
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    if (dst[q] >= 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) buf[padded(dst[q] + r * ns)] = make_float2(v[q][r].re, v[q][r].im);
    }
  }
  __syncthreads();
}

// Full FFT of size n = 2^kLog: radix-16 passes, then one radix-8/4/2 pass for the rest.
template <int kLog, bool kInv, int kThreads>
__device__ __forceinline__ void fft(float2* buf, const float2* __restrict__ tw) {
  constexpr int n16 = kLog / 4;
  constexpr int rem = kLog % 4;
  int ns = 1;
  if constexpr (n16 > 0) {
#pragma unroll
    for (int p = 0; p < n16; ++p) {
      stockham_pass<kLog, 16, kInv, kThreads>(buf, ns, tw);
      ns *= 16;
    }
  }
  if constexpr (rem == 3) stockham_pass<kLog, 8, kInv, kThreads>(buf, ns, tw);
  if constexpr (rem == 2) stockham_pass<kLog, 4, kInv, kThreads>(buf, ns, tw);
  if constexpr (rem == 1) stockham_pass<kLog, 2, kInv, kThreads>(buf, ns, tw);
}

}  // namespace fft
}  // namespace dlr
