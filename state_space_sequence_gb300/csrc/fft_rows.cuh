// fft_rows.cuh -- register-resident Stockham passes for the per-row FFT convolution.
//
// Same Stockham auto-sort recurrence as fft_smem.cuh, arranged so that data stays in
// registers wherever the layouts allow:
//   * the first forward pass reads its inputs x[j + r n/R0] straight from global memory,
//   * every later pass loads from one shared buffer and stores into the other (double
//     buffering: one barrier per pass; a single buffer and two barriers for large n),
//   * the spectral step reads each point k and its mirror n - k from the forward output and
//     produces, in registers, exactly the inputs of the first inverse pass,
//   * the last inverse pass writes its outputs straight to global memory.
// Plan: n = R0 * 16^p with R0 in {2, 4, 8, 16}; twiddles only in the radix-16 passes.
#pragma once

#include "fft_smem.cuh"

namespace dlr {
namespace fftr {

constexpr int kSiteFileRows = 21;  // bounds-checked build: this header's site number

using fft::padded;
using fft::padded_size;

template <int kLog>
struct Plan {
  static constexpr int n = 1 << kLog;
  static constexpr int rem = kLog % 4;
  static constexpr int R0 = kLog == 0 ? 1 : (rem == 0 ? 16 : (1 << rem));
  static constexpr int n16 = kLog == 0 ? 0 : (rem == 0 ? kLog / 4 - 1 : kLog / 4);
  static constexpr int T = (n / 16) < 32 ? 32 : ((n / 16) > 512 ? 512 : n / 16);
  static constexpr int NB0 = n / R0;
  static constexpr int PER0 = (NB0 + T - 1) / T;
  static constexpr int NB16 = n / 16;
  static constexpr int PER16 = n16 > 0 ? (NB16 + T - 1) / T : 1;
  static constexpr size_t buf_elems = padded_size(n);
  static constexpr bool kDouble = 2 * buf_elems * sizeof(float2) <= 72 * 1024;
  static constexpr size_t smem = (kDouble ? 2 : 1) * buf_elems * sizeof(float2);
};

// e^{-i pi r / 16}, r < 16 (cosines and sines of multiples of pi/16)
__device__ __forceinline__ cf half16(int r) {
  constexpr float c[9] = {1.0f, 0.98078528040323044913f, 0.92387953251128675613f,
                          0.83146961230254523708f, 0.70710678118654752440f,
                          0.55557023301960222474f, 0.38268343236508977173f,
                          0.19509032201612826785f, 0.0f};
  // r < 8: (cos, -sin) = (c[r], -c[8 - r]); r >= 8: multiply by e^{-i pi/2} = -i
  if (r < 8) return {c[r], -c[8 - r]};
  const int q = r - 8;
  return {-c[8 - q], -c[q]};
}

// v[r] *= w^{r k}, w = exp(-+2 pi i / (ns*16)); tw[m] = exp(-2 pi i m / n).
// w^1, w^2, w^4, w^8 come from the table; the others are products of at most three of them.
template <bool kInv>
__device__ __forceinline__ void twiddle16(cf (&v)[16], int e, const float2* __restrict__ tw) {
  auto ld = [&](int i) {
    float2 f = __ldg(&tw[i]);
    return cf{f.x, kInv ? -f.y : f.y};
  };
  cf w[16];
  w[1] = ld(e);
  w[2] = ld(2 * e);
  w[4] = ld(4 * e);
  w[8] = ld(8 * e);
  w[3] = cmul(w[1], w[2]);
  w[5] = cmul(w[1], w[4]);
  w[6] = cmul(w[2], w[4]);
  w[7] = cmul(w[3], w[4]);
  w[9] = cmul(w[1], w[8]);
  w[10] = cmul(w[2], w[8]);
  w[11] = cmul(w[3], w[8]);
  w[12] = cmul(w[4], w[8]);
  w[13] = cmul(w[5], w[8]);
  w[14] = cmul(w[6], w[8]);
  w[15] = cmul(w[7], w[8]);
#pragma unroll
  for (int r = 1; r < 16; ++r) v[r] = cmul(v[r], w[r]);
}

// One radix-16 pass reading `src` (natural Stockham input positions j + r n/16) and either
// storing to `dst` at the Stockham output positions or leaving the outputs in `v`.
template <int kLog, bool kInv>
__device__ __forceinline__ void pass16_load_compute(const float2* src, int ns,
                                                     const float2* __restrict__ tw,
                                                     cf (&v)[Plan<kLog>::PER16][16]) {
  using P = Plan<kLog>;
#pragma unroll
  for (int q = 0; q < P::PER16; ++q) {
    const int j = threadIdx.x + q * P::T;
    if (P::NB16 % P::T == 0 || j < P::NB16) {
      if constexpr (P::NB16 % 16 == 0) {
        const float2* s0 = src + padded(j);  // padded(j + r NB) = padded(j) + r * 17 NB / 16
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int e = padded(j) + r * (P::NB16 + P::NB16 / 16);
          float2 f = DLR_IN_FILE(e, P::buf_elems, kSiteFileRows) ? s0[r * (P::NB16 + P::NB16 / 16)]
                                                                 : make_float2(0.f, 0.f);
          v[q][r] = {f.x, f.y};
        }
      } else {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int e = padded(j + r * P::NB16);
          float2 f = DLR_IN_FILE(e, P::buf_elems, kSiteFileRows) ? src[e] : make_float2(0.f, 0.f);
          v[q][r] = {f.x, f.y};
        }
      }
      const int k = j & (ns - 1);
      if (ns > 1) twiddle16<kInv>(v[q], k * (P::n / (ns * 16)), tw);
      fft::dft<16, kInv>(v[q]);
    }
  }
}

template <int kLog>
__device__ __forceinline__ void pass16_store(float2* dst, int ns,
                                             const cf (&v)[Plan<kLog>::PER16][16]) {
  using P = Plan<kLog>;
#pragma unroll
  for (int q = 0; q < P::PER16; ++q) {
    const int j = threadIdx.x + q * P::T;
    if (P::NB16 % P::T == 0 || j < P::NB16) {
      const int k = j & (ns - 1);
      const int d = (j - k) * 16 + k;
      if (ns >= 16) {  // ns is a multiple of 16: padded(d + r ns) = padded(d) + r * 17 ns / 16
        float2* d0 = dst + padded(d);
        const int st = ns + (ns >> 4);
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (DLR_IN_FILE(padded(d) + r * st, P::buf_elems, kSiteFileRows))
            d0[r * st] = make_float2(v[q][r].re, v[q][r].im);
      } else {
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (DLR_IN_FILE(padded(d + r * ns), P::buf_elems, kSiteFileRows))
            dst[padded(d + r * ns)] = make_float2(v[q][r].re, v[q][r].im);
      }
    }
  }
}

template <int kLog>
__device__ __forceinline__ void pass0_store(float2* dst, const cf (&a)[Plan<kLog>::PER0][Plan<kLog>::R0]) {
  using P = Plan<kLog>;
#pragma unroll
  for (int q = 0; q < P::PER0; ++q) {
    const int j = threadIdx.x + q * P::T;
    if (P::NB0 % P::T == 0 || j < P::NB0) {
      // R0 divides 16, so padded(j R0 + r) = padded(j R0) + r for r < R0
      float2* d0 = dst + padded(j * P::R0);
#pragma unroll
      for (int r = 0; r < P::R0; ++r)
        if (DLR_IN_FILE(padded(j * P::R0) + r, P::buf_elems, kSiteFileRows))
          d0[r] = make_float2(a[q][r].re, a[q][r].im);
    }
  }
}

// Stockham FFT of n = 2^kLog points held in `buf` (padded layout; natural order in and out),
// in place: every pass loads all of a thread's points, synchronises, then stores. Forward
// (e^{-2 pi i jk/n}) or, with kInv, the unnormalised inverse; tw is the n-point table above.
// Every thread of the CTA (Plan<kLog>::T of them) must call it. kAfterPass0: the caller has
// already written the first pass's output (for a radix-2 first pass over an input whose upper
// half is zero that is each point x_j at positions 2j and 2j + 1).
template <int kLog, bool kInv, bool kAfterPass0 = false>
__device__ __forceinline__ void local_fft(float2* buf, const float2* __restrict__ tw) {
  using P = Plan<kLog>;
  if constexpr (!kAfterPass0) {
    cf a[P::PER0][P::R0];
#pragma unroll
    for (int q = 0; q < P::PER0; ++q) {
      const int j = threadIdx.x + q * P::T;
      if (P::NB0 % P::T == 0 || j < P::NB0) {
#pragma unroll
        for (int r = 0; r < P::R0; ++r) {
          const float2 f = DLR_IN_FILE(padded(j + r * P::NB0), P::buf_elems, kSiteFileRows)
                               ? buf[padded(j + r * P::NB0)]
                               : make_float2(0.f, 0.f);
          a[q][r] = {f.x, f.y};
        }
        fft::dft<P::R0, kInv>(a[q]);
      }
    }
    __syncthreads();
    pass0_store<kLog>(buf, a);
    __syncthreads();
  }
  int ns = P::R0;
#pragma unroll 1
  for (int p = 0; p < P::n16; ++p) {
    cf v[P::PER16][16];
    pass16_load_compute<kLog, kInv>(buf, ns, tw, v);
    __syncthreads();
    pass16_store<kLog>(buf, ns, v);
    __syncthreads();
    ns *= 16;
  }
}

}  // namespace fftr
}  // namespace dlr
