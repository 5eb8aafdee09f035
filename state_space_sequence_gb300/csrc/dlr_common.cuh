// dlr_common.cuh -- device helpers shared by the libdlr kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "dlr.h"

#ifdef DLR_BOUNDS_CHECK
// the library's device status word and first failing site (defined once, in api.cu)
extern __device__ int g_dlr_device_status;
extern __device__ int g_dlr_bounds_site;
#endif

namespace dlr {

struct cf {
  float re, im;
};

__device__ __forceinline__ cf cmul(cf a, cf b) {
  return {fmaf(a.re, b.re, -a.im * b.im), fmaf(a.re, b.im, a.im * b.re)};
}
__device__ __forceinline__ cf cadd(cf a, cf b) { return {a.re + b.re, a.im + b.im}; }
__device__ __forceinline__ cf cconj(cf a) { return {a.re, -a.im}; }
// a*b + c
__device__ __forceinline__ cf cfma(cf a, cf b, cf c) {
  return {fmaf(a.re, b.re, fmaf(-a.im, b.im, c.re)), fmaf(a.re, b.im, fmaf(a.im, b.re, c.im))};
}

// Per-state parameters prepared once: a2 = (log Lambda)_re^2 and the phase theta / pi reduced
// to about [-1, 1] and split into float hi + lo.
struct lam_param {
  float a2;
  float th_hi, th_lo;  // theta / pi = th_hi + th_lo (mod 2)
};

// theta / pi in two-float arithmetic (no double precision, which is slow on this GPU):
// 1/pi = kInvPiHi + kInvPiLo (float hi part, then the float rounding of the remainder), so
// theta * kInvPiHi = p + e exactly (e from fmaf) and theta * kInvPiLo adds the next ~24 bits;
// p - 2 round(p / 2) is exact (both are multiples of ulp(p), difference at most 1 in
// magnitude). The result is theta / pi mod 2 to about 2^-45 relative to |theta / pi|.
__device__ __forceinline__ lam_param make_lam_param(float log_re, float log_im) {
  constexpr float kInvPiHi = 0.318309873f;        // float nearest to 1/pi
  constexpr float kInvPiLo = 1.28412765e-08f;     // float nearest to 1/pi - kInvPiHi
  lam_param p;
  p.a2 = log_re * log_re;
  const float hi = log_im * kInvPiHi;
  const float e = fmaf(log_im, kInvPiHi, -hi) + log_im * kInvPiLo;
  const float r = hi - 2.0f * rintf(0.5f * hi);
  const float s = r + e;
  p.th_hi = s;
  p.th_lo = e - (s - r);
  return p;
}

// Reduced phase of j * theta in half-turns, in about [-1, 1]:
//  - j * th_hi is carried exactly as hi + lo (fmaf returns the rounding error of the product;
//    j < 2^24 is exact in float),
//  - hi - 2 round(hi / 2) is exact (both are multiples of ulp(hi) and the difference is at
//    most 1 in magnitude),
//  - lo and j * th_lo are added last.
// The absolute error is about 2^-24 half-turns, independent of j.
__device__ __forceinline__ float reduce_halfturns(float jf, float th_hi, float th_lo) {
  const float hi = jf * th_hi;
  const float lo = fmaf(jf, th_hi, -hi);
  const float r = hi - 2.0f * rintf(0.5f * hi);
  return r + fmaf(jf, th_lo, lo);
}

// lambda^j = exp(-j a^2) * (cos(j theta) + i sin(j theta)), j >= 0, evaluated directly from
// the parameters. Magnitude: the argument j*a2 carries a relative error of one rounding, which
// changes exp(-x) by x*2^-24 relative -- at most e^-1 * 2^-24 of the largest term. Phase: the
// reduction above, then CUDA's sincospif (compiled without fast-math).
__device__ __forceinline__ cf lam_pow(const lam_param& p, int j) {
  const float jf = (float)j;
  const float mag = expf(-jf * p.a2);
  float s, c;
  sincospif(reduce_halfturns(jf, p.th_hi, p.th_lo), &s, &c);
  return {mag * c, mag * s};
}

// ---------------------------------------------------------------------------------------
// Two-float ("double-float") arithmetic, after Dekker (1971) and Knuth's TwoSum: a value is
// hi + lo with |lo| <= ulp(hi)/2.
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b) {
  float s = a + b;
  float bb = s - a;
  float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
  float s = a + b;
  return {s, b - (s - a)};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  float lo = s.lo + (a.lo + b.lo);
  return fast_two_sum(s.hi, lo);
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
  return fast_two_sum(p, e);
}
__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }

struct cff {
  ff re, im;
};
// a*b + c in two-float complex arithmetic
__device__ __forceinline__ cff cff_fma(cff a, cff b, cff c) {
  ff re = ff_add(ff_add(ff_mul(a.re, b.re), ff_neg(ff_mul(a.im, b.im))), c.re);
  ff im = ff_add(ff_add(ff_mul(a.re, b.im), ff_mul(a.im, b.re)), c.im);
  return {re, im};
}

// Index checks of the bounds-checked build. Compiled with DLR_BOUNDS_CHECK (relocatable device
// code, so that every kernel reaches the same two device words), DLR_IN(i, n) is true when
// 0 <= i < n; otherwise it records DLR_ERR_BOUNDS in the device status word and the first
// failing site (kSiteFile * 100000 + source line, kSiteFile set per source file; headers use
// DLR_IN_FILE with their own number) and returns false, and the guarded access is skipped. In
// the normal build both are the constant true.
#ifdef DLR_BOUNDS_CHECK
__device__ __forceinline__ bool dlr_in(long long i, long long n, int site) {
  if (i >= 0 && i < n) return true;
  atomicMax(&::g_dlr_device_status, 6);  // DLR_ERR_BOUNDS
  atomicCAS(&::g_dlr_bounds_site, 0, site);
  return false;
}
#define DLR_IN(i, n) dlr_in((long long)(i), (long long)(n), kSiteFile * 100000 + __LINE__)
#define DLR_IN_FILE(i, n, file) dlr_in((long long)(i), (long long)(n), (file) * 100000 + __LINE__)
#else
#define DLR_IN(i, n) true
#define DLR_IN_FILE(i, n, file) true
#endif

// Kernels whose bounded waits run out record the reason in the library's device status
// word (its address is passed to them as a kernel argument); dlr_get_device_status() reads
// and clears it.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicMax(status, code);
}

// Raise a kernel's dynamic shared-memory limit once per device (later launches -- including
// ones recorded into a CUDA graph -- skip the call).
template <auto Kernel>
inline cudaError_t max_smem_once(size_t bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace dlr
