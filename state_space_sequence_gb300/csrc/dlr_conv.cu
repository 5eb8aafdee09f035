// dlr_conv.cu -- causal / bidirectional DLR convolution by FFT ("Simplifying and
// Understanding State Space Models with Diagonal Linear RNNs", section 2.1 and appendix A.1:
// the Toeplitz matrix-vector product computed as a circulant product of size 2L via FFT;
// "The Annotated S4", part 1 "Convolutive view": zero-pad to 2L, multiply spectra, keep the
// first L outputs).
//
// Layout of the work:
//   * twiddle table  tw[m] = exp(-2 pi i m / n), n = FFT size / 2 (one launch, n threads)
//   * spectrum       one CTA per channel h: the real length-M (M = 2n >= 2L) circulant column
//                    c (causal: [K, 0]; bidirectional: [K1_0 + K2_0, K1_1.., 0.., K2_{L-1}..K2_1])
//                    -> real FFT -> S_k = C_k / M for k = 0..n, kept in the workspace.
//   * convolution    one CTA per (b, h) row: the row u (L floats) is read as n packed complex
//                    points z_m = u_{2m} + i u_{2m+1} (zero beyond L), one complex FFT of size n,
//                    a single pass that unpacks the real spectrum, multiplies by S and re-packs
//                    for the inverse, one inverse complex FFT, and the first L reals are y.
// The row never leaves shared memory between its HBM read and its HBM write.
#include "fft_smem.cuh"

namespace dlr {
namespace {

using fft::padded;
using fft::padded_size;

__global__ void twiddle_table(float2* __restrict__ tw, int logn) {
  const int n = 1 << logn;
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < n; m += gridDim.x * blockDim.x) {
    float s, c;
    // 2m/n is exact in float for a power-of-two n: exp(-2 pi i m/n) = cos(pi x) - i sin(pi x)
    sincospif(ldexpf((float)m, 1 - logn), &s, &c);
    tw[m] = make_float2(c, -s);
  }
}

template <int kLog>
struct Cfg {
  static constexpr int n = 1 << kLog;
  static constexpr int threads = (n / 16) < 32 ? 32 : ((n / 16) > 512 ? 512 : n / 16);
  static constexpr size_t smem = sizeof(float2) * padded_size(n);
};

// e^{-i pi k / n} (the M-point twiddle used to split the packed spectrum)
__device__ __forceinline__ cf half_twiddle(int k, int logn) {
  float s, c;
  sincospif(ldexpf((float)k, -logn), &s, &c);
  return {c, -s};
}

template <int kLog>
__global__ void __launch_bounds__(Cfg<kLog>::threads)
conv_spectrum(const float* __restrict__ K1, const float* __restrict__ K2, int L,
              const float2* __restrict__ tw, float2* __restrict__ spec) {
  constexpr int n = Cfg<kLog>::n;
  constexpr int T = Cfg<kLog>::threads;
  extern __shared__ float2 buf[];
  float* fb = reinterpret_cast<float*>(buf);
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const float* k1 = K1 + (size_t)h * L;
  const float* k2 = K2 ? K2 + (size_t)h * L : nullptr;
  for (int m = tid; m < n; m += T) buf[padded(m)] = make_float2(0.f, 0.f);
  __syncthreads();
  // real circulant column c of length M = 2n; c[j] lives at float slot 2*padded(j/2) + j%2
  for (int j = tid; j < L; j += T) {
    float v = k1[j];
    if (j == 0 && k2) v += k2[0];
    fb[2 * padded(j >> 1) + (j & 1)] = v;
  }
  if (k2) {
    for (int j = 1 + tid; j < L; j += T) {
      int m = 2 * n - j;
      fb[2 * padded(m >> 1) + (m & 1)] = k2[j];
    }
  }
  __syncthreads();
  fft::fft<kLog, false, T>(buf, tw);
  const float scale = 1.0f / (float)(2 * n);
  float2* out = spec + (size_t)h * (n + 1);
  for (int k = tid; k <= n / 2; k += T) {
    float2 a = buf[padded(k)], b = buf[padded((n - k) & (n - 1))];
    cf zk = {a.x, a.y}, zp = {b.x, b.y};
    cf E = {0.5f * (zk.re + zp.re), 0.5f * (zk.im - zp.im)};
    cf O = {0.5f * (zk.im + zp.im), -0.5f * (zk.re - zp.re)};  // -i/2 (zk - conj zp)
    cf wO = cmul(half_twiddle(k, kLog), O);
    cf Xk = cadd(E, wO);
    cf Xn = {E.re - wO.re, -(E.im - wO.im)};
    out[k] = make_float2(Xk.re * scale, Xk.im * scale);
    out[n - k] = make_float2(Xn.re * scale, Xn.im * scale);
  }
}

template <int kLog>
__global__ void __launch_bounds__(Cfg<kLog>::threads)
conv_rows(const float* __restrict__ u, const float2* __restrict__ spec,
          const float2* __restrict__ tw, float* __restrict__ y, int H, int L) {
  constexpr int n = Cfg<kLog>::n;
  constexpr int T = Cfg<kLog>::threads;
  extern __shared__ float2 buf[];
  float* fb = reinterpret_cast<float*>(buf);
  const int row = blockIdx.x;
  const int h = row % H;
  const int tid = threadIdx.x;
  const float* ur = u + (size_t)row * L;
  float* yr = y + (size_t)row * L;

  // 1) load the row as packed complex points, zero padded to n
  const int half = (L + 1) >> 1;  // packed points holding data
  if ((L & 3) == 0) {
    const float4* u4 = reinterpret_cast<const float4*>(ur);
    for (int i = tid; i < (L >> 2); i += T) {
      float4 f = __ldg(&u4[i]);
      buf[padded(2 * i)] = make_float2(f.x, f.y);
      buf[padded(2 * i + 1)] = make_float2(f.z, f.w);
    }
  } else {
    for (int m = tid; m < half; m += T) {
      float a = ur[2 * m];
      float b = (2 * m + 1 < L) ? ur[2 * m + 1] : 0.f;
      buf[padded(m)] = make_float2(a, b);
    }
  }
  for (int m = half + tid; m < n; m += T) buf[padded(m)] = make_float2(0.f, 0.f);
  __syncthreads();

  // 2) forward FFT of the packed row
  fft::fft<kLog, false, T>(buf, tw);

  // 3) unpack to the real spectrum X, multiply by S, re-pack for the inverse
  const float2* S = spec + (size_t)h * (n + 1);
  for (int k = tid; k <= n / 2; k += T) {
    const int kp = (n - k) & (n - 1);
    float2 a = buf[padded(k)], b = buf[padded(kp)];
    cf zk = {a.x, a.y}, zp = {b.x, b.y};
    cf E = {0.5f * (zk.re + zp.re), 0.5f * (zk.im - zp.im)};
    cf O = {0.5f * (zk.im + zp.im), -0.5f * (zk.re - zp.re)};
    cf w = half_twiddle(k, kLog);
    cf wO = cmul(w, O);
    cf Xk = cadd(E, wO);
    cf Xn = {E.re - wO.re, -(E.im - wO.im)};
    float2 sk = __ldg(&S[k]), sn = __ldg(&S[n - k]);
    cf Yk = cmul(Xk, {sk.x, sk.y});
    cf Yn = cmul(Xn, {sn.x, sn.y});
    cf Ep = {Yk.re + Yn.re, Yk.im - Yn.im};                       // Yk + conj(Yn)
    cf Op = cmul({Yk.re - Yn.re, Yk.im + Yn.im}, cconj(w));       // (Yk - conj(Yn)) conj(w)
    buf[padded(k)] = make_float2(Ep.re - Op.im, Ep.im + Op.re);   // Ep + i Op
    if (k != 0 && k != kp)
      buf[padded(kp)] = make_float2(Ep.re + Op.im, -Ep.im + Op.re);  // conj(Ep) + i conj(Op)
  }
  __syncthreads();

  // 4) inverse FFT; z'_m = y_{2m} + i y_{2m+1}
  fft::fft<kLog, true, T>(buf, tw);

  // 5) store the first L reals
  if ((L & 3) == 0) {
    float4* y4 = reinterpret_cast<float4*>(yr);
    for (int i = tid; i < (L >> 2); i += T) {
      float2 a = buf[padded(2 * i)], b = buf[padded(2 * i + 1)];
      y4[i] = make_float4(a.x, a.y, b.x, b.y);
    }
  } else {
    for (int j = tid; j < L; j += T) yr[j] = fb[2 * padded(j >> 1) + (j & 1)];
  }
}

template <int kLog>
cudaError_t launch_spectrum(const float* K1, const float* K2, int H, int L, float2* tw,
                            float2* spec, cudaStream_t s) {
  using C = Cfg<kLog>;
  if (C::smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(conv_spectrum<kLog>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem);
    if (e != cudaSuccess) return e;
  }
  twiddle_table<<<(C::n + 255) / 256, 256, 0, s>>>(tw, kLog);
  conv_spectrum<kLog><<<H, C::threads, C::smem, s>>>(K1, K2, L, tw, spec);
  return cudaGetLastError();
}

template <int kLog>
cudaError_t launch_apply(const float* u, int B, int H, int L, float* y, const float2* tw,
                         const float2* spec, cudaStream_t s) {
  using C = Cfg<kLog>;
  if (C::smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(conv_rows<kLog>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem);
    if (e != cudaSuccess) return e;
  }
  conv_rows<kLog><<<(unsigned)((size_t)B * H), C::threads, C::smem, s>>>(u, spec, tw, y, H, L);
  return cudaGetLastError();
}

struct ConvWs {
  float2* tw;
  float2* spec;
};

ConvWs carve_conv(const void* ws, int lg) {
  const size_t n = size_t(1) << lg;
  const size_t twb = (sizeof(float2) * n + 255) & ~size_t(255);
  char* base = const_cast<char*>(reinterpret_cast<const char*>(ws));
  return {reinterpret_cast<float2*>(base), reinterpret_cast<float2*>(base + twb)};
}

}  // namespace

int conv_log2_size(int64_t L) {
  int lg = 0;
  while ((int64_t(1) << lg) < L) ++lg;
  return lg;  // n = 2^lg >= L complex points, FFT size M = 2n
}

size_t conv_workspace_bytes(int64_t H, int64_t L) {
  const int64_t n = int64_t(1) << conv_log2_size(L);
  size_t tw = sizeof(float2) * (size_t)n;
  tw = (tw + 255) & ~size_t(255);
  return tw + sizeof(float2) * (size_t)H * (size_t)(n + 1);
}

#define DLR_CONV_SWITCH(CALL)                                                              \
  switch (lg) {                                                                            \
    case 0: return CALL(0); case 1: return CALL(1); case 2: return CALL(2);                \
    case 3: return CALL(3); case 4: return CALL(4); case 5: return CALL(5);                \
    case 6: return CALL(6); case 7: return CALL(7); case 8: return CALL(8);                \
    case 9: return CALL(9); case 10: return CALL(10); case 11: return CALL(11);            \
    case 12: return CALL(12); case 13: return CALL(13); case 14: return CALL(14);          \
    default: return cudaErrorInvalidValue;                                                 \
  }

cudaError_t launch_dlr_conv_spectrum(const float* K1, const float* K2, int H, int L, void* ws,
                                     cudaStream_t s) {
  const int lg = conv_log2_size(L);
  ConvWs w = carve_conv(ws, lg);
#define SPEC_CALL(G) launch_spectrum<G>(K1, K2, H, L, w.tw, w.spec, s)
  DLR_CONV_SWITCH(SPEC_CALL)
#undef SPEC_CALL
}

cudaError_t launch_dlr_conv_apply(const float* u, int B, int H, int L, float* y, const void* ws,
                                  cudaStream_t s) {
  const int lg = conv_log2_size(L);
  ConvWs w = carve_conv(ws, lg);
#define APPLY_CALL(G) launch_apply<G>(u, B, H, L, y, w.tw, w.spec, s)
  DLR_CONV_SWITCH(APPLY_CALL)
#undef APPLY_CALL
}

}  // namespace dlr
