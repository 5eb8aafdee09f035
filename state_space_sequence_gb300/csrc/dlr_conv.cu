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
#include "fft_rows.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 3;
namespace {

using fft::padded;
using fft::padded_size;

// tw[m] = exp(-2 pi i m / n) for m < n = 2^logn; when tw2 is given, also the 2n-point table.
__global__ void twiddle_table(float2* __restrict__ tw, int logn, float2* __restrict__ tw2) {
  const int n = 1 << logn;
  const int total = tw2 ? 3 * n : n;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    const bool second = e >= n;
    const int m = second ? e - n : e;
    const int lg = second ? logn + 1 : logn;
    float s, c;
    // 2m/N is exact in float for a power-of-two N: exp(-2 pi i m/N) = cos(pi x) - i sin(pi x)
    sincospif(ldexpf((float)m, 1 - lg), &s, &c);
    (second ? tw2 : tw)[m] = make_float2(c, -s);
  }
}

// e^{-i pi k / n} (the M-point twiddle used to split the packed spectrum)
__device__ __forceinline__ cf half_twiddle(int k, int logn) {
  float s, c;
  sincospif(ldexpf((float)k, -logn), &s, &c);
  return {c, -s};
}

// One CTA per channel h: the real circulant column c (length M = 2n) is read as n packed
// complex points z_m = c_{2m} + i c_{2m+1} straight into the first pass, transformed, and the
// Hermitian half S_k, k = 0..n, of its real spectrum is written (scaled, see below).
template <int kLog>
__global__ void __launch_bounds__(fftr::Plan<kLog>::T)
conv_spectrum(const float* __restrict__ K1, const float* __restrict__ K2, int L,
              const float2* __restrict__ tw, float2* __restrict__ spec) {
  using P = fftr::Plan<kLog>;
  constexpr int n = P::n, T = P::T, R0 = P::R0, NB0 = P::NB0;
  extern __shared__ float2 smem[];
  float2* cur = smem;
  float2* nxt = P::kDouble ? smem + P::buf_elems : smem;
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const float* k1 = K1 + (size_t)h * L;
  const float* k2 = K2 ? K2 + (size_t)h * L : nullptr;
  // circulant column: c_0 = K1_0 (+ K2_0), c_i = K1_i (0 < i < L), c_{2n-i} = K2_i (0 < i < L)
  auto col = [&](int i) -> float {
    float v = (i < L) ? k1[i] : 0.f;
    if (k2) {
      if (i == 0) v += k2[0];
      else if (i > 2 * n - L) v += k2[2 * n - i];
    }
    return v;
  };
  cf a[P::PER0][R0];
#pragma unroll
  for (int q = 0; q < P::PER0; ++q) {
    const int j = tid + q * T;
    if (NB0 % T == 0 || j < NB0) {
#pragma unroll
      for (int r = 0; r < R0; ++r) {
        const int m = j + r * NB0;
        a[q][r] = {col(2 * m), col(2 * m + 1)};
      }
      fft::dft<R0, false>(a[q]);
    }
  }
  fftr::pass0_store<kLog>(cur, a);
  __syncthreads();
  int ns = R0;
#pragma unroll 1
  for (int p = 0; p < P::n16; ++p) {
    cf v[P::PER16][16];
    fftr::pass16_load_compute<kLog, false>(cur, ns, tw, v);
    if (!P::kDouble) __syncthreads();
    fftr::pass16_store<kLog>(nxt, ns, v);
    __syncthreads();
    float2* t = cur;
    cur = nxt;
    nxt = t;
    ns *= 16;
  }
  // 1/M for the inverse transform and 1/2 for the row kernel's unscaled unpack (M = 2n)
  const float scale = 1.0f / (float)(4 * n);
  float2* out = spec + (size_t)h * (n + 1);
  for (int k = tid; k <= n / 2; k += T) {
    const int ea = padded(k), eb = padded((n - k) & (n - 1));
    const float2 fa = DLR_IN(ea, P::buf_elems) ? cur[ea] : make_float2(0.f, 0.f);
    const float2 fb = DLR_IN(eb, P::buf_elems) ? cur[eb] : make_float2(0.f, 0.f);
    const cf E = {0.5f * (fa.x + fb.x), 0.5f * (fa.y - fb.y)};
    const cf O = {0.5f * (fa.y + fb.y), -0.5f * (fa.x - fb.x)};  // -i/2 (zk - conj zp)
    const cf wO = cmul(half_twiddle(k, kLog), O);
    const cf Xk = cadd(E, wO);
    const cf Xn = {E.re - wO.re, -(E.im - wO.im)};
    if (DLR_IN(k, n + 1)) out[k] = make_float2(Xk.re * scale, Xk.im * scale);
    if (DLR_IN(n - k, n + 1)) out[n - k] = make_float2(Xn.re * scale, Xn.im * scale);
  }
}

template <int kLog>
__global__ void __launch_bounds__(fftr::Plan<kLog>::T)
conv_rows(const float* __restrict__ u, const float2* __restrict__ spec,
          const float2* __restrict__ tw, float* __restrict__ y, int H, int L) {
  using P = fftr::Plan<kLog>;
  constexpr int n = P::n, T = P::T, R0 = P::R0, NB0 = P::NB0;
  extern __shared__ float2 smem[];
  float2* cur = smem;
  float2* nxt = P::kDouble ? smem + P::buf_elems : smem;
  const int row = blockIdx.x;
  const int h = row % H;
  const int tid = threadIdx.x;
  const float* ur = u + (size_t)row * L;
  float* yr = y + (size_t)row * L;
  const int half = (L + 1) >> 1;  // packed points that hold data
  const bool even = (L & 1) == 0;

  // ---- forward pass 0 (radix R0, no twiddles): inputs straight from global memory ----
  cf a[P::PER0][R0];
#pragma unroll
  for (int q = 0; q < P::PER0; ++q) {
    const int j = tid + q * T;
    if (NB0 % T == 0 || j < NB0) {
#pragma unroll
      for (int r = 0; r < R0; ++r) {
        const int m = j + r * NB0;
        cf z = {0.f, 0.f};
        if (m < half) {
          if (even) {
            float2 f = __ldg(reinterpret_cast<const float2*>(ur) + m);
            z = {f.x, f.y};
          } else {
            z.re = ur[2 * m];
            z.im = (2 * m + 1 < L) ? ur[2 * m + 1] : 0.f;
          }
        }
        a[q][r] = z;
      }
      // inputs m >= n/2 (r >= R0/2) are the zero padding: L <= n
      if constexpr (R0 == 16) fft::dft16_lowhalf<false>(a[q]);
      else fft::dft<R0, false>(a[q]);
    }
  }
  fftr::pass0_store<kLog>(cur, a);
  __syncthreads();

  // ---- forward radix-16 passes ----
  int ns = R0;
#pragma unroll 1
  for (int p = 0; p < P::n16; ++p) {
    cf v[P::PER16][16];
    fftr::pass16_load_compute<kLog, false>(cur, ns, tw, v);
    if (!P::kDouble) __syncthreads();
    fftr::pass16_store<kLog>(nxt, ns, v);
    __syncthreads();
    float2* t = cur;
    cur = nxt;
    nxt = t;
    ns *= 16;
  }

  // ---- spectral step: unpack the real spectrum, multiply, re-pack; the results are the
  // inputs k = j + r n/R0 of the first inverse pass ----
  const float2* S = spec + (size_t)h * (n + 1);
#pragma unroll
  for (int q = 0; q < P::PER0; ++q) {
    const int j = tid + q * T;
    if (NB0 % T == 0 || j < NB0) {
      cf base = {1.f, 0.f};
      if constexpr (NB0 % 2 == 0) {
        float sb, cb;
        sincospif(ldexpf((float)j, -kLog), &sb, &cb);
        base = {cb, -sb};  // e^{-i pi j / n}
      }
#pragma unroll
      for (int r = 0; r < R0; ++r) {
        const int k = j + r * NB0;
        const int kp = (n - k) & (n - 1);
        cf w;
        if constexpr (R0 == 16 && NB0 % 2 == 0) {
          w = cmul(base, fftr::half16(r));     // e^{-i pi r / 16}
        } else if constexpr (NB0 % 2 == 0) {
          float2 c = __ldg(&tw[r * (NB0 / 2)]);  // e^{-i pi r / R0}
          w = cmul(base, {c.x, c.y});
        } else {
          float sw, cw;
          sincospif(ldexpf((float)k, -kLog), &sw, &cw);
          w = {cw, -sw};
        }
        const int ea = padded(k), eb = padded(kp);
        float2 fa = DLR_IN(ea, P::buf_elems) ? cur[ea] : make_float2(0.f, 0.f);
        float2 fb = DLR_IN(eb, P::buf_elems) ? cur[eb] : make_float2(0.f, 0.f);
        // 2E = Zk + conj(Zp), 2O = -i (Zk - conj(Zp)); the 1/2 lives in the spectrum
        cf E = {fa.x + fb.x, fa.y - fb.y};
        cf O = {fa.y + fb.y, fb.x - fa.x};
        cf wO = cmul(w, O);
        cf X = cadd(E, wO);
        cf Xn = {E.re - wO.re, wO.im - E.im};
        float2 sk = DLR_IN(k, n + 1) ? __ldg(&S[k]) : make_float2(0.f, 0.f);
        float2 sn = DLR_IN(n - k, n + 1) ? __ldg(&S[n - k]) : make_float2(0.f, 0.f);
        cf Yk = cmul(X, {sk.x, sk.y});
        cf Yn = cmul(Xn, {sn.x, sn.y});
        cf Ep = {Yk.re + Yn.re, Yk.im - Yn.im};
        cf Op = cmul({Yk.re - Yn.re, Yk.im + Yn.im}, cconj(w));
        a[q][r] = {Ep.re - Op.im, Ep.im + Op.re};
      }
      fft::dft<R0, true>(a[q]);
    }
  }
  if (!P::kDouble) __syncthreads();
  fftr::pass0_store<kLog>(nxt, a);
  __syncthreads();
  {
    float2* t = cur;
    cur = nxt;
    nxt = t;
  }
  ns = R0;

  // ---- inverse radix-16 passes; the last one writes y ----
  if constexpr (P::n16 == 0) {
    for (int m = tid; m < half; m += T) {
      float2 z = DLR_IN(padded(m), P::buf_elems) ? cur[padded(m)] : make_float2(0.f, 0.f);
      if (even) {
        reinterpret_cast<float2*>(yr)[m] = z;
      } else {
        yr[2 * m] = z.x;
        if (2 * m + 1 < L) yr[2 * m + 1] = z.y;
      }
    }
  } else {
#pragma unroll 1
    for (int p = 0; p < P::n16; ++p) {
      cf v[P::PER16][16];
      fftr::pass16_load_compute<kLog, true>(cur, ns, tw, v);
      if (p < P::n16 - 1) {
        if (!P::kDouble) __syncthreads();
        fftr::pass16_store<kLog>(nxt, ns, v);
        __syncthreads();
        float2* t = cur;
        cur = nxt;
        nxt = t;
        ns *= 16;
      } else {
        // last pass: thread j holds outputs j + r n/16 (ns = n/16, so k = j)
#pragma unroll
        for (int q = 0; q < P::PER16; ++q) {
          const int j = tid + q * T;
          if (P::NB16 % T == 0 || j < P::NB16) {
#pragma unroll
            for (int r = 0; r < 16; ++r) {
              const int m = j + r * P::NB16;
              if (m < half) {
                if (even) {
                  reinterpret_cast<float2*>(yr)[m] = make_float2(v[q][r].re, v[q][r].im);
                } else {
                  yr[2 * m] = v[q][r].re;
                  if (2 * m + 1 < L) yr[2 * m + 1] = v[q][r].im;
                }
              }
            }
          }
        }
      }
    }
  }
}

// Two rows of the same channel per CTA, as the real and imaginary parts of one complex
// sequence z = u_b0 + i u_b1 of M = 2n points (zero beyond L): one forward and one inverse
// complex FFT of size M per pair, and between them a plain complex product with the full
// kernel spectrum (the spectrum of a real kernel is Hermitian, so Re / Im of the result are the
// two rows' convolutions). Because z is zero on its upper half, the first radix-2 pass of the
// forward transform only duplicates points: the first real pass reads z[i >> 1] straight from
// global memory. The last inverse pass (radix 2) computes only the outputs m < L.
template <int kG>
struct PairPlan {
  using P = fftr::Plan<kG>;                     // radix-16 passes over M points
  static constexpr int M = 1 << kG;
  static constexpr int G1 = kG - 1;             // bits after the duplicating radix-2 pass
  static constexpr int R1 = (G1 % 4 == 0) ? 16 : (1 << (G1 % 4));
  static constexpr int n16 = (G1 % 4 == 0) ? G1 / 4 - 1 : G1 / 4;
  static constexpr int T = P::T;
  static constexpr int NB1 = M / R1;
  static constexpr int PER1 = (NB1 + T - 1) / T;
  static constexpr size_t buf_elems = padded_size(M);
  static constexpr bool kDouble = 2 * buf_elems * sizeof(float2) <= 72 * 1024;
  static constexpr size_t smem = (kDouble ? 2 : 1) * buf_elems * sizeof(float2);
};

template <int kG>
__global__ void __launch_bounds__(PairPlan<kG>::T)
conv_pairs(const float* __restrict__ u, const float2* __restrict__ spec,
           const float2* __restrict__ twM, float* __restrict__ y, int B, int H, int L) {
  using PP = PairPlan<kG>;
  using P = typename PP::P;
  constexpr int M = PP::M, T = PP::T, R1 = PP::R1, NB1 = PP::NB1;
  constexpr int n = M / 2;
  extern __shared__ float2 smem[];
  float2* cur = smem;
  float2* nxt = PP::kDouble ? smem + PP::buf_elems : smem;
  const int pair = blockIdx.x / H, h = blockIdx.x % H;
  const int b0 = 2 * pair, b1 = 2 * pair + 1;
  const bool has1 = b1 < B;
  const float* u0 = u + ((size_t)b0 * H + h) * L;
  const float* u1 = u + ((size_t)(has1 ? b1 : b0) * H + h) * L;
  const int tid = threadIdx.x;

  // ---- forward pass 1 (radix R1, ns = 2): inputs z[i >> 1] from global memory ----
  {
    cf a[PP::PER1][R1];
    int dst[PP::PER1];
#pragma unroll
    for (int q = 0; q < PP::PER1; ++q) {
      const int j = tid + q * T;
      dst[q] = -1;
      if (NB1 % T == 0 || j < NB1) {
#pragma unroll
        for (int r = 0; r < R1; ++r) {
          const int m = (j >> 1) + r * (NB1 / 2);
          cf z = {0.f, 0.f};
          if (m < L) z = {__ldg(&u0[m]), has1 ? __ldg(&u1[m]) : 0.f};
          a[q][r] = z;
        }
        const int k = j & 1;
        if (k) {
#pragma unroll
          for (int r = 1; r < R1; ++r) a[q][r] = cmul(a[q][r], fftr::half16(r * (16 / R1)));
        }
        fft::dft<R1, false>(a[q]);
        dst[q] = (j - k) * R1 + k;
      }
    }
#pragma unroll
    for (int q = 0; q < PP::PER1; ++q)
      if (dst[q] >= 0) {
#pragma unroll
        for (int r = 0; r < R1; ++r)
          if (DLR_IN(padded(dst[q] + 2 * r), PP::buf_elems))
            cur[padded(dst[q] + 2 * r)] = make_float2(a[q][r].re, a[q][r].im);
      }
  }
  __syncthreads();

  // ---- forward radix-16 passes; the last leaves Z[j + r M/16] in registers ----
  int ns = 2 * R1;
  cf v[P::PER16][16];
#pragma unroll 1
  for (int p = 0; p < PP::n16; ++p) {
    fftr::pass16_load_compute<kG, false>(cur, ns, twM, v);
    if (p < PP::n16 - 1) {
      if (!PP::kDouble) __syncthreads();
      fftr::pass16_store<kG>(nxt, ns, v);
      __syncthreads();
      float2* t = cur;
      cur = nxt;
      nxt = t;
      ns *= 16;
    }
  }

  // ---- spectral product: Y_k = Z_k * C_k, C_k = 2 S_k (k <= n), conj(2 S_{M-k}) (k > n) ----
  const float2* S = spec + (size_t)h * (n + 1);
#pragma unroll
  for (int q = 0; q < P::PER16; ++q) {
    const int j = tid + q * T;
    if (P::NB16 % T == 0 || j < P::NB16) {
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int k = j + r * P::NB16;
        float2 c = make_float2(0.f, 0.f);
        if (k <= n) {
          if (DLR_IN(k, n + 1)) c = __ldg(&S[k]);
        } else {
          if (DLR_IN(M - k, n + 1)) c = __ldg(&S[M - k]);
          c.y = -c.y;
        }
        v[q][r] = cmul(v[q][r], {2.f * c.x, 2.f * c.y});
      }
    }
  }

  // ---- inverse pass 1 (radix R1, ns = 1) ----
  if constexpr (R1 == 16) {
    // the registers already hold the inputs x[j + r M/16] of a radix-16 first pass
#pragma unroll
    for (int q = 0; q < P::PER16; ++q) {
      const int j = tid + q * T;
      if (P::NB16 % T == 0 || j < P::NB16) fft::dft<16, true>(v[q]);
    }
    if (!PP::kDouble) __syncthreads();
#pragma unroll
    for (int q = 0; q < P::PER16; ++q) {
      const int j = tid + q * T;
      if (P::NB16 % T == 0 || j < P::NB16) {
        float2* d0 = nxt + padded(16 * j);
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (DLR_IN(padded(16 * j) + r, PP::buf_elems)) d0[r] = make_float2(v[q][r].re, v[q][r].im);
      }
    }
  } else {
    // park Y in natural order, then run the radix-R1 pass from shared memory
    if (!PP::kDouble) __syncthreads();
    fftr::pass16_store<kG>(nxt, P::NB16, v);  // ns = M/16: positions j + r M/16
    __syncthreads();
    {
      float2* t = cur;
      cur = nxt;
      nxt = t;
    }
    cf a[PP::PER1][R1];
#pragma unroll
    for (int q = 0; q < PP::PER1; ++q) {
      const int j = tid + q * T;
      if (NB1 % T == 0 || j < NB1) {
#pragma unroll
        for (int r = 0; r < R1; ++r) {
          const float2 f = DLR_IN(padded(j + r * NB1), PP::buf_elems) ? cur[padded(j + r * NB1)]
                                                                      : make_float2(0.f, 0.f);
          a[q][r] = {f.x, f.y};
        }
        fft::dft<R1, true>(a[q]);
      }
    }
    if (!PP::kDouble) __syncthreads();
#pragma unroll
    for (int q = 0; q < PP::PER1; ++q) {
      const int j = tid + q * T;
      if (NB1 % T == 0 || j < NB1) {
        float2* d0 = nxt + padded(j * R1);
#pragma unroll
        for (int r = 0; r < R1; ++r)
          if (DLR_IN(padded(j * R1) + r, PP::buf_elems)) d0[r] = make_float2(a[q][r].re, a[q][r].im);
      }
    }
  }
  __syncthreads();
  {
    float2* t = cur;
    cur = nxt;
    nxt = t;
  }

  // ---- inverse radix-16 passes (ns = R1 ... M/32) ----
  ns = R1;
#pragma unroll 1
  for (int p = 0; p < PP::n16; ++p) {
    fftr::pass16_load_compute<kG, true>(cur, ns, twM, v);
    if (!PP::kDouble) __syncthreads();
    fftr::pass16_store<kG>(nxt, ns, v);
    __syncthreads();
    float2* t = cur;
    cur = nxt;
    nxt = t;
    ns *= 16;
  }

  // ---- last inverse pass (radix 2, ns = M/2), only outputs m < L: x_m + w^m x_{m + M/2} ----
  float* y0 = y + ((size_t)b0 * H + h) * L;
  float* y1 = y + ((size_t)(has1 ? b1 : b0) * H + h) * L;
  for (int m = tid; m < L; m += T) {
    const float2 a = DLR_IN(padded(m), PP::buf_elems) ? cur[padded(m)] : make_float2(0.f, 0.f);
    const float2 b = DLR_IN(padded(m + n), PP::buf_elems) ? cur[padded(m + n)] : make_float2(0.f, 0.f);
    const float2 w = __ldg(&twM[m]);
    const cf t = cmul({b.x, b.y}, {w.x, -w.y});
    y0[m] = a.x + t.re;
    if (has1) y1[m] = a.y + t.im;
  }
}

template <int kG>
cudaError_t launch_pairs(const float* u, int B, int H, int L, float* y, const float2* twM,
                         const float2* spec, cudaStream_t s) {
  using PP = PairPlan<kG>;
  if (PP::smem > 48 * 1024) {
    cudaError_t e = max_smem_once<conv_pairs<kG>>(PP::smem);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = (unsigned)(((size_t)B + 1) / 2 * H);
  conv_pairs<kG><<<grid, PP::T, PP::smem, s>>>(u, spec, twM, y, B, H, L);
  return cudaGetLastError();
}

template <int kLog>
cudaError_t launch_spectrum(const float* K1, const float* K2, int H, int L, float2* tw,
                            float2* spec, cudaStream_t s) {
  using P = fftr::Plan<kLog>;
  if (P::smem > 48 * 1024) {
    cudaError_t e = max_smem_once<conv_spectrum<kLog>>(P::smem);
    if (e != cudaSuccess) return e;
  }
  conv_spectrum<kLog><<<H, P::T, P::smem, s>>>(K1, K2, L, tw, spec);
  return cudaGetLastError();
}

template <int kLog>
cudaError_t launch_apply(const float* u, int B, int H, int L, float* y, const float2* tw,
                         const float2* spec, cudaStream_t s) {
  using P = fftr::Plan<kLog>;
  if (P::smem > 48 * 1024) {
    cudaError_t e = max_smem_once<conv_rows<kLog>>(P::smem);
    if (e != cudaSuccess) return e;
  }
  conv_rows<kLog><<<(unsigned)((size_t)B * H), P::T, P::smem, s>>>(u, spec, tw, y, H, L);
  return cudaGetLastError();
}

struct ConvWs {
  float2* tw;    // n-point table  e^{-2 pi i m / n}
  float2* tw2;   // 2n-point table e^{-2 pi i m / 2n}
  float2* spec;  // [H][n + 1]
};

ConvWs carve_conv(const void* ws, int lg) {
  const size_t n = size_t(1) << lg;
  const size_t twb = (sizeof(float2) * n + 255) & ~size_t(255);
  const size_t tw2b = (sizeof(float2) * 2 * n + 255) & ~size_t(255);
  char* base = const_cast<char*>(reinterpret_cast<const char*>(ws));
  return {reinterpret_cast<float2*>(base), reinterpret_cast<float2*>(base + twb),
          reinterpret_cast<float2*>(base + twb + tw2b)};
}

}  // namespace

int conv_log2_size(int64_t L) {
  int lg = 0;
  while ((int64_t(1) << lg) < L) ++lg;
  return lg;  // n = 2^lg >= L complex points, FFT size M = 2n
}

size_t conv_workspace_bytes(int64_t H, int64_t L) {
  const int64_t n = int64_t(1) << conv_log2_size(L);
  const size_t tw = (sizeof(float2) * (size_t)n + 255) & ~size_t(255);
  const size_t tw2 = (sizeof(float2) * 2 * (size_t)n + 255) & ~size_t(255);
  return tw + tw2 + sizeof(float2) * (size_t)H * (size_t)(n + 1);
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

cudaError_t launch_cluster_spectrum(const float* K1, const float* K2, int H, int L, int lg,
                                    const float2* tw_loc, float2* spec, cudaStream_t s);
cudaError_t launch_cluster_apply(const float* u, int B, int H, int L, int lg,
                                 const float2* tw_loc, const float2* spec, float* y,
                                 cudaStream_t s);

cudaError_t launch_dlr_conv_spectrum(const float* K1, const float* K2, int H, int L, void* ws,
                                     cudaStream_t s) {
  const int lg = conv_log2_size(L);
  ConvWs w = carve_conv(ws, lg);
  if (lg > 14) {  // a cluster of 8 CTAs per channel; local transforms of n / 8 points
    const int lloc = lg - 3;
    twiddle_table<<<((1 << lloc) + 255) / 256, 256, 0, s>>>(w.tw, lloc, nullptr);
    return launch_cluster_spectrum(K1, K2, H, L, lg, w.tw, w.spec, s);
  }
  // one launch for the n-point table and, where the two-rows-per-transform kernel may run,
  // the 2n-point table
  const bool pairs = lg >= 11 && lg <= 13;
  twiddle_table<<<((pairs ? 3 : 1) * (1 << lg) + 255) / 256, 256, 0, s>>>(w.tw, lg,
                                                                            pairs ? w.tw2 : nullptr);
#define SPEC_CALL(G) launch_spectrum<G>(K1, K2, H, L, w.tw, w.spec, s)
  DLR_CONV_SWITCH(SPEC_CALL)
#undef SPEC_CALL
}

// The twiddle tables of the convolution workspace alone (for a spectrum written by another
// route): the n-point table, and the 2n-point one where the two-rows-per-transform kernel may
// run, or the local n/8-point table of the cluster transform.
cudaError_t launch_twiddles(int lg, void* ws, cudaStream_t s) {
  ConvWs w = carve_conv(ws, lg);
  if (lg > 14) {
    const int lloc = lg - 3;
    twiddle_table<<<((1 << lloc) + 255) / 256, 256, 0, s>>>(w.tw, lloc, nullptr);
    return cudaGetLastError();
  }
  const bool pairs = lg >= 11 && lg <= 13;
  twiddle_table<<<((pairs ? 3 : 1) * (1 << lg) + 255) / 256, 256, 0, s>>>(w.tw, lg,
                                                                            pairs ? w.tw2 : nullptr);
  return cudaGetLastError();
}

// The spectra region of a convolution workspace for rows of L (n = 2^conv_log2_size(L) + 1
// bins per row, in the transform's own bin order), for another module that forms spectra
// pointwise from spectra this file wrote.
float2* conv_spectra(void* ws, int64_t L) { return carve_conv(ws, conv_log2_size(L)).spec; }

// tw[m] = exp(-2 pi i m / n), m < n = 2^logn, for another module's transforms.
cudaError_t launch_twiddle_table(float2* tw, int logn, cudaStream_t s) {
  twiddle_table<<<((1 << logn) + 255) / 256, 256, 0, s>>>(tw, logn, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_dlr_conv_apply(const float* u, int B, int H, int L, float* y, const void* ws,
                                  cudaStream_t s) {
  const int lg = conv_log2_size(L);
  ConvWs w = carve_conv(ws, lg);
  if (lg > 14) return launch_cluster_apply(u, B, H, L, lg, w.tw, w.spec, y, s);
  if (B >= 2 && lg >= 11 && lg <= 13) {  // two rows per complex transform of size 2n
    if (lg == 11) return launch_pairs<12>(u, B, H, L, y, w.tw2, w.spec, s);
    if (lg == 12) return launch_pairs<13>(u, B, H, L, y, w.tw2, w.spec, s);
    return launch_pairs<14>(u, B, H, L, y, w.tw2, w.spec, s);
  }
#define APPLY_CALL(G) launch_apply<G>(u, B, H, L, y, w.tw, w.spec, s)
  DLR_CONV_SWITCH(APPLY_CALL)
#undef APPLY_CALL
}

}  // namespace dlr
