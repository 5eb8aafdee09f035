// dlr_conv_cluster.cu -- FFT convolution for rows too long for one CTA's shared memory
// (16384 < L <= 65536): the packed transform of n = 8 * n_loc complex points is spread over a
// cluster of 8 CTAs and exchanged through distributed shared memory.
//
// Four-step factorisation with m = c n_loc + i (c = CTA rank) and k = k1 + 8 k2:
//   Z[k1 + 8 k2] = sum_i W_{n_loc}^{i k2} ( W_n^{i k1} sum_c z[c n_loc + i] W_8^{c k1} )
// so a row is transformed by
//   F1  radix-8 DFT across the cluster (each CTA takes n_loc/8 columns i, reads the 8 values
//       z[c n_loc + i] from the 8 CTAs, twiddles by W_n^{i k1} and writes output k1 into CTA k1),
//   F2  a local n_loc-point Stockham FFT in each CTA: CTA k1 then holds Z[k1 + 8 k2] at k2,
// the spectral step pairs k with n - k (the mirror sits in CTA (8 - k1) mod 8), and the inverse
// runs the same two steps backwards: local inverse FFT, then the radix-8 inverse DFT across the
// cluster, whose outputs go straight to global memory. Same arithmetic as the one-CTA row
// kernel otherwise ("Simplifying and Understanding State Space Models with Diagonal Linear
// RNNs", section 2.1 and appendix A.1: Toeplitz product as a circulant product of size >= 2L).
// Spectra are stored in cluster order S'[k1 n_loc + k2] = S[k1 + 8 k2], with S[n] last.
//
// Every step works in place in one shared buffer of n_loc points (70 KB at n_loc = 8192), so
// two CTAs (of different clusters) share an SM and hide each other's barrier and load
// latency:
//   F1 / I1  the thread of column i reads position i of the 8 CTAs and writes position i of
//            the 8 CTAs (F1) or global memory (I1); no other thread touches position i;
//   F2 / I2  each Stockham pass loads all of a thread's points, synchronises, stores them;
//   spectral step: one thread per pair (k, n - k) reads both points and writes both outputs
//            (the partner may sit in the mirror CTA), so each point is read and written by
//            one thread.
#include "fft_rows.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 4;
namespace {

using fft::padded;
using fft::padded_size;
using fftr::local_fft;
constexpr int kC = 8;  // CTAs per cluster

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
               : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// x^e for e < 8, at most three multiplications deep
__device__ __forceinline__ void powers8(cf (&p)[8], cf x) {
  p[0] = {1.f, 0.f};
  p[1] = x;
  p[2] = cmul(x, x);
  p[3] = cmul(p[2], x);
  p[4] = cmul(p[2], p[2]);
  p[5] = cmul(p[4], x);
  p[6] = cmul(p[4], p[2]);
  p[7] = cmul(p[4], p[3]);
}

// The spectral step's output at bin k from the packed transform's Z_k (fa) and Z_{n-k} (fb),
// the kernel spectra S_k (sk) and S_{n-k} (sn; S_n at k = 0), w = e^{-i pi k / n}: the real
// spectra X_k, X_{n-k} unpacked, multiplied, and repacked as the inverse transform's input.
__device__ __forceinline__ float2 spectral_point(float2 fa, float2 fb, float2 sk, float2 sn,
                                                 cf w) {
  const cf E = {fa.x + fb.x, fa.y - fb.y};
  const cf O = {fa.y + fb.y, fb.x - fa.x};
  const cf wO = cmul(w, O);
  const cf X = cadd(E, wO);
  const cf Xn = {E.re - wO.re, wO.im - E.im};
  const cf Yk = cmul(X, {sk.x, sk.y});
  const cf Yn = cmul(Xn, {sn.x, sn.y});
  const cf Ep = {Yk.re + Yn.re, Yk.im - Yn.im};
  const cf Op = cmul({Yk.re - Yn.re, Yk.im + Yn.im}, cconj(w));
  return make_float2(Ep.re - Op.im, Ep.im + Op.re);
}

template <int kLog>
__device__ __forceinline__ cf half_turn_twiddle(int k) {  // e^{-i pi k / n}, n = 8 n_loc
  float s, co;
  sincospif(ldexpf((float)k, -(kLog + 3)), &s, &co);
  return {co, -s};
}

// kSpectrum: transform the circulant column of channel `row` and write its spectrum.
// Otherwise: convolve row `row` of u with the spectra and write y.
template <int kLog, bool kSpectrum>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(fftr::Plan<kLog>::T, 2)
conv_cluster(const float* __restrict__ src, const float* __restrict__ src2, int H, int L,
             const float2* __restrict__ tw, float2* __restrict__ spec, float* __restrict__ y) {
  using P = fftr::Plan<kLog>;
  constexpr int nl = P::n;          // points per CTA
  constexpr int n = kC * nl;        // packed points per row
  constexpr int T = P::T;
  constexpr int colsPer = nl / kC;  // F1 / I1 columns per CTA
  extern __shared__ float2 smem[];
  float2* buf = smem;
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / kC;
  const int tid = threadIdx.x;
  const int half = (L + 1) >> 1;
  const uint32_t bufAddr = smem_addr(buf);

  // ---- 0) this CTA's slice of the packed row: z[rank * nl + i] ----
  // All of a thread's loads are issued before the first shared-memory store, so their latency
  // is paid once rather than once per point.
  constexpr int PER = nl / T;
  static_assert(nl % T == 0, "points per thread");
  {
    float2 z[PER];
    if constexpr (kSpectrum) {
      const float* k1 = src + (size_t)row * L;
      const float* k2 = src2 ? src2 + (size_t)row * L : nullptr;
      auto col = [&](int i) -> float {  // circulant column of length 2n
        float v = (i < L) ? __ldg(k1 + i) : 0.f;
        if (k2) {
          if (i == 0) v += __ldg(k2);
          else if (i > 2 * n - L) v += __ldg(k2 + (2 * n - i));
        }
        return v;
      };
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int m = (int)rank * nl + tid + q * T;
        z[q] = make_float2(col(2 * m), col(2 * m + 1));
      }
    } else {
      const float* ur = src + (size_t)row * L;
      const bool even = (L & 1) == 0;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int m = (int)rank * nl + tid + q * T;
        z[q] = make_float2(0.f, 0.f);
        if (m < half) {
          if (even) z[q] = __ldg(reinterpret_cast<const float2*>(ur) + m);
          else z[q] = make_float2(__ldg(ur + 2 * m), (2 * m + 1 < L) ? __ldg(ur + 2 * m + 1) : 0.f);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < PER; ++q)
      if (DLR_IN(padded(tid + q * T), P::buf_elems)) buf[padded(tid + q * T)] = z[q];
  }
  cluster_sync();

  // ---- F1: radix-8 DFT across the cluster, twiddle W_n^{i k1}, output k1 -> CTA k1 ----
  for (int ii = tid; ii < colsPer; ii += T) {
    const int i = (int)rank * colsPer + ii;
    const uint32_t off = 8u * padded(i);
    cf v[8];
#pragma unroll
    for (int c = 0; c < kC; ++c) {
      // the conv input is zero for m >= n/2, i.e. c >= 4
      if (!kSpectrum && c >= kC / 2) {
        v[c] = {0.f, 0.f};
      } else {
        const float2 f = ld_cluster(map_rank(bufAddr, c) + off);
        v[c] = {f.x, f.y};
      }
    }
    fft::dft<8, false>(v);
    float s, co;
    sincospif(-ldexpf((float)i, 1 - (kLog + 3)), &s, &co);  // W_n^i = e^{-2 pi i i / n}
    cf w[8];
    powers8(w, {co, s});
#pragma unroll
    for (int k1 = 0; k1 < kC; ++k1) {
      const cf t = k1 ? cmul(v[k1], w[k1]) : v[k1];
      st_cluster(map_rank(bufAddr, k1) + off, make_float2(t.re, t.im));
    }
  }
  cluster_sync();

  // ---- F2: local FFT over i; CTA k1 = rank then holds Z[k1 + 8 k2] at k2 ----
  local_fft<kLog, false>(buf, tw);
  cluster_sync();  // every CTA's Z is complete before mirrors are read

  const int k1 = (int)rank;
  const uint32_t mirrorRank = (kC - k1) & (kC - 1);
  const uint32_t mirrorBase = map_rank(bufAddr, mirrorRank);
  auto mirror_local = [&](int k2) { return k1 == 0 ? (nl - k2) & (nl - 1) : nl - 1 - k2; };

  if constexpr (kSpectrum) {
    // ---- real spectrum X_k, k = k1 + 8 k2, scaled by 1/(4n), stored in cluster order ----
    const float scale = 1.0f / (float)(4 * n);
    float2* out = spec + (size_t)row * (n + 1);
    constexpr int kBatch = 4;
    static_assert(PER % kBatch == 0, "batches");
#pragma unroll 1
    for (int q0 = 0; q0 < PER; q0 += kBatch) {
      float2 fa[kBatch], fb[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int k2 = tid + (q0 + b) * T;
        const bool in = DLR_IN(padded(mirror_local(k2)), P::buf_elems) && DLR_IN(padded(k2), P::buf_elems);
        fb[b] = in ? ld_cluster(mirrorBase + 8u * padded(mirror_local(k2))) : make_float2(0.f, 0.f);
        fa[b] = in ? buf[padded(k2)] : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int k2 = tid + (q0 + b) * T;
        const int k = k1 + kC * k2;
        const cf E = {0.5f * (fa[b].x + fb[b].x), 0.5f * (fa[b].y - fb[b].y)};
        const cf O = {0.5f * (fa[b].y + fb[b].y), -0.5f * (fa[b].x - fb[b].x)};
        const cf wO = cmul(half_turn_twiddle<kLog>(k), O);
        const cf Xk = cadd(E, wO);
        if (DLR_IN(k1 * nl + k2, n + 1)) out[k1 * nl + k2] = make_float2(Xk.re * scale, Xk.im * scale);
        if (k == 0) {  // X_n = E - O at k = 0
          const cf Xn = {E.re - wO.re, -(E.im - wO.im)};
          out[n] = make_float2(Xn.re * scale, Xn.im * scale);
        }
      }
    }
    cluster_sync();  // mirrors read before any CTA exits
    return;
  } else {
    // ---- spectral step, one thread per pair of bins (k, n - k), in place ----
    // Item p in [0, nl/2) of CTA k1 is the pair (k1, p) <-> (mirror CTA, mirror_local(p)):
    // CTA k1 and its mirror each take the first half of their own positions, which covers
    // the second half of the other's. CTA 0 pairs p with nl - p (p = 0 with itself) and its
    // item 0 also takes position nl/2 (bin n/2, paired with itself); CTA 4 pairs p with
    // nl - 1 - p inside itself.
    const float2* S = spec + (size_t)(row % H) * (n + 1);
    constexpr int kItems = nl / 2 / T;
    constexpr int kBatch = 4;
    static_assert(kItems % kBatch == 0 || kItems < kBatch, "batches");
    constexpr int kB = kItems < kBatch ? kItems : kBatch;
    const bool local_pair = mirrorRank == (uint32_t)k1;
#pragma unroll 1
    for (int q0 = 0; q0 < kItems; q0 += kB) {
      float2 fa[kB], fb[kB], s1[kB], s2[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int p1 = tid + (q0 + b) * T;
        const int p2 = mirror_local(p1);
        const int i2 = (k1 == 0 && p1 == 0) ? n : (int)mirrorRank * nl + p2;
        const bool in = DLR_IN(padded(p1), P::buf_elems) && DLR_IN(padded(p2), P::buf_elems) &&
                        DLR_IN(k1 * nl + p1, n + 1) && DLR_IN(i2, n + 1);
        fa[b] = in ? buf[padded(p1)] : make_float2(0.f, 0.f);
        fb[b] = !in ? make_float2(0.f, 0.f)
                    : local_pair ? buf[padded(p2)] : ld_cluster(mirrorBase + 8u * padded(p2));
        s1[b] = in ? __ldg(&S[k1 * nl + p1]) : make_float2(0.f, 0.f);
        s2[b] = in ? __ldg(&S[i2]) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int p1 = tid + (q0 + b) * T;
        const int p2 = mirror_local(p1);
        const int ka = k1 + kC * p1;                     // bin of p1
        const int kb = (int)mirrorRank + kC * p2;        // bin of p2 = n - ka (mod n)
        if (DLR_IN(padded(p1), P::buf_elems))
          buf[padded(p1)] = spectral_point(fa[b], fb[b], s1[b], s2[b], half_turn_twiddle<kLog>(ka));
        if (!(k1 == 0 && p1 == 0) && DLR_IN(padded(p2), P::buf_elems)) {
          const float2 o2 = spectral_point(fb[b], fa[b], s2[b], s1[b], half_turn_twiddle<kLog>(kb));
          if (local_pair) buf[padded(p2)] = o2;
          else st_cluster(mirrorBase + 8u * padded(p2), o2);
        }
      }
    }
    if (k1 == 0 && tid == 0) {  // bin n/2 at position nl/2 of CTA 0, paired with itself
      const float2 f = buf[padded(nl / 2)];
      const float2 sh = __ldg(&S[nl / 2]);
      buf[padded(nl / 2)] = spectral_point(f, f, sh, sh, half_turn_twiddle<kLog>(n / 2));
    }
    cluster_sync();  // every CTA's inputs of the inverse transform are written

    // ---- I2: local inverse FFT over k2 -> index i ----
    local_fft<kLog, true>(buf, tw);
    cluster_sync();

    // ---- I1: twiddle conj(W_n^{i k1}) and radix-8 inverse DFT across the cluster ----
    float* yr = y + (size_t)row * L;
    const bool even = (L & 1) == 0;
    for (int ii = tid; ii < colsPer; ii += T) {
      const int i = (int)rank * colsPer + ii;
      float s, co;
      sincospif(ldexpf((float)i, 1 - (kLog + 3)), &s, &co);  // W_n^{-i}
      cf w[8];
      powers8(w, {co, s});
      cf v[8];
#pragma unroll
      for (int c = 0; c < kC; ++c) {
        const float2 f = ld_cluster(map_rank(bufAddr, c) + 8u * padded(i));
        v[c] = c ? cmul({f.x, f.y}, w[c]) : cf{f.x, f.y};
      }
      fft::dft<8, true>(v);
#pragma unroll
      for (int c = 0; c < kC / 2; ++c) {  // outputs m = c nl + i < n/2 hold y
        const int m = c * nl + i;
        if (m < half) {
          if (even) {
            reinterpret_cast<float2*>(yr)[m] = make_float2(v[c].re, v[c].im);
          } else {
            yr[2 * m] = v[c].re;
            if (2 * m + 1 < L) yr[2 * m + 1] = v[c].im;
          }
        }
      }
    }
    cluster_sync();  // no CTA exits while others still read its shared memory
  }
}

template <int kLog, bool kSpectrum>
cudaError_t launch_cluster(const float* src, const float* src2, int rows, int H, int L,
                           const float2* tw, float2* spec, float* y, cudaStream_t s) {
  using P = fftr::Plan<kLog>;
  const size_t smem = P::buf_elems * sizeof(float2);
  cudaError_t e = max_smem_once<conv_cluster<kLog, kSpectrum>>(smem);
  if (e != cudaSuccess) return e;
  conv_cluster<kLog, kSpectrum><<<(unsigned)(rows * kC), P::T, smem, s>>>(src, src2, H, L, tw,
                                                                        spec, y);
  return cudaGetLastError();
}

}  // namespace

// n = next power of two >= L lies in (16384, 65536]; n_loc = n / 8 points per CTA.
cudaError_t launch_cluster_spectrum(const float* K1, const float* K2, int H, int L, int lg,
                                    const float2* tw_loc, float2* spec, cudaStream_t s) {
  if (lg == 15) return launch_cluster<12, true>(K1, K2, H, H, L, tw_loc, spec, nullptr, s);
  if (lg == 16) return launch_cluster<13, true>(K1, K2, H, H, L, tw_loc, spec, nullptr, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_cluster_apply(const float* u, int B, int H, int L, int lg,
                                 const float2* tw_loc, const float2* spec, float* y,
                                 cudaStream_t s) {
  float2* sp = const_cast<float2*>(spec);
  if (lg == 15) return launch_cluster<12, false>(u, nullptr, B * H, H, L, tw_loc, sp, y, s);
  if (lg == 16) return launch_cluster<13, false>(u, nullptr, B * H, H, L, tw_loc, sp, y, s);
  return cudaErrorInvalidValue;
}

}  // namespace dlr
