// dlr_kernel.cu -- DLR convolution kernel K_{h,j} = sum_n W_{h,n} lambda_{h,n}^j, cast to
// Re K or Re K * Im K ("Simplifying and Understanding State Space Models with Diagonal Linear
// RNNs", section 2, Eq. 3/4; section 2.1 for the DLR-prod cast; section 2.2 for lambda).
//
// Chunked powers: write j = j0 + c*T + t (T = 64 lags, c < 32 chunks per CTA). Then
//   K_j = sum_n (W_n lambda_n^{j0 + cT}) * lambda_n^t = sum_n A[c][n] * Bm[n][t],
// a complex [32 x N] x [N x 64] product per CTA, done as an FFMA register-tiled GEMM out of
// shared memory (4 chunks x 4 lags per thread).
// The factors come from five directly evaluated powers per state -- lambda, lambda^8,
// lambda^64, lambda^512 and W lambda^{j0} -- combined by short product trees:
//   lambda^t       = lambda^{t mod 8} * (lambda^8)^{floor(t/8)}
//   lambda^{j0+cT} = (lambda^64)^{c mod 8} * W lambda^{j0} (lambda^512)^{floor(c/8)}
// with every small power built from at most three multiplications, so each term of the sum
// is within ~12 roundings of exact, whatever j is (never a j-long multiplication chain).
#include "dlr_common.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 6;
namespace {

constexpr int kT = 64;         // lags per chunk (t)
constexpr int kC = 32;         // chunks per CTA (c)
constexpr int kGroup = 128;    // threads per state group: 16 (t pairs) x 8 (c groups of 4)
constexpr int kThreads = 2 * kGroup;  // two groups split the states, then reduce

// p[e] = x^e for e < 8 from p[1] = x, at most three multiplications deep
__device__ __forceinline__ void small_powers(cf (&p)[8], cf x) {
  p[0] = {1.f, 0.f};
  p[1] = x;
  p[2] = cmul(x, x);
  p[3] = cmul(p[2], x);
  p[4] = cmul(p[2], p[2]);
  p[5] = cmul(p[4], x);
  p[6] = cmul(p[4], p[2]);
  p[7] = cmul(p[4], p[3]);
}

// per state group: A[c][n], Bm[n][t], five evaluations per state, small-power tables, for
// blocks of kNB = 16 states (up to six CTAs per SM, so the whole grid of the usual shapes runs
// in one wave; N >= 256 goes to the tensor-core generator)
template <int kNB>
struct GroupSmem {
  float2 sA[kC][kNB + 1];
  float2 sB[kNB][kT];
  float2 sE[kNB][5];
  float2 sPw[4][kNB][9];  // lambda^t0, lambda^{8 t1}, lambda^{64 c0}, W lambda^{j0 + 512 c1}
};
template <int kNB>
constexpr size_t gen_smem() { return 2 * sizeof(GroupSmem<kNB>); }

// barrier over one state group only (named barriers 1 and 2; 0 is __syncthreads)
__device__ __forceinline__ void group_sync(int g) {
  if (g == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
  else asm volatile("bar.sync 2, 128;" ::: "memory");
}

// kMode: 0 writes Re K, 1 Re K * Im K (DLR-prod), 2 the complex K as float2 pairs.
template <int kMode, int kNB>
__global__ void __launch_bounds__(kThreads)
dlr_kernel_gen(const float* __restrict__ log_re, const float* __restrict__ log_im,
               const float2* __restrict__ W, int N, int L, float* __restrict__ K) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  using GS = GroupSmem<kNB>;
  GS* gs = reinterpret_cast<GS*>(smem_raw);

  const int h = blockIdx.y;
  const int j0 = blockIdx.x * (kT * kC);
  const int g = threadIdx.x / kGroup;   // state group: blocks nb = 32 g, 32 g + 64, ...
  const int tid = threadIdx.x % kGroup;
  const int tx = tid & 15;  // t in {2 tx, 2 tx + 1, 32 + 2 tx, 33 + 2 tx}
  const int ty = tid >> 4;  // c = ty + 8 i, i < 4
  GS& S = gs[g];

  float acc_re[4][4], acc_im[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc_re[i][k] = acc_im[i][k] = 0.f;

  for (int nb = g * kNB; nb < N; nb += 2 * kNB) {
    // 1) five direct evaluations per state
    for (int e = tid; e < kNB * 5; e += kGroup) {
      const int nl = e / 5, which = e % 5, n = nb + nl;
      cf v = {0.f, 0.f};
      if (n < N) {
        const lam_param p = make_lam_param(log_re[(size_t)h * N + n], log_im[(size_t)h * N + n]);
        if (which < 4) {
          v = lam_pow(p, which == 0 ? 1 : (which == 1 ? 8 : (which == 2 ? 64 : 512)));
        } else {
          const float2 w = W[(size_t)h * N + n];
          v = cmul({w.x, w.y}, lam_pow(p, j0));
        }
      }
      S.sE[nl][which] = make_float2(v.re, v.im);
    }
    group_sync(g);
    // 2) small powers, one table per thread: (state nl, table part)
    if (tid < 4 * kNB) {
      const int nl = tid >> 2, part = tid & 3;
      cf p[8];
      if (part < 3) {
        const float2 e = S.sE[nl][part];  // lambda, lambda^8, lambda^64
        small_powers(p, {e.x, e.y});
      } else {
        const float2 ew = S.sE[nl][4], e5 = S.sE[nl][3];
        const cf s512 = {e5.x, e5.y};
        p[0] = {ew.x, ew.y};
        p[1] = cmul(p[0], s512);
        const cf s2 = cmul(s512, s512);
        p[2] = cmul(p[0], s2);
        p[3] = cmul(p[1], s2);
#pragma unroll
        for (int i = 4; i < 8; ++i) p[i] = {0.f, 0.f};
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) S.sPw[part][nl][i] = make_float2(p[i].re, p[i].im);
    }
    group_sync(g);
    // 3) expand (consecutive threads write consecutive entries)
    for (int e = tid; e < kNB * kT; e += kGroup) {
      const int nl = e / kT, t = e % kT;
      const float2 a = S.sPw[0][nl][t & 7], b = S.sPw[1][nl][t >> 3];
      const cf v = cmul({a.x, a.y}, {b.x, b.y});
      S.sB[nl][t] = make_float2(v.re, v.im);
    }
    for (int e = tid; e < kNB * kC; e += kGroup) {
      const int c = e / kNB, nl = e % kNB;
      const float2 a = S.sPw[2][nl][c & 7], b = S.sPw[3][nl][c >> 3];
      const cf v = cmul({a.x, a.y}, {b.x, b.y});
      S.sA[c][nl] = make_float2(v.re, v.im);
    }
    group_sync(g);
    // 4) register-tiled complex GEMM over this block of states (missing states are zero)
#pragma unroll 4
    for (int nl = 0; nl < kNB; ++nl) {
      float2 a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = S.sA[ty + 8 * i][nl];
      const float4 b01 = *reinterpret_cast<const float4*>(&S.sB[nl][2 * tx]);
      const float4 b23 = *reinterpret_cast<const float4*>(&S.sB[nl][32 + 2 * tx]);
      const float2 b[4] = {make_float2(b01.x, b01.y), make_float2(b01.z, b01.w),
                           make_float2(b23.x, b23.y), make_float2(b23.z, b23.w)};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc_re[i][k] = fmaf(a[i].x, b[k].x, fmaf(-a[i].y, b[k].y, acc_re[i][k]));
          if (kMode != 0) acc_im[i][k] = fmaf(a[i].x, b[k].y, fmaf(a[i].y, b[k].x, acc_im[i][k]));
        }
    }
    group_sync(g);
  }

  // 5) the second group hands its partial sums to the first through shared memory
  __syncthreads();
  float* red = reinterpret_cast<float*>(&gs[1]);  // 128 threads x 32 floats
  static_assert(sizeof(GS) >= sizeof(float) * 32 * kGroup, "reduction scratch");
  if (g == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        red[(i * 4 + k) * kGroup + tid] = acc_re[i][k];
        if (kMode != 0) red[(16 + i * 4 + k) * kGroup + tid] = acc_im[i][k];
      }
  }
  __syncthreads();
  if (g == 1) return;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc_re[i][k] += red[(i * 4 + k) * kGroup + tid];
      if (kMode != 0) acc_im[i][k] += red[(16 + i * 4 + k) * kGroup + tid];
    }

  // 6) store: row h, j = j0 + c T + t for t in {2 tx, 2 tx + 1} and {32 + 2 tx, 33 + 2 tx}
  if constexpr (kMode == 2) {
    float2* kc = reinterpret_cast<float2*>(K) + (size_t)h * L;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int jc = j0 + (ty + 8 * i) * kT;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = jc + 32 * (k >> 1) + 2 * tx + (k & 1);
        if (j < L && DLR_IN(j, L)) kc[j] = make_float2(acc_re[i][k], acc_im[i][k]);
      }
    }
    return;
  }
  float* krow = K + (size_t)h * L;
  const bool vec = ((L & 1) == 0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int jc = j0 + (ty + 8 * i) * kT;
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = kMode == 1 ? acc_re[i][k] * acc_im[i][k] : acc_re[i][k];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int j = jc + 32 * half + 2 * tx;
      if (vec && j + 1 < L) {
        *reinterpret_cast<float2*>(krow + j) = make_float2(v[2 * half], v[2 * half + 1]);
      } else {
        if (j < L) krow[j] = v[2 * half];
        if (j + 1 < L) krow[j + 1] = v[2 * half + 1];
      }
    }
  }
}

template <int kMode, int kNB>
cudaError_t launch_gen(const float* log_re, const float* log_im, const float* W, int H, int N,
                       int L, float* K, cudaStream_t s) {
  dim3 grid((L + kT * kC - 1) / (kT * kC), H);
  cudaError_t e = max_smem_once<dlr_kernel_gen<kMode, kNB>>(gen_smem<kNB>());
  if (e != cudaSuccess) return e;
  dlr_kernel_gen<kMode, kNB><<<grid, kThreads, gen_smem<kNB>(), s>>>(
      log_re, log_im, reinterpret_cast<const float2*>(W), N, L, K);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dlr_kernel_tc(const float* log_re, const float* log_im, const float* W, int H,
                                 int N, int L, bool re_im, float* K, int* status,
                                 cudaStream_t s);

// N >= 256 states, or N >= 64 on kernels of 16384 lags or more: the tensor-core generator
// (dlr_kernel_tc.cu; 0.117 ms against 0.162 ms for H = 256, N = 64, L = 65536); otherwise
// this FFMA one.
cudaError_t launch_dlr_kernel(const float* log_re, const float* log_im, const float* W, int H,
                              int N, int L, bool re_im, float* K, int* status, cudaStream_t s) {
  if (N >= 256 || (N >= 64 && L >= 16384))
    return launch_dlr_kernel_tc(log_re, log_im, W, H, N, L, re_im, K, status, s);
  return re_im ? launch_gen<1, 16>(log_re, log_im, W, H, N, L, K, s)
               : launch_gen<0, 16>(log_re, log_im, W, H, N, L, K, s);
}

cudaError_t launch_dlr_kernel_tc_complex(const float* log_re, const float* log_im,
                                         const float* W, int H, int N, int L, float2* K,
                                         int* status, cudaStream_t s);

// The complex kernel K [H, L] as float2 pairs (for the DLR-prod gradients), on the same two
// generators as the casts.
cudaError_t launch_dlr_kernel_complex(const float* log_re, const float* log_im, const float* W,
                                      int H, int N, int L, float2* K, int* status,
                                      cudaStream_t s) {
  if (N >= 256 || (N >= 64 && L >= 16384))
    return launch_dlr_kernel_tc_complex(log_re, log_im, W, H, N, L, K, status, s);
  return launch_gen<2, 16>(log_re, log_im, W, H, N, L, reinterpret_cast<float*>(K), s);
}

}  // namespace dlr
