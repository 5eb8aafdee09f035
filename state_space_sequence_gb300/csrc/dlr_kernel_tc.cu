// dlr_kernel_tc.cu -- the DLR convolution kernel K_{h,j} = sum_n W_{h,n} lambda_{h,n}^j (cast
// Re K or Re K * Im K; "Simplifying and Understanding State Space Models with Diagonal Linear
// RNNs", section 2, Eq. 3/4, section 2.1) on the tensor cores, for many states.
//
// Chunked powers as in the FFMA generator: with j = j0 + 64 c + t (one CTA: 128 chunks c of
// 64 lags t, j0 = 8192 blockIdx.x),
//   K_j = sum_n A[c][n] Bm[n][t],   A[c][n] = W_n lambda_n^{j0 + 64 c},  Bm[n][t] = lambda_n^t,
// a complex [128 x N] x [N x 64] product per CTA. As a real product over K = 2N (Re, Im of each
// state): Re K = A' . [Re Bm, -Im Bm], Im K = A' . [Im Bm, Re Bm] with A' = [Re A, Im A], so one
// MMA of N = 128 columns (64 lags Re | 64 lags Im) gives both.
//
// Precision: every operand x is scaled by a power of two and split into f16 halves
// x_hi + x_lo; each product is hi*hi + hi*lo + lo*hi (three kind::f16 MMAs with f32
// accumulation; lo*lo is below 2^-22 relative). The blocks of states go round-robin into
// four TMEM accumulators, added in float32 at the end, so no accumulator takes more than a
// quarter of the 3 (2N / 16) MMA steps (with N = 1024 one accumulator's rounding drift
// reached 1e-5 of K). A's rows are scaled so the row's largest |A|
// lies below 2^13 (the bound log2|W_n| - a_n^2 j log2(e) maximised over the states in a
// pre-pass); Bm (|lambda^t| <= 1) by 2^14. The factors come from directly evaluated powers
// (lambda, lambda^8, lambda^64, lambda^512, lambda^4096, W lambda^{j0}) combined by product
// trees of depth <= 3, so no term is more than about a dozen roundings from exact.
//
// Roles (288 threads, one CTA per SM): warps 0-7 generate, per block of 32 states, the power
// tables and then the A and Bm tiles straight into the f16 operand layout (K-major, 128-byte
// swizzle) of a 2-stage ring; warp 8 allocates 4 x 128 TMEM columns and one of its threads
// issues the MMAs; warps 0-3 then read the accumulators (thread = chunk row) and store K.
#include <cuda_fp16.h>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
namespace {

constexpr int kT = 64;           // lags per chunk
constexpr int kRows = 128;       // chunks per CTA (MMA M)
constexpr int kSB = 32;          // complex states per K-block (64 f16 = 128 bytes per row)
constexpr int kGen = 256;        // generator threads
constexpr int kThreads = kGen + 32;
constexpr int kStages = 2;
constexpr uint32_t kTile = kRows * 128;          // 128 rows x 128 bytes
constexpr uint32_t kStageBytes = 4 * kTile;      // A hi, A lo, B hi, B lo
constexpr uint32_t kTabOff = kStages * kStageBytes;
constexpr int kDirect = 6;                       // lambda^{1,8,64,512,4096}, W lambda^{j0}
constexpr uint32_t kTabBytes = (kSB * kDirect + 5 * kSB * 8) * 8;
constexpr int kPreChunk = 1024;                  // states per pre-pass pass
constexpr uint32_t kPreOff = kTabOff + kTabBytes;
constexpr uint32_t kScaleOff = kPreOff + kPreChunk * 8;
constexpr uint32_t kBarOff = kScaleOff + 3 * kRows * 4;
constexpr size_t kSmemBytes = 1024 + kBarOff + 64;
constexpr int kAcc = 4;                           // accumulators, K-blocks round-robin
constexpr uint32_t kTmemCols = 128 * kAcc;
constexpr float kLog2e = 1.44269504088896341f;

__device__ __forceinline__ void gen_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGen) : "memory");
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity)) != 0;
}
__device__ __forceinline__ float exp2i(int s) { return __int_as_float((s + 127) << 23); }

// p[e] = x^e for e < 8, at most three multiplications deep
__device__ __forceinline__ void small_powers8(float2* p, cf x) {
  cf q[8];
  q[0] = {1.f, 0.f};
  q[1] = x;
  q[2] = cmul(x, x);
  q[3] = cmul(q[2], x);
  q[4] = cmul(q[2], q[2]);
  q[5] = cmul(q[4], x);
  q[6] = cmul(q[4], q[2]);
  q[7] = cmul(q[4], q[3]);
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = make_float2(q[i].re, q[i].im);
}

// (a, b) scaled by s as f16 pairs: hi = f16(a s, b s), lo = f16 of the remainders
__device__ __forceinline__ void split_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <bool kReIm>
__global__ void __launch_bounds__(kThreads, 1)
dlr_kernel_tc(const float* __restrict__ log_re, const float* __restrict__ log_im,
              const float2* __restrict__ W, int N, int L, float* __restrict__ K, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float2* sE = reinterpret_cast<float2*>(sm + kTabOff);            // [kSB][kDirect]
  float2* sP = sE + kSB * kDirect;                                  // [5][kSB][8]
  float2* sPre = reinterpret_cast<float2*>(sm + kPreOff);           // [kPreChunk]
  float* sMax = reinterpret_cast<float*>(sm + kScaleOff);           // [2][kRows]
  int* sExp = reinterpret_cast<int*>(sm + kScaleOff) + 2 * kRows;   // [kRows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint64_t* full = bars;               // [kStages] tiles written (8 warp arrivals)
  uint64_t* empty = bars + kStages;    // [kStages] tiles consumed by the MMAs
  uint64_t* done = bars + 2 * kStages; // accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int j0 = blockIdx.x * kRows * kT;
  const int nkb = (N + kSB - 1) / kSB;
  const float* lr_h = log_re + (size_t)h * N;
  const float* li_h = log_im + (size_t)h * N;
  const float2* w_h = W + (size_t)h * N;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], kGen / 32);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(done, 1);
    tc::mbar_fence_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp < 8) {
    // ---- row scales: the largest log2|A[c][n]| = log2|W_n| - a_n^2 (j0 + 64 c) log2(e) ----
    const int row = tid & (kRows - 1), half = tid >> 7;
    const float jr = (float)(j0 + row * kT);
    float mx = -INFINITY;
    for (int n0 = 0; n0 < N; n0 += kPreChunk) {
      const int cnt = min(kPreChunk, N - n0);
      gen_sync();
      for (int i = tid; i < cnt; i += kGen) {
        const float lr = lr_h[n0 + i];
        const float2 w = w_h[n0 + i];
        sPre[i] = make_float2(0.5f * log2f(w.x * w.x + w.y * w.y), lr * lr * kLog2e);
      }
      gen_sync();
      for (int i = half; i < cnt; i += 2) mx = fmaxf(mx, fmaf(-sPre[i].y, jr, sPre[i].x));
    }
    sMax[half * kRows + row] = mx;
    gen_sync();
    if (half == 0) {
      const float m = fmaxf(sMax[row], sMax[kRows + row]);
      sExp[row] = (m > -1e30f) ? max(-100, min(100, 13 - (int)ceilf(m))) : 0;
    }
    gen_sync();

    // ---- K-blocks of 32 states ----
    const uint32_t sw = uint32_t(row & 7);
    const float a_scale = exp2i(sExp[row]);
    // every generator warp runs every iteration (the named barriers count all 256 threads);
    // after a failed wait a warp only stops writing tiles
    for (int kb = 0; kb < nkb; ++kb) {
      const int n0 = kb * kSB, s = kb % kStages;
      // direct powers of each state
      if (tid < kSB * kDirect) {
        const int nl = tid / kDirect, which = tid % kDirect, n = n0 + nl;
        cf v = {0.f, 0.f};
        if (n < N) {
          const lam_param p = make_lam_param(lr_h[n], li_h[n]);
          if (which < 5) {
            v = lam_pow(p, which == 0 ? 1 : which == 1 ? 8 : which == 2 ? 64 : which == 3 ? 512
                                                                                      : 4096);
          } else {
            const float2 w = w_h[n];
            v = cmul({w.x, w.y}, lam_pow(p, j0));
          }
        }
        sE[nl * kDirect + which] = make_float2(v.re, v.im);
      }
      gen_sync();
      // small-power tables: part 0..3 = (lambda, lambda^8, lambda^64, lambda^512)^{0..7},
      // part 4 = W lambda^{j0} (lambda^4096)^{0, 1}
      if (tid < kSB * 5) {
        const int nl = tid / 5, part = tid % 5;
        float2* dst = sP + (part * kSB + nl) * 8;
        if (part < 4) {
          const float2 e = sE[nl * kDirect + part];
          small_powers8(dst, {e.x, e.y});
        } else {
          const float2 e = sE[nl * kDirect + 5], f = sE[nl * kDirect + 4];
          const cf b = cmul({e.x, e.y}, {f.x, f.y});
          dst[0] = e;
          dst[1] = make_float2(b.re, b.im);
        }
      }
      gen_sync();
      if (ok && kb >= kStages) ok = warp_wait(&empty[s], ((kb / kStages) - 1) & 1);
      if (!ok) continue;
      uint8_t* st = sm + s * kStageBytes;
      // A: row c = chunk, 16 states of this thread's half; each state's (Re, Im) = 4 bytes
      {
        const int c = row, c0 = c & 7, c1 = (c >> 3) & 7, c2 = c >> 6;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 16-byte chunk 4 half + q: states 16 half + 4 q + i
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int nl = half * 16 + q * 4 + i;
            const float2 pw = sP[(4 * kSB + nl) * 8 + c2];
            const float2 p64 = sP[(2 * kSB + nl) * 8 + c0];
            const float2 p512 = sP[(3 * kSB + nl) * 8 + c1];
            const cf a = cmul(cmul({pw.x, pw.y}, {p512.x, p512.y}), {p64.x, p64.y});
            split_h2(a.re * a_scale, a.im * a_scale, hi[i], lo[i]);
          }
          const uint32_t off = uint32_t(row) * 128u + (((uint32_t(half * 4 + q)) ^ sw) << 4);
          *reinterpret_cast<uint4*>(st + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(st + kTile + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      // Bm: row r = lag t (r < 64: the Re-part row [Re, -Im]; r >= 64: the Im-part row
      // [Im, Re] of lag r - 64), scaled by 2^14
      {
        const int t = row & 63;
        const bool imrow = row >= 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int nl = half * 16 + q * 4 + i;
            const float2 p1 = sP[(0 * kSB + nl) * 8 + (t & 7)];
            const float2 p8 = sP[(1 * kSB + nl) * 8 + (t >> 3)];
            const cf b = cmul({p1.x, p1.y}, {p8.x, p8.y});
            const float x = 16384.f * (imrow ? b.im : b.re);
            const float y = 16384.f * (imrow ? b.re : -b.im);
            split_h2(x, y, hi[i], lo[i]);
          }
          const uint32_t off = uint32_t(row) * 128u + (((uint32_t(half * 4 + q)) ^ sw) << 4);
          *reinterpret_cast<uint4*>(st + 2 * kTile + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(st + 3 * kTile + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&full[s]);
    }
  } else if (lane == 0) {
    // ---- MMA issuer ----
    constexpr uint32_t idesc = tc::idesc_f16_f32(kRows, 128);
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % kStages;
      if (!(ok = tc::mbar_wait(&full[s], (kb / kStages) & 1))) break;
      tc::fence_after_sync();
      const uint8_t* st = sm + s * kStageBytes;
      const uint32_t d = tmem + uint32_t(kb % kAcc) * 128u;
      const uint32_t first = kb < kAcc ? 0u : 1u;  // accumulate after the first block
      const uint64_t ah = tc::smem_desc_k_sw128(st), al = tc::smem_desc_k_sw128(st + kTile);
      const uint64_t bh = tc::smem_desc_k_sw128(st + 2 * kTile);
      const uint64_t bl = tc::smem_desc_k_sw128(st + 3 * kTile);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // 16 f16 = 32 bytes = 2 descriptor units
        tc::mma_kind_f16(d, ah + 2 * kk, bh + 2 * kk, idesc, kk ? 1u : first);
        tc::mma_kind_f16(d, ah + 2 * kk, bl + 2 * kk, idesc, 1);
        tc::mma_kind_f16(d, al + 2 * kk, bh + 2 * kk, idesc, 1);
      }
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(done);
  }

  // ---- epilogue: warps 0-3, thread = chunk row c (TMEM lane c) ----
  if (warp < 4) {
    const bool acc_ok = ok && warp_wait(done, 0);
    tc::fence_after_sync();
    const int c = tid;
    const float unscale = exp2i(-(sExp[c] + 14));
    float* krow = K + (size_t)h * L;
    const int jc = j0 + c * kT;
    const bool vec = (L & 3) == 0;
    // accumulators that received a block (nkb may be below kAcc)
    const int nacc = min(kAcc, nkb);
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    auto sum_acc = [&](uint32_t col, float (&out)[32]) {
      tc::tmem_ld32(lane_base + col, out);
      for (int a = 1; a < nacc; ++a) {
        float t[32];
        tc::tmem_ld32(lane_base + uint32_t(a) * 128u + col, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) out[i] += t[i];
      }
    };
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {  // lags 32 part .. 32 part + 31
      float re[32];
      sum_acc(uint32_t(part * 32), re);
      float v[32];
      if (kReIm) {
        float im[32];
        sum_acc(uint32_t(64 + part * 32), im);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = (re[i] * unscale) * (im[i] * unscale);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = re[i] * unscale;
      }
      if (!acc_ok) continue;
      const int jb = jc + part * 32;
      if (vec && jb + 32 <= L) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(krow + jb + 4 * i) =
              make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      } else {
        for (int i = 0; i < 32; ++i)
          if (jb + i < L) krow[jb + i] = v[i];
      }
    }
  }
  if (!ok) report_status(status, DLR_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_dlr_kernel_tc(const float* log_re, const float* log_im, const float* W, int H,
                                 int N, int L, bool re_im, float* K, int* status,
                                 cudaStream_t s) {
  dim3 grid((L + kRows * kT - 1) / (kRows * kT), H);
  const float2* w2 = reinterpret_cast<const float2*>(W);
  cudaError_t e;
  if (re_im) {
    if ((e = max_smem_once<dlr_kernel_tc<true>>(kSmemBytes)) != cudaSuccess) return e;
    dlr_kernel_tc<true><<<grid, kThreads, kSmemBytes, s>>>(log_re, log_im, w2, N, L, K, status);
  } else {
    if ((e = max_smem_once<dlr_kernel_tc<false>>(kSmemBytes)) != cudaSuccess) return e;
    dlr_kernel_tc<false><<<grid, kThreads, kSmemBytes, s>>>(log_re, log_im, w2, N, L, K, status);
  }
  return cudaGetLastError();
}

}  // namespace dlr
