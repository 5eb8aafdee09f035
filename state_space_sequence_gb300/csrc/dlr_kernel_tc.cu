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
// Roles (416 threads, one CTA per SM), joined by mbarriers:
//   warps 0-3   tables, one block of 32 states ahead, into a double buffer: the directly
//               evaluated powers, then per state (lambda, lambda^8, lambda^64)^{0..7} and
//               W lambda^{j0 + 512 c1 + 4096 c2} for the 16 (c1, c2) of the tile's chunks;
//   warps 4-11  tiles: A[c][n] = (W lambda^{j0 + 512 c1 + 4096 c2}) (lambda^64)^{c0} (c = c0 +
//               8 c1 + 64 c2) and Bm[n][t] = lambda^{t mod 8} (lambda^8)^{t / 8}, scaled, split
//               into f16 halves and written straight into the operand layout (K-major,
//               128-byte swizzle) of a 2-stage ring; warps 4-7 then read the accumulators
//               (thread = chunk row) and store K;
//   warp 12     allocates 4 x 128 TMEM columns; one of its threads issues the MMAs.
#include <cuda_fp16.h>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 7;
namespace {

constexpr int kT = 64;           // lags per chunk
constexpr int kRows = 128;       // chunks per CTA (MMA M)
constexpr int kSB = 32;          // complex states per K-block (64 f16 = 128 bytes per row)
constexpr int kTab = 128;        // table threads (warps 0-3)
constexpr int kGen = 256;        // tile threads (warps 4-11)
constexpr int kThreads = kTab + kGen + 32;
constexpr int kStages = 2;
constexpr uint32_t kTile = kRows * 128;          // 128 rows x 128 bytes
constexpr uint32_t kStageBytes = 4 * kTile;      // A hi, A lo, B hi, B lo
// table buffer: (lambda, lambda^8, lambda^64)^e [3][kSB][8], W lambda^{j0+512 c1+4096 c2}
// [kSB][16]
constexpr uint32_t kPOff = 0, kQOff = 3 * kSB * 8 * 8;
constexpr uint32_t kTabBuf = kQOff + kSB * 16 * 8;
constexpr uint32_t kTabOff = kStages * kStageBytes;
constexpr int kDirect = 6;                       // lambda^{1,8,64,512,4096}, W lambda^{j0}
// table warps' scratch: direct powers [kSB][6], small powers [5][kSB][8]
constexpr uint32_t kScrOff = kTabOff + 2 * kTabBuf;
constexpr uint32_t kScrBytes = (kSB * kDirect + 5 * kSB * 8) * 8;
constexpr int kPreChunk = 1024;                  // states per pre-pass pass
constexpr uint32_t kPreOff = kScrOff + kScrBytes;
constexpr uint32_t kScaleOff = kPreOff + kPreChunk * 8;
constexpr uint32_t kBarOff = kScaleOff + 3 * kRows * 4;
constexpr size_t kSmemBytes = 1024 + kBarOff + 128;
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr int kAcc = 4;                           // accumulators, K-blocks round-robin
constexpr uint32_t kTmemCols = 128 * kAcc;
constexpr float kLog2e = 1.44269504088896341f;

__device__ __forceinline__ void tile_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGen) : "memory");
}
__device__ __forceinline__ void tab_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kTab) : "memory");
}
// Bounded wait by a whole warp with one verdict for its lanes; the tries may suspend the warp,
// which keeps waiting warps off the issue slots the table and tile warps need.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, tc::mbar_wait_sleep(bar, parity)) != 0;
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

// v * (s, s) as an f16 pair: hi = f16 of the scaled values, lo = f16 of the remainders; the
// scaling and the remainders in two-wide float instructions (each lane rounds as the scalar
// operation would).
__device__ __forceinline__ void split_h2s(float2 v, float s, uint32_t& hi, uint32_t& lo) {
  const float2 x = __fmul2_rn(v, make_float2(s, s));
  const __half2 h = __floats2half2_rn(x.x, x.y);
  const float2 f = __half22float2(h);
  const float2 r = __ffma2_rn(f, make_float2(-1.f, -1.f), x);  // x - f
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float2 f2mul(float2 a, float2 b) {
  const cf r = cmul({a.x, a.y}, {b.x, b.y});
  return make_float2(r.re, r.im);
}

// kMode: 0 writes Re K, 1 Re K * Im K (DLR-prod), 2 the complex K as float2 pairs.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
dlr_kernel_tc(const float* __restrict__ log_re, const float* __restrict__ log_im,
              const float2* __restrict__ W, int N, int L, float* __restrict__ K, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float2* sE = reinterpret_cast<float2*>(sm + kScrOff);            // [kSB][kDirect]
  float2* sSp = sE + kSB * kDirect;                                 // [5][kSB][8]
  float2* sPre = reinterpret_cast<float2*>(sm + kPreOff);           // [kPreChunk]
  float* sMax = reinterpret_cast<float*>(sm + kScaleOff);           // [2][kRows]
  int* sExp = reinterpret_cast<int*>(sm + kScaleOff) + 2 * kRows;   // [kRows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint64_t* full = bars;                 // [kStages] tiles written (8 warp arrivals)
  uint64_t* empty = bars + kStages;      // [kStages] tiles consumed by the MMAs
  uint64_t* done = bars + 2 * kStages;   // accumulators complete
  uint64_t* tab_full = done + 1;         // [2] table buffer written (2 warp arrivals)
  uint64_t* tab_empty = tab_full + 2;    // [2] table buffer read (8 warp arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tab_empty + 2);

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
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tab_full[b], kTab / 32);
      tc::mbar_init(&tab_empty[b], kGen / 32);
    }
    tc::mbar_fence_init();
  }
  if (warp == 12) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp < 4) {
    // ---- tables, one block of states ahead of the tiles ----
    // every table warp runs every iteration (the named barriers count both); after a failed
    // wait a warp only stops writing the shared buffer
    // the parameters of this thread's (at most two) direct-power items, fetched one block
    // ahead so the loads from L2 overlap the current block's work
    constexpr int kItems = (kSB * kDirect + kTab - 1) / kTab;
    float par_r[kItems], par_i[kItems];
    float2 par_w[kItems];
    auto fetch = [&](int kb, float (&r)[kItems], float (&im)[kItems], float2 (&w)[kItems]) {
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        const int item = tid + k * kTab, n = kb * kSB + item / kDirect;
        const bool in = item < kSB * kDirect && kb < nkb && n < N;
        r[k] = in ? lr_h[n] : 0.f;
        im[k] = in ? li_h[n] : 0.f;
        w[k] = in && item % kDirect == 5 ? w_h[n] : make_float2(0.f, 0.f);
      }
    };
    fetch(0, par_r, par_i, par_w);
    for (int kb = 0; kb < nkb; ++kb) {
      const int n0 = kb * kSB, b = kb & 1;
      float2* buf = reinterpret_cast<float2*>(sm + kTabOff + b * kTabBuf);
      float nx_r[kItems], nx_i[kItems];
      float2 nx_w[kItems];
      fetch(kb + 1, nx_r, nx_i, nx_w);
      // direct powers: 32 states x 6
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        const int item = tid + k * kTab;
        if (item >= kSB * kDirect) break;
        const int nl = item / kDirect, which = item % kDirect, n = n0 + nl;
        cf v = {0.f, 0.f};
        if (n < N) {
          const lam_param p = make_lam_param(par_r[k], par_i[k]);
          if (which < 5) {
            v = lam_pow(p, which == 0 ? 1 : which == 1 ? 8 : which == 2 ? 64 : which == 3 ? 512
                                                                                      : 4096);
          } else {
            v = cmul({par_w[k].x, par_w[k].y}, lam_pow(p, j0));
          }
        }
        sE[item] = make_float2(v.re, v.im);
      }
#pragma unroll
      for (int k = 0; k < kItems; ++k) {
        par_r[k] = nx_r[k];
        par_i[k] = nx_i[k];
        par_w[k] = nx_w[k];
      }
      tab_sync();
      // small powers: parts 0..3 = (lambda, lambda^8, lambda^64, lambda^512)^{0..7};
      // part 4 = W lambda^{j0} (lambda^4096)^{0, 1}
      for (int item = tid; item < kSB * 5; item += kTab) {
        const int part = item / kSB, nl = item % kSB;
        float2* dst = sSp + (part * kSB + nl) * 8;
        if (part < 4) {
          const float2 e = sE[nl * kDirect + part];
          small_powers8(dst, {e.x, e.y});
        } else {
          const float2 e = sE[nl * kDirect + 5], f = sE[nl * kDirect + 4];
          dst[0] = e;
          dst[1] = f2mul(e, f);
        }
      }
      tab_sync();
      if (ok && kb >= 2) ok = warp_wait(&tab_empty[b], ((kb >> 1) - 1) & 1);
      if (ok) {
        float2* pt = buf + kPOff / 8;
        float2* q = buf + kQOff / 8;
        for (int item = tid; item < 3 * kSB * 8; item += kTab) pt[item] = sSp[item];
        for (int item = tid; item < kSB * 16; item += kTab) {  // W lambda^{j0+512 c1+4096 c2}
          const int nl = item >> 4, k = item & 15;
          q[item] = f2mul(sSp[(4 * kSB + nl) * 8 + (k >> 3)], sSp[(3 * kSB + nl) * 8 + (k & 7)]);
        }
      }
      __syncwarp();
      if (ok && lane == 0) tc::mbar_arrive(&tab_full[b]);
      tab_sync();  // the scratch is rewritten by the next iteration
    }
  } else if (warp < 12) {
    // ---- row scales: the largest log2|A[c][n]| = log2|W_n| - a_n^2 (j0 + 64 c) log2(e) ----
    const int tt = tid - kTab;
    const int row = tt & (kRows - 1), half = tt >> 7;
    const float jr = (float)(j0 + row * kT);
    float mx = -INFINITY;
    for (int n0 = 0; n0 < N; n0 += kPreChunk) {
      const int cnt = min(kPreChunk, N - n0);
      tile_sync();
      for (int i = tt; i < cnt; i += kGen) {
        const float lr = lr_h[n0 + i];
        const float2 w = w_h[n0 + i];
        sPre[i] = make_float2(0.5f * log2f(w.x * w.x + w.y * w.y), lr * lr * kLog2e);
      }
      tile_sync();
      for (int i = half; i < cnt; i += 2) mx = fmaxf(mx, fmaf(-sPre[i].y, jr, sPre[i].x));
    }
    sMax[half * kRows + row] = mx;
    tile_sync();
    if (half == 0) {
      const float m = fmaxf(sMax[row], sMax[kRows + row]);
      sExp[row] = (m > -1e30f) ? max(-100, min(100, 13 - (int)ceilf(m))) : 0;
    }
    tile_sync();

    // ---- tiles ----
    const uint32_t sw = uint32_t(row & 7);
    const float a_scale = exp2i(sExp[row]);
    const int c = row, cq = c >> 3, c0 = c & 7;  // A row: chunk c
    const int t = row & 63;                       // Bm row: lag t, Re (row < 64) or Im part
    const bool imrow = row >= 64;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb & 1;
      if (ok) ok = warp_wait(&tab_full[s], (kb >> 1) & 1);
      if (ok && kb >= kStages) ok = warp_wait(&empty[s], ((kb >> 1) - 1) & 1);
      if (!ok) continue;
      const float2* buf = reinterpret_cast<const float2*>(sm + kTabOff + s * kTabBuf);
      const float2* p1 = buf + kPOff / 8;   // [kSB][8] lambda^e
      const float2* p8 = p1 + kSB * 8;      // (lambda^8)^e
      const float2* p64 = p8 + kSB * 8;     // (lambda^64)^e
      const float2* q = buf + kQOff / 8;
      uint8_t* st = sm + s * kStageBytes;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {  // 16-byte chunk 4 half + qq: states 16 half + 4 qq + i
        uint32_t ahi[4], alo[4], bhi[4], blo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nl = DLR_IN(half * 16 + qq * 4 + i, kSB) ? half * 16 + qq * 4 + i : 0;
          const float2 a = f2mul(q[nl * 16 + cq], p64[nl * 8 + c0]);
          split_h2s(a, a_scale, ahi[i], alo[i]);
          const float2 l = f2mul(p1[nl * 8 + (t & 7)], p8[nl * 8 + (t >> 3)]);
          split_h2s(imrow ? make_float2(l.y, l.x) : make_float2(l.x, -l.y), 16384.f, bhi[i],
                    blo[i]);
        }
        const uint32_t off = uint32_t(row) * 128u + (((uint32_t(half * 4 + qq)) ^ sw) << 4);
        if (!DLR_IN(off + 15, kTile)) continue;
        *reinterpret_cast<uint4*>(st + off) = make_uint4(ahi[0], ahi[1], ahi[2], ahi[3]);
        *reinterpret_cast<uint4*>(st + kTile + off) = make_uint4(alo[0], alo[1], alo[2], alo[3]);
        *reinterpret_cast<uint4*>(st + 2 * kTile + off) =
            make_uint4(bhi[0], bhi[1], bhi[2], bhi[3]);
        *reinterpret_cast<uint4*>(st + 3 * kTile + off) =
            make_uint4(blo[0], blo[1], blo[2], blo[3]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&full[s]);
        tc::mbar_arrive(&tab_empty[s]);
      }
    }
  } else if (lane == 0) {
    // ---- MMA issuer ----
    constexpr uint32_t idesc = tc::idesc_f16_f32(kRows, 128);
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % kStages;
      if (!(ok = tc::mbar_wait_sleep(&full[s], (kb / kStages) & 1))) break;
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

  // ---- epilogue: warps 4-7, thread = chunk row c (TMEM lane c) ----
  if (warp >= 4 && warp < 8) {
    const bool acc_ok = ok && warp_wait(done, 0);
    tc::fence_after_sync();
    const int q4 = warp & 3, c = q4 * 32 + lane;
    const float unscale = exp2i(-(sExp[c] + 14));
    float* krow = K + (size_t)h * L;
    const int jc = j0 + c * kT;
    const bool vec = (L & 3) == 0;
    // accumulators that received a block (nkb may be below kAcc)
    const int nacc = min(kAcc, nkb);
    const uint32_t lane_base = tmem + (uint32_t(q4 * 32) << 16);
    auto sum_acc = [&](uint32_t col, float (&out)[32]) {
      tc::tmem_ld32(lane_base + col, out);
      for (int a = 1; a < nacc; ++a) {
        float tv[32];
        tc::tmem_ld32(lane_base + uint32_t(a) * 128u + col, tv);
#pragma unroll
        for (int i = 0; i < 32; ++i) out[i] += tv[i];
      }
    };
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {  // lags 32 part .. 32 part + 31
      float re[32];
      sum_acc(uint32_t(part * 32), re);
      if constexpr (kMode == 2) {
        float im[32];
        sum_acc(uint32_t(64 + part * 32), im);
        if (!acc_ok) continue;
        const int jb = jc + part * 32;
        float2* kc = reinterpret_cast<float2*>(K) + (size_t)h * L;
        if ((L & 1) == 0 && jb + 32 <= L) {  // 16-byte aligned pairs of lags
#pragma unroll
          for (int i = 0; i < 16; ++i)
            *reinterpret_cast<float4*>(kc + jb + 2 * i) =
                make_float4(re[2 * i] * unscale, im[2 * i] * unscale, re[2 * i + 1] * unscale,
                            im[2 * i + 1] * unscale);
        } else {
          for (int i = 0; i < 32; ++i)
            if (jb + i < L) kc[jb + i] = make_float2(re[i] * unscale, im[i] * unscale);
        }
        continue;
      }
      float v[32];
      if (kMode == 1) {
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
  if (warp == 12) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_dlr_kernel_tc(const float* log_re, const float* log_im, const float* W, int H,
                                 int N, int L, bool re_im, float* K, int* status,
                                 cudaStream_t s) {
  dim3 grid((L + kRows * kT - 1) / (kRows * kT), H);
  const float2* w2 = reinterpret_cast<const float2*>(W);
  cudaError_t e;
  if (re_im) {
    if ((e = max_smem_once<dlr_kernel_tc<1>>(kSmemBytes)) != cudaSuccess) return e;
    dlr_kernel_tc<1><<<grid, kThreads, kSmemBytes, s>>>(log_re, log_im, w2, N, L, K, status);
  } else {
    if ((e = max_smem_once<dlr_kernel_tc<0>>(kSmemBytes)) != cudaSuccess) return e;
    dlr_kernel_tc<0><<<grid, kThreads, kSmemBytes, s>>>(log_re, log_im, w2, N, L, K, status);
  }
  return cudaGetLastError();
}

// The complex kernel K [H, L] as float2 pairs.
cudaError_t launch_dlr_kernel_tc_complex(const float* log_re, const float* log_im,
                                         const float* W, int H, int N, int L, float2* K,
                                         int* status, cudaStream_t s) {
  dim3 grid((L + kRows * kT - 1) / (kRows * kT), H);
  cudaError_t e = max_smem_once<dlr_kernel_tc<2>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  dlr_kernel_tc<2><<<grid, kThreads, kSmemBytes, s>>>(
      log_re, log_im, reinterpret_cast<const float2*>(W), N, L, reinterpret_cast<float*>(K),
      status);
  return cudaGetLastError();
}

}  // namespace dlr
