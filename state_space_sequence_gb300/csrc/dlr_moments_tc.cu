// dlr_moments_tc.cu -- the power sums of the parameter gradients on the tensor cores
// ("Simplifying and Understanding State Space Models with Diagonal Linear RNNs", section 2,
// gradient analysis):
//   S0_n = sum_j w_j lambda_n^j,   S1_n = sum_j j w_j lambda_n^j,   j < L,
// with w_j the lag correlation c_j (Re cast) or c_j K_j (DLR-prod cast, K the complex kernel).
//
// Chunked powers, as in the kernel generators but transposed: with j = 64 C + t,
//   S0_n = sum_C lambda_n^{64 C} P[n][C],   P[n][C] = sum_t lambda_n^t w_{64 C + t},
// and S1 the same with the weights j w_j. For 128 states and a block of 32 chunks, P (for both
// weight sets) is one real product [128 states x 128] . [128 x 128] (4 columns per chunk):
//   A[n][k] = Re lambda_n^k (k < 64), Im lambda_n^(k-64);
//   B row (C, Re) = [Re w_t, -Im w_t],  B row (C, Im) = [Im w_t, Re w_t]  (and the same for
//   j w_j), so that A . B^T gives Re P and Im P in adjacent columns,
// run as three kind::f16 MMAs per K step (hi*hi + hi*lo + lo*hi of operands scaled by powers
// of two and split into f16 halves: A by 2^14, each B row so that its largest entry lies near
// 2^13), accumulated in TMEM in float32. The epilogue thread of state n then adds
// lambda_n^{64 C} P[n][C] over the block's chunks; lambda^t and lambda^{64 C} come from
// directly evaluated powers combined by one product (lambda^{8a} lambda^b, lambda^{512a}
// lambda^{64b}).
//
// One CTA of 256 threads per (channel, 128 states), blocks of 32 chunks in a two-deep pipeline:
// all threads write block k + 1's B operand (two buffers) while thread 0's MMAs of block k run
// into one of two TMEM accumulators, then all eight warps read block k's accumulator (thread =
// TMEM lane = state, the two warps of a lane quarter taking half the columns each). Each MMA
// completion is an mbarrier wait bounded by the global timer (DLR_ERR_TIMEOUT on expiry).
#include <cuda_fp16.h>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 15;
namespace {

constexpr int kThreads = 256;
constexpr int kStates = 128;  // MMA M
constexpr int kChunks = 32;   // chunks per block; MMA N = 4 * kChunks
constexpr int kN = 4 * kChunks;
constexpr uint32_t kATile = kStates * 128;  // one K-block (64 f16 per row) of A, bytes
constexpr uint32_t kBTile = kN * 128;       // one K-block of B
constexpr uint32_t kBBuf = 4 * kBTile;      // one B buffer: [2 K-blocks][hi, lo]
// shared memory: A [2 K-blocks][hi, lo], B [2 buffers], their row exponents [2][kN], the
// partial sums of the second column half [kStates][4], barriers [2], TMEM slot
constexpr uint32_t kAOff = 0;
constexpr uint32_t kBOff = kAOff + 4 * kATile;
constexpr uint32_t kEOff = kBOff + 2 * kBBuf;
constexpr uint32_t kPOff = kEOff + 2 * 4 * kN;
constexpr uint32_t kBarOff = kPOff + kStates * 16;
constexpr uint32_t kSlotOff = kBarOff + 16;
constexpr uint32_t kSmemBytes = kSlotOff + 16 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 2 * kN;                 // two accumulators

__device__ __forceinline__ float round11(float a) {
  return __uint_as_float((__float_as_uint(a) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ float exp2i(int s) { return __int_as_float((s + 127) << 23); }

// Eight values of K-major operand row `row` (16-byte chunk `chunk` of its 128-byte line) as the
// f16 pair hi (rounded to 11 significant bits) and lo (the f16 rounding of the remainder).
__device__ __forceinline__ void put8(uint8_t* hi_tile, uint8_t* lo_tile, int row, int chunk,
                                     const float (&v)[8], uint32_t tile_bytes) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float a = v[2 * q], b = v[2 * q + 1];
    const float ah = round11(a), bh = round11(b);
    const __half2 hh = __floats2half2_rn(ah, bh);
    const __half2 ll = __floats2half2_rn(a - ah, b - bh);
    h[q] = *reinterpret_cast<const uint32_t*>(&hh);
    l[q] = *reinterpret_cast<const uint32_t*>(&ll);
  }
  const uint32_t off = uint32_t(row) * 128u + ((uint32_t(chunk) ^ uint32_t(row & 7)) << 4);
  if (DLR_IN(off + 15, tile_bytes)) {
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// exponent e with |m| < 2^e (0 for m = 0), clamped so that the scales stay normal
__device__ __forceinline__ int exp_of(float m) {
  if (!(m > 0.f)) return 0;
  return max(-99, min(100, int((__float_as_uint(m) >> 23) & 0xFFu) - 126));
}

template <bool kProd>
__global__ void __launch_bounds__(kThreads, 1)
    grad_moments_tc(const float* __restrict__ c, const float2* __restrict__ Kc,
                    const float* __restrict__ log_re, const float* __restrict__ log_im,
                    const float2* __restrict__ W, int N, int L, int tiles_per_h,
                    float* __restrict__ d_log_re, float* __restrict__ d_log_im,
                    float2* __restrict__ dW, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* sE = reinterpret_cast<int*>(sm + kEOff);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kSlotOff);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x / tiles_per_h;
  const int n0 = (blockIdx.x - h * tiles_per_h) * kStates;
  const float* ch = c + (size_t)h * (size_t)L;
  const float2* kh = kProd ? Kc + (size_t)h * (size_t)L : nullptr;

  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(slot, kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- A: row r = state n0 + r, lambda^t for t = 32 half .. 32 half + 31, times 2^14 ----
  {
    const int r = tid & (kStates - 1), half = tid >> 7;
    const int n = n0 + r;
    const bool on = n < N;
    const lam_param p = make_lam_param(on ? log_re[(size_t)h * N + n] : 0.f,
                                       on ? log_im[(size_t)h * N + n] : 0.f);
    cf lb[8];  // lambda^b
#pragma unroll
    for (int b = 0; b < 8; ++b) lb[b] = lam_pow(p, b);
    uint8_t* a_re_hi = sm + kAOff;  // K-block 0: the real parts
    uint8_t* a_re_lo = a_re_hi + kATile;
    uint8_t* a_im_hi = a_re_lo + kATile;  // K-block 1: the imaginary parts
    uint8_t* a_im_lo = a_im_hi + kATile;
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // lags t = 32 half + 8 q + b
      const cf la = lam_pow(p, 32 * half + 8 * q);
      float vr[8], vi[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const cf z = cmul(la, lb[b]);
        vr[b] = on ? z.re * 16384.f : 0.f;
        vi[b] = on ? z.im * 16384.f : 0.f;
      }
      put8(a_re_hi, a_re_lo, r, 4 * half + q, vr, kATile);
      put8(a_im_hi, a_im_lo, r, 4 * half + q, vi, kATile);
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  // ---- the epilogue thread: state n0 + r, accumulator columns of chunk half hc ----
  const int r = 32 * (warp & 3) + (tid & 31), hc = warp >> 2;
  const int ns = n0 + r;
  lam_param pe{};
  cf l64[8];  // lambda^{64 b}
  cf s0 = {0.f, 0.f}, s1 = {0.f, 0.f};
  {
    const bool on = ns < N;
    pe = make_lam_param(on ? log_re[(size_t)h * N + ns] : 0.f,
                        on ? log_im[(size_t)h * N + ns] : 0.f);
#pragma unroll
    for (int b = 0; b < 8; ++b) l64[b] = lam_pow(pe, 64 * b);
  }
  const int nchunks = (L + 63) / 64;
  const int nblocks = (nchunks + kChunks - 1) / kChunks;

  // B of block blk into buffer buf: rows 4 cc + kind (kind 0/1: Re/Im rows of w, 2/3: of j w)
  // for chunk 32 blk + cc. Thread (cc, p) loads lags 8p .. 8p + 7 of its chunk once and writes
  // their 16-byte piece of all four rows; the rows' scales come from the chunk's largest |w|
  // and |j w|, reduced over its eight threads (adjacent lanes).
  auto build_b = [&](int blk, int buf) {
    const int cc = tid >> 3, p = tid & 7;
    const int j0 = 64 * (blk * kChunks + cc) + 8 * p;
    float wr[8], wi[8], vr[8], vi[8];  // w_j and j w_j
    float mw = 0.f, mv = 0.f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int j = j0 + b;
      float xr = 0.f, xi = 0.f;
      if (j < L) {
        const float cj = __ldg(ch + j);
        if constexpr (kProd) {
          const float2 kj = __ldg(kh + j);
          xr = cj * kj.x;
          xi = cj * kj.y;
        } else {
          xr = cj;
        }
      }
      wr[b] = xr;
      wi[b] = xi;
      vr[b] = (float)j * xr;
      vi[b] = (float)j * xi;
      mw = fmaxf(mw, fmaxf(fabsf(xr), fabsf(xi)));
      mv = fmaxf(mv, fmaxf(fabsf(vr[b]), fabsf(vi[b])));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
      mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
    }
    const int ew = exp_of(mw), ev = exp_of(mv);  // |entries| < 2^e: scaled by 2^(13 - e)
    const float sw = exp2i(13 - ew), sv = exp2i(13 - ev);
    if (p == 0 && DLR_IN(buf * kN + 4 * cc + 3, 2 * kN)) {
      sE[buf * kN + 4 * cc] = ew;
      sE[buf * kN + 4 * cc + 1] = ew;
      sE[buf * kN + 4 * cc + 2] = ev;
      sE[buf * kN + 4 * cc + 3] = ev;
    }
    uint8_t* b_re_hi = sm + kBOff + buf * kBBuf;  // K-block 0 (multiplies Re lambda^t)
    uint8_t* b_re_lo = b_re_hi + kBTile;
    uint8_t* b_im_hi = b_re_lo + kBTile;  // K-block 1 (multiplies Im lambda^t)
    uint8_t* b_im_lo = b_im_hi + kBTile;
#pragma unroll
    for (int kind = 0; kind < 4; ++kind) {
      const bool jw = kind >= 2, im_row = kind & 1;
      const float* xr = jw ? vr : wr;
      const float* xi = jw ? vi : wi;
      const float sc = jw ? sv : sw;
      float v0[8], v1[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        // Re row: [Re w, -Im w]; Im row: [Im w, Re w]
        v0[b] = (im_row ? xi[b] : xr[b]) * sc;
        v1[b] = (im_row ? xr[b] : -xi[b]) * sc;
      }
      put8(b_re_hi, b_re_lo, 4 * cc + kind, p, v0, kBTile);
      put8(b_im_hi, b_im_lo, 4 * cc + kind, p, v1, kBTile);
    }
  };
  // the three-product MMAs of the block in buffer buf into accumulator buf (thread 0)
  auto issue = [&](int buf) {
    constexpr uint32_t idesc = tc::idesc_f16_f32(kStates, kN);
    const uint32_t d = tmem + uint32_t(buf * kN);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      const uint64_t ah = tc::smem_desc_k_sw128(sm + kAOff + (2 * kb) * kATile);
      const uint64_t al = tc::smem_desc_k_sw128(sm + kAOff + (2 * kb + 1) * kATile);
      const uint64_t bh = tc::smem_desc_k_sw128(sm + kBOff + buf * kBBuf + (2 * kb) * kBTile);
      const uint64_t bl =
          tc::smem_desc_k_sw128(sm + kBOff + buf * kBBuf + (2 * kb + 1) * kBTile);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // 16 f16 = 32 bytes = 2 descriptor units
        tc::mma_kind_f16(d, ah + 2 * kk, bh + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
        tc::mma_kind_f16(d, ah + 2 * kk, bl + 2 * kk, idesc, 1u);
        tc::mma_kind_f16(d, al + 2 * kk, bh + 2 * kk, idesc, 1u);
      }
    }
    tc::mma_commit(&bar[buf]);
  };

  // The pipeline: B of block k + 1 is written while the MMAs of block k run; then every warp
  // reads block k's accumulator. Buffer and accumulator k & 1 are free again once block k - 1's
  // readers passed the barrier that ends its iteration (they waited for its MMAs first).
  bool ok = true;
  build_b(0, 0);
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0 && nblocks > 0) issue(0);
#pragma unroll 1
  for (int blk = 0; blk < nblocks; ++blk) {
    const int buf = blk & 1;
    if (blk + 1 < nblocks) {
      build_b(blk + 1, buf ^ 1);
      tc::fence_proxy_async_smem();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (blk + 1 < nblocks && tid == 0) issue(buf ^ 1);
    ok = ok && tc::mbar_wait(&bar[buf], (blk >> 1) & 1);
    tc::fence_after_sync();
    const int C0 = blk * kChunks + 16 * hc;  // this thread's first chunk of the block
    const uint32_t lane_base = tmem + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(buf * kN);
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {  // chunks C0 + 8 part .. C0 + 8 part + 7
      float v[32];
      tc::tmem_ld32(lane_base + uint32_t(64 * hc + 32 * part), v);
      if (!ok || C0 + 8 * part >= nchunks) continue;
      // lambda^{64 C} = lambda^{512 (C / 8)} lambda^{64 (C % 8)}
      const cf l512 = lam_pow(pe, 512 * ((C0 >> 3) + part));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int cc = 16 * hc + 8 * part + q;  // chunk within the block
        if (C0 + 8 * part + q >= nchunks) break;
        // undo the operand scales: 2^14 (A) and 2^(13 - e) (the B row)
        const float u0 = exp2i(sE[buf * kN + 4 * cc] - 27);
        const float u1 = exp2i(sE[buf * kN + 4 * cc + 2] - 27);
        const cf P = {v[4 * q] * u0, v[4 * q + 1] * u0};
        const cf P1 = {v[4 * q + 2] * u1, v[4 * q + 3] * u1};
        const cf wgt = cmul(l512, l64[q]);
        s0 = cfma(wgt, P, s0);
        s1 = cfma(wgt, P1, s1);
      }
    }
    tc::fence_before_sync();
    __syncthreads();  // accumulator and exponents of buffer buf read: free for block k + 2
  }
  if (!ok) report_status(status, DLR_ERR_TIMEOUT);
  // the two column halves of each state: the second half's sums through shared memory
  float4* sP = reinterpret_cast<float4*>(sm + kPOff);
  if (hc == 1) sP[r] = make_float4(s0.re, s0.im, s1.re, s1.im);
  __syncthreads();
  if (hc == 0 && ns < N && ok) {
    const float4 o = sP[r];
    s0 = {s0.re + o.x, s0.im + o.y};
    s1 = {s1.re + o.z, s1.im + o.w};
    // S0, S1 -> the three gradients
    const size_t hn = (size_t)h * N + ns;
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
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// The power sums and gradients of one parameter set on the tensor cores (see above).
cudaError_t launch_moments_tc(const float* c, const float2* Kc, bool prod, const float* log_re,
                              const float* log_im, const float* W, int H, int N, int L,
                              float* d_log_re, float* d_log_im, float* dW, int* status,
                              cudaStream_t s) {
  const int tiles = (N + kStates - 1) / kStates;
  const unsigned grid = (unsigned)((int64_t)H * tiles);
  const float2* Wc = reinterpret_cast<const float2*>(W);
  float2* dWc = reinterpret_cast<float2*>(dW);
  cudaError_t e;
  if (prod) {
    if ((e = max_smem_once<grad_moments_tc<true>>(kSmemBytes)) != cudaSuccess) return e;
    grad_moments_tc<true><<<grid, kThreads, kSmemBytes, s>>>(c, Kc, log_re, log_im, Wc, N, L,
                                                            tiles, d_log_re, d_log_im, dWc,
                                                            status);
  } else {
    if ((e = max_smem_once<grad_moments_tc<false>>(kSmemBytes)) != cudaSuccess) return e;
    grad_moments_tc<false><<<grid, kThreads, kSmemBytes, s>>>(c, Kc, log_re, log_im, Wc, N, L,
                                                             tiles, d_log_re, d_log_im, dWc,
                                                             status);
  }
  return cudaGetLastError();
}

}  // namespace dlr
