// dlr_scan_tc.cu -- the DLR layer ("Simplifying and Understanding State Space Models with
// Diagonal Linear RNNs", section 2, Eq. 1 with the Re cast)
//     x_{n,k} = lambda_n x_{n,k-1} + u_k,      y_k = sum_n Re(W_n x_{n,k})
// evaluated as a chunked scan ("Simplified State Space Layers for Sequence Modeling", section
// 2.2: the recurrence is a scan under an associative operator) whose three dense contractions
// run on the 5th-generation tensor cores.
//
// Chunks of T = 64 steps; a tile is 128 chunks of one channel h (columns g). For chunk g with
// samples u_{g,t}:
//   1. chunk-end states from a zero start (GEMM, M = 2N = 128 state rows, N = 128 chunks,
//      K = 64):      S[r, g] = sum_t Q[r, t] u_{g,t},   Q[2n|2n+1, t] = Re|Im lambda_n^{63-t}
//   2. carries (fp32, registers): X_g = mu X_{g-1} + S_g (mu = lambda^64) along the chunks of
//      a row; Xin_g = X_{g-1} is the state just before chunk g (zero at the start of a row).
//      The float mu differs from lambda^64 by a rounding that a plain chain would compound once
//      per chunk; so every 32 chunks the chain is re-anchored: with A the state at the previous
//      anchor, X += (lambda^2048 - mu^32) A, where lambda^2048 is evaluated directly and mu^32
//      in two-float arithmetic. The chain then carries at most 31 roundings of mu plus one
//      rounding of lambda^2048 per 32 chunks.
//   3. outputs (two GEMMs, M = 128 chunks, N = 64 steps):
//        Y1[g, t] = sum_s u_{g,s} K_{t-s}                      (K_j = Re sum_n W_n lambda_n^j)
//        Y2[g, t] = sum_r Xin[g, r] G[t, r],  G[t, 2n|2n+1] = Re|-Im (W_n lambda_n^{t+1})
//      y_{g,t} = Y1 + Y2.
// Work per output element: 2N (step 1) + T (Y1) + 2N (Y2) multiply-adds = 320 at N = 64.
//
// Precision: every operand is split into two f16 halves a = a_hi + a_lo (a_lo = the f16
// rounding of a - a_hi), and each product is hi*hi + hi*lo + lo*hi (three MMAs, f32
// accumulation in tensor memory; the dropped lo*lo term is below 2^-22 relative). Before the
// split every operand is scaled by a power of two so that its largest entry lies in
// [2^13, 2^14): per chunk for u, per batch row and tile for Xin, per channel for K and G,
// 2^14 for Q (|Q| <= 1), so that one row's scale never depends on another row's magnitude.
// The scalings are exact and undone in fp32 when S is read and when y is written.
// Powers lambda^j are evaluated from an exactly reduced phase (lam_pow) for j = 8a and j < 8
// and combined by one complex product, so no power carries a long multiplication chain.
//
// One CTA per SM (persistent), 4 warps; thread i owns TMEM lane i: a state row r in step 2,
// a chunk g in the u conversion and the output epilogue. Thread 0 issues the MMAs.
// Units of work: a tile holds floor(128 / C) whole rows when a row has C <= 128 chunks
// (several batch rows of one channel), otherwise one row walks its tiles in order and carries
// its state from tile to tile. Per-channel tables are rebuilt when the channel changes.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
namespace {

constexpr int kT = 64;        // steps per chunk
constexpr int kCols = 128;    // chunks per tile
constexpr int kThreads = 128;
constexpr int kNMax = 64;     // complex states (2N real rows of the state GEMM)
constexpr int kPw = kT + 1;   // powers lambda^0 .. lambda^64
constexpr uint32_t kTmemCols = 256;  // S: 0..127, Y1: 128..191, Y2: 192..255

// shared memory (bytes from a 1024-byte aligned base); f16 tiles in the K-major 128-byte
// swizzled layout (rows of 64 elements, 8-row atoms of 1024 bytes, 16-byte chunk index XOR
// (row & 7)); K = 128 operands are two such tiles ("K-blocks") one after the other
constexpr uint32_t kQHi = 0, kQLo = 16384;         // Q        [128 rows x 64]
constexpr uint32_t kUHi = 32768, kULo = 49152;     // u chunks [128 chunks x 64]
constexpr uint32_t kXHi = 65536, kXLo = 98304;     // Xin      [128 chunks x 128]
constexpr uint32_t kTkHi = 131072, kTkLo = 139264; // Toeplitz [64 t x 64 s]
constexpr uint32_t kGHi = 147456, kGLo = 163840;   // G        [64 t x 128]
constexpr uint32_t kInvU = 180224;                 // float[128]: 2^-14 / (u scale of chunk g)
constexpr uint32_t kRed = kInvU + 512;             // float[8] reductions
constexpr uint32_t kKtap = kRed + 64;              // float[64] K_0..K_63
constexpr uint32_t kPar = kKtap + 256;             // lam_param[64]
constexpr uint32_t kWs = kPar + 64 * sizeof(lam_param);  // float2[64]
constexpr uint32_t kDelta = kWs + 512;             // float2[64] lambda^2048 - mu^32
constexpr uint32_t kRowMax = kDelta + 512;         // float[128][4] per-row, per-warp max |Xin|
constexpr uint32_t kColSx = kRowMax + 2048;        // float[128] Xin scale of chunk g
constexpr uint32_t kBar = (kColSx + 512 + 7) & ~7u; // mbarrier
constexpr uint32_t kSlot = kBar + 8;               // TMEM base address
constexpr uint32_t kEnd = kSlot + 8;
constexpr size_t kSmemBytes = kEnd + 1024;         // + alignment slack
// scratch while building the per-channel tables (inside the Xin region, which is idle then)
constexpr uint32_t kPow = kXHi;                          // float2 [64][65] lambda_n^j
constexpr uint32_t kPow8 = kPow + kNMax * kPw * 8;       // float2 [64][9]  lambda_n^{8a}
constexpr uint32_t kPow1 = kPow8 + kNMax * 9 * 8;        // float2 [64][8]  lambda_n^b
static_assert(kPow1 + kNMax * 8 * 8 <= kTkHi, "table scratch must fit the Xin region");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct TcScanArgs {
  const float* u;
  float* y;
  const float* log_re;
  const float* log_im;
  const float2* W;
  int B, H, N, L;
  int C;            // chunks per row
  int R;            // rows per tile (C <= 128), 0: one row per unit, walked tile by tile
  int tiles_per_h;  // ceil(B / R) when R > 0
  int units;
  int* status;
};

// 2^(14 - e) for the e with m < 2^e (1 for m = 0), so that m times it lies below 2^14; the
// exponent is clamped so that the scale and its inverse are normal floats.
__device__ __forceinline__ int scale_exp(float m) {
  if (!(m > 0.f)) return 0;
  const int e = ((__float_as_int(m) >> 23) & 0xFF) - 126;
  return max(-126, min(126, 14 - e));
}
__device__ __forceinline__ float exp2i(int s) { return __int_as_float((s + 127) << 23); }

// a, b -> f16 pairs hi = rn(a, b), lo = rn(a - hi, b - hi)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// One 64-element K-major row of an f16 operand tile pair (swizzled as described above).
__device__ __forceinline__ void store_row64(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                            const float (&v)[64]) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) split2(v[8 * p + 2 * q], v[8 * p + 2 * q + 1], h[q], l[q]);
    const uint32_t off = uint32_t(row) * 128u + ((uint32_t(p) ^ uint32_t(row & 7)) << 4);
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

__device__ __forceinline__ float block_max(float v, float* red, int slot) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[slot * 4 + (threadIdx.x >> 5)] = v;
  __syncthreads();
  const float m = fmaxf(fmaxf(red[slot * 4], red[slot * 4 + 1]),
                        fmaxf(red[slot * 4 + 2], red[slot * 4 + 3]));
  return m;
}

// u_{g,t} for t < 64 of the chunk starting at step k0 of a row (the reversed row when kRev);
// zero past the end of the row or for an unused column.
template <bool kRev>
__device__ __forceinline__ void load_chunk(const float* __restrict__ row, int L, int k0,
                                           bool valid, float (&v)[64]) {
  const int len = valid ? min(kT, L - k0) : 0;
  if (len == kT && (L & 3) == 0) {
    if (!kRev) {
      const float4* p = reinterpret_cast<const float4*>(row + k0);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 x = __ldg(p + q);
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(row + (L - k0 - kT));
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 x = __ldg(p + q);
        v[63 - 4 * q] = x.x; v[62 - 4 * q] = x.y; v[61 - 4 * q] = x.z; v[60 - 4 * q] = x.w;
      }
    }
  } else {
#pragma unroll
    for (int t = 0; t < kT; ++t)
      v[t] = (t < len) ? __ldg(row + (kRev ? (L - 1 - k0 - t) : (k0 + t))) : 0.f;
  }
}

// y at steps kb .. kb+31 of a row: stored (forward) or added at the mirrored steps (kRev).
template <bool kRev>
__device__ __forceinline__ void store_part(float* __restrict__ row, int L, int kb,
                                           const float (&o)[32]) {
  const int len = min(32, L - kb);
  if (len <= 0) return;
  if (len == 32 && (L & 3) == 0) {
    if (!kRev) {
      float4* p = reinterpret_cast<float4*>(row + kb);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        p[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    } else {
      float4* p = reinterpret_cast<float4*>(row + (L - kb - 32));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 c = p[q];
        c.x += o[31 - 4 * q]; c.y += o[30 - 4 * q]; c.z += o[29 - 4 * q]; c.w += o[28 - 4 * q];
        p[q] = c;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < len) {
        if (!kRev) row[kb + j] = o[j];
        else row[L - 1 - kb - j] += o[j];
      }
  }
}

// Per-channel tables: Q, the Toeplitz block of K_0..K_63, G (all as scaled f16 pairs), the
// chunk multiplier lambda^64 of this thread's state and the scales of K and G.
__device__ void build_tables(const TcScanArgs& a, int h, uint8_t* sm, float& mu_re,
                             float& mu_im_signed, float& dl_re, float& dl_im_signed,
                             float& sig_k, float& sig_g) {
  const int tid = threadIdx.x;
  float2* sPow = reinterpret_cast<float2*>(sm + kPow);
  float2* sPow8 = reinterpret_cast<float2*>(sm + kPow8);
  float2* sPow1 = reinterpret_cast<float2*>(sm + kPow1);
  lam_param* sPar = reinterpret_cast<lam_param*>(sm + kPar);
  float2* sW = reinterpret_cast<float2*>(sm + kWs);
  float* sK = reinterpret_cast<float*>(sm + kKtap);
  float* sRed = reinterpret_cast<float*>(sm + kRed);
  const int N = a.N;

  __syncthreads();  // the previous tile is done with every region reused below
  if (tid < kNMax) {
    const bool on = tid < N;
    sPar[tid] = on ? make_lam_param(a.log_re[(size_t)h * N + tid], a.log_im[(size_t)h * N + tid])
                   : lam_param{0.f, 0.f, 0.f};
    sW[tid] = on ? a.W[(size_t)h * N + tid] : make_float2(0.f, 0.f);
  }
  __syncthreads();
  // directly evaluated powers lambda^{8a} (a <= 8) and lambda^b (b < 8)
  for (int e = tid; e < kNMax * 17; e += kThreads) {
    const int n = e / 17, k = e % 17;
    const int j = (k < 9) ? 8 * k : (k - 9);
    cf v = {0.f, 0.f};
    if (n < N) v = lam_pow(sPar[n], j);
    if (k < 9) sPow8[n * 9 + k] = make_float2(v.re, v.im);
    else sPow1[n * 8 + (k - 9)] = make_float2(v.re, v.im);
  }
  __syncthreads();
  for (int e = tid; e < kNMax * kPw; e += kThreads) {
    const int n = e / kPw, j = e % kPw;
    const float2 p8 = sPow8[n * 9 + (j >> 3)], p1 = sPow1[n * 8 + (j & 7)];
    const cf v = cmul({p8.x, p8.y}, {p1.x, p1.y});
    sPow[e] = make_float2(v.re, v.im);
  }
  __syncthreads();
  // K_j = Re sum_n W_n lambda_n^j (threads 0..63) and the scales
  float kj = 0.f, wabs = 0.f;
  if (tid < kT) {
    for (int n = 0; n < N; ++n) {
      const float2 w = sW[n], p = sPow[n * kPw + tid];
      kj = fmaf(w.x, p.x, fmaf(-w.y, p.y, kj));
    }
    sK[tid] = kj;
    const float2 w = sW[tid];
    wabs = fmaxf(fabsf(w.x), fabsf(w.y));
  }
  const float kmax = block_max(fabsf(kj), sRed, 0);
  const float wmax = block_max(wabs, sRed, 1);
  const int ek = scale_exp(kmax), eg = scale_exp(wmax);
  sig_k = exp2i(ek);
  sig_g = exp2i(eg);
  float v[64];
  // Q row r = tid: Re|Im lambda_n^{63-t}, times 2^14
  {
    const int n = tid >> 1, c = tid & 1;
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      const float2 p = sPow[n * kPw + (kT - 1 - t)];
      v[t] = (c ? p.y : p.x) * 16384.f;
    }
    store_row64(sm + kQHi, sm + kQLo, tid, v);
  }
  // Toeplitz row t = tid (< 64): K_{t-s} for s <= t
  if (tid < kT) {
#pragma unroll
    for (int s = 0; s < kT; ++s) v[s] = (s <= tid) ? sK[tid - s] * sig_k : 0.f;
    store_row64(sm + kTkHi, sm + kTkLo, tid, v);
  }
  // G row t = tid >> 1, K-block tid & 1: Re(W_n lambda_n^{t+1}), -Im(...)
  {
    const int t = tid >> 1, kb = tid & 1;
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      const int r = kb * 64 + k, n = r >> 1;
      const float2 w = sW[n], p = sPow[n * kPw + t + 1];
      const cf g = cmul({w.x, w.y}, {p.x, p.y});
      v[k] = ((r & 1) ? -g.im : g.re) * sig_g;
    }
    store_row64(sm + kGHi + kb * 8192, sm + kGLo + kb * 8192, t, v);
  }
  // re-anchoring correction lambda^2048 - mu^32 (mu = the float lambda^64 the chain uses)
  float2* sDelta = reinterpret_cast<float2*>(sm + kDelta);
  if (tid < kNMax) {
    float2 d = make_float2(0.f, 0.f);
    if (tid < N) {
      const float2 m = sPow[tid * kPw + kT];
      cff p = {{m.x, 0.f}, {m.y, 0.f}};
#pragma unroll 1
      for (int i = 0; i < 5; ++i) p = cff_fma(p, p, cff{{0.f, 0.f}, {0.f, 0.f}});
      const cf a32 = lam_pow(sPar[tid], 32 * kT);
      const ff dr = ff_add(ff{a32.re, 0.f}, ff_neg(p.re));
      const ff di = ff_add(ff{a32.im, 0.f}, ff_neg(p.im));
      d = make_float2(dr.hi + dr.lo, di.hi + di.lo);
    }
    sDelta[tid] = d;
  }
  __syncthreads();
  {
    const int n = tid >> 1;
    const float2 m = sPow[n * kPw + kT];
    const float2 d = sDelta[n];
    mu_re = m.x;
    dl_re = d.x;
    // the state recurrence below keeps (own, other) components; the Im row runs it with the
    // sign of the imaginary parts flipped
    mu_im_signed = (tid & 1) ? -m.y : m.y;
    dl_im_signed = (tid & 1) ? -d.y : d.y;
  }
  __syncthreads();
}

template <bool kRev>
__global__ void __launch_bounds__(kThreads, 1) dlr_scan_tc_kernel(const TcScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sInvU = reinterpret_cast<float*>(sm + kInvU);
  float* sRowMax = reinterpret_cast<float*>(sm + kRowMax);
  float* sColSx = reinterpret_cast<float*>(sm + kColSx);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBar);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kSlot);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  const uint32_t tS = tmem + (uint32_t(warp * 32) << 16);  // this warp's lanes
  const uint32_t tY1 = tS + 128, tY2 = tS + 192;

  const int u0 = (int)((long long)blockIdx.x * a.units / gridDim.x);
  const int u1 = (int)((long long)(blockIdx.x + 1) * a.units / gridDim.x);
  const int segs = (a.R > 0) ? 1 : (a.C + kCols - 1) / kCols;
  const int reset_every = a.C;

  int cur_h = -1;
  float mu_re = 0.f, mu_im = 0.f, dl_re = 0.f, dl_im = 0.f, sig_k = 1.f, sig_g = 1.f;
  uint32_t parity = 0;
  bool ok = true;

  for (int unit = u0; unit < u1 && ok; ++unit) {
    int h, b0, nrows;
    if (a.R > 0) {
      h = unit / a.tiles_per_h;
      b0 = (unit - h * a.tiles_per_h) * a.R;
      nrows = min(a.R, a.B - b0);
    } else {
      h = unit / a.B;
      b0 = unit - h * a.B;
      nrows = 1;
    }
    if (h != cur_h) {
      build_tables(a, h, sm, mu_re, mu_im, dl_re, dl_im, sig_k, sig_g);
      cur_h = h;
    }
    // this thread's state and the last anchor, as (own component, other component)
    float xo = 0.f, xt = 0.f, ao = 0.f, at = 0.f;

    for (int seg = 0; seg < segs && ok; ++seg) {
      // ---- u chunks -> scaled f16 pairs (thread = chunk column) ----
      int rl, c;
      if (a.R > 0) {
        rl = tid / a.C;
        c = tid - rl * a.C;
      } else {
        rl = 0;
        c = seg * kCols + tid;
      }
      const bool valid = (a.R > 0) ? (rl < nrows) : (c < a.C);
      const size_t rowoff = ((size_t)(b0 + (valid ? rl : 0)) * a.H + h) * (size_t)a.L;
      const int k0 = c * kT;
      float inv_su;
      {
        float v[64];
        load_chunk<kRev>(a.u + rowoff, a.L, k0, valid, v);
        float m = 0.f;
#pragma unroll
        for (int t = 0; t < kT; ++t) m = fmaxf(m, fabsf(v[t]));
        const int es = scale_exp(m);
        const float su = exp2i(es);
#pragma unroll
        for (int t = 0; t < kT; ++t) v[t] *= su;
        store_row64(sm + kUHi, sm + kULo, tid, v);
        inv_su = exp2i(-es);
        sInvU[tid] = inv_su * (1.f / 16384.f);  // also undoes the 2^14 of Q
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t id1 = tc::idesc_f16_f32(128, 128);
        const uint64_t qh = tc::smem_desc_k_sw128(sm + kQHi), ql = tc::smem_desc_k_sw128(sm + kQLo);
        const uint64_t uh = tc::smem_desc_k_sw128(sm + kUHi), ul = tc::smem_desc_k_sw128(sm + kULo);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_kind_f16(tmem, qh + 2 * kk, uh + 2 * kk, id1, kk != 0);
          tc::mma_kind_f16(tmem, qh + 2 * kk, ul + 2 * kk, id1, 1);
          tc::mma_kind_f16(tmem, ql + 2 * kk, uh + 2 * kk, id1, 1);
        }
        tc::mma_commit(bar);
      }
      ok = __syncthreads_and(tc::mbar_wait(bar, parity));
      parity ^= 1;
      if (!ok) break;
      tc::fence_after_sync();

      // ---- carries along the chunks (thread = state row) ----
      // The largest |Xin| of each batch row in the tile goes to sRowMax[row][warp].
      float lmax = 0.f;
      int row_i = 0;
      {
        // row mode: a row starts every C columns and is anchored 32, 64, .. chunks into it;
        // one-row mode: anchors at every 32nd column (tiles hold 128 = 4 x 32 chunks)
        int next_reset = (a.R > 0) ? 0 : (1 << 30);
        int next_anchor = 0;
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          float s[32], o[32];
          tc::tmem_ld32(tS + blk * 32, s);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int g = blk * 32 + j;
            const float sother = __shfl_xor_sync(0xffffffffu, s[j], 1);
            const float iv = sInvU[g];
            if (g == next_anchor) {
              xo = fmaf(dl_re, ao, fmaf(-dl_im, at, xo));
              xt = fmaf(dl_re, at, fmaf(dl_im, ao, xt));
              ao = xo;
              at = xt;
              next_anchor += 32;
            }
            if (g == next_reset) {
              if (g > 0) {
                const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(lmax));
                if (lane == 0) sRowMax[row_i * 4 + warp] = __uint_as_float(m);
                ++row_i;
                lmax = 0.f;
              }
              xo = xt = ao = at = 0.f;
              next_reset += reset_every;
              next_anchor = g + 32;
            }
            o[j] = xo;
            lmax = fmaxf(lmax, fabsf(xo));
            const float no = fmaf(mu_re, xo, fmaf(-mu_im, xt, s[j] * iv));
            const float nt = fmaf(mu_re, xt, fmaf(mu_im, xo, sother * iv));
            xo = no;
            xt = nt;
          }
          tc::tmem_st32(tS + blk * 32, o);
        }
        tc::tmem_wait_st();
        const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(lmax));
        if (lane == 0) sRowMax[row_i * 4 + warp] = __uint_as_float(m);
      }
      __syncthreads();
      // Xin scale of this thread's chunk column (the scale of its batch row)
      float inv_sx;
      {
        const int row = (a.R > 0) ? tid / a.C : 0;
        const float xmax = fmaxf(fmaxf(sRowMax[row * 4], sRowMax[row * 4 + 1]),
                                 fmaxf(sRowMax[row * 4 + 2], sRowMax[row * 4 + 3]));
        const int ex = scale_exp(xmax);
        sColSx[tid] = exp2i(ex);
        inv_sx = exp2i(-ex);
      }
      __syncthreads();
      // ---- Xin -> scaled f16 pairs, A operand [chunk g][state row r] ----
      {
        const int r = tid;
        const uint32_t kbase = uint32_t(r >> 6) * 16384u + uint32_t(r & 7) * 2u;
        const uint32_t kc = uint32_t((r & 63) >> 3);
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          float v[32];
          tc::tmem_ld32(tS + blk * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int g = blk * 32 + j;
            const float x = v[j] * sColSx[g];
            const __half hh = __float2half_rn(x);
            const __half hl = __float2half_rn(x - __half2float(hh));
            const uint32_t off = kbase + uint32_t(g) * 128u + ((kc ^ uint32_t(g & 7)) << 4);
            *reinterpret_cast<__half*>(sm + kXHi + off) = hh;
            *reinterpret_cast<__half*>(sm + kXLo + off) = hl;
          }
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t id2 = tc::idesc_f16_f32(128, 64);
        const uint64_t uh = tc::smem_desc_k_sw128(sm + kUHi), ul = tc::smem_desc_k_sw128(sm + kULo);
        const uint64_t th = tc::smem_desc_k_sw128(sm + kTkHi), tl = tc::smem_desc_k_sw128(sm + kTkLo);
        const uint64_t xh = tc::smem_desc_k_sw128(sm + kXHi), xl = tc::smem_desc_k_sw128(sm + kXLo);
        const uint64_t gh = tc::smem_desc_k_sw128(sm + kGHi), gl = tc::smem_desc_k_sw128(sm + kGLo);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_kind_f16(tmem + 128, uh + 2 * kk, th + 2 * kk, id2, kk != 0);
          tc::mma_kind_f16(tmem + 128, uh + 2 * kk, tl + 2 * kk, id2, 1);
          tc::mma_kind_f16(tmem + 128, ul + 2 * kk, th + 2 * kk, id2, 1);
        }
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ao = kb * (16384 >> 4) + 2 * kk, bo = kb * (8192 >> 4) + 2 * kk;
            tc::mma_kind_f16(tmem + 192, xh + ao, gh + bo, id2, (kb | kk) != 0);
            tc::mma_kind_f16(tmem + 192, xh + ao, gl + bo, id2, 1);
            tc::mma_kind_f16(tmem + 192, xl + ao, gh + bo, id2, 1);
          }
        tc::mma_commit(bar);
      }
      ok = __syncthreads_and(tc::mbar_wait(bar, parity));
      parity ^= 1;
      if (!ok) break;
      tc::fence_after_sync();

      // ---- outputs (thread = chunk column) ----
      {
        const float ay = inv_su / sig_k;
        const float by = inv_sx / sig_g;
        float* yrow = a.y + rowoff;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float y1[32], y2[32];
          tc::tmem_ld32(tY1 + half * 32, y1);
          tc::tmem_ld32(tY2 + half * 32, y2);
#pragma unroll
          for (int j = 0; j < 32; ++j) y1[j] = fmaf(y1[j], ay, y2[j] * by);
          if (valid) store_part<kRev>(yrow, a.L, k0 + half * 32, y1);
        }
      }
      tc::fence_before_sync();
    }
  }
  if (!ok) report_status(a.status, DLR_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <bool kRev>
cudaError_t launch_one(const TcScanArgs& a, cudaStream_t s) {
  cudaError_t e = max_smem_once<dlr_scan_tc_kernel<kRev>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorUnknown;
  const int grid = std::min(a.units, sms);
  dlr_scan_tc_kernel<kRev><<<grid, kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

// N <= 64 complex states; u, y [B, H, L]; bidirectional adds the reversed pass.
cudaError_t launch_dlr_scan_tc(const float* u, const float* lr, const float* li, const float* W,
                               const float* lr2, const float* li2, const float* W2, bool bidir,
                               int B, int H, int N, int L, float* y, int* status,
                               cudaStream_t s) {
  TcScanArgs a{};
  a.u = u;
  a.y = y;
  a.B = B;
  a.H = H;
  a.N = N;
  a.L = L;
  a.C = (L + kT - 1) / kT;
  if (a.C <= kCols) {
    a.R = kCols / a.C;
    a.tiles_per_h = (B + a.R - 1) / a.R;
    a.units = H * a.tiles_per_h;
  } else {
    a.R = 0;
    a.tiles_per_h = 0;
    a.units = B * H;
  }
  a.status = status;
  a.log_re = lr;
  a.log_im = li;
  a.W = reinterpret_cast<const float2*>(W);
  cudaError_t e = launch_one<false>(a, s);
  if (e != cudaSuccess || !bidir) return e;
  a.log_re = lr2;
  a.log_im = li2;
  a.W = reinterpret_cast<const float2*>(W2);
  return launch_one<true>(a, s);
}

}  // namespace dlr
