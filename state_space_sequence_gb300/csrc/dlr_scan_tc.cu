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
// Two kernels. dlr_scan_tc_tables (one CTA per channel) evaluates the per-channel tables --
// Q, the Toeplitz block of K_0..K_63 and G as scaled f16 pairs in the exact byte layout the
// MMAs read, lambda^64, the re-anchoring correction and the two scales -- into a workspace
// blob per channel. dlr_scan_tc_kernel then runs one persistent CTA per SM with three warp
// roles joined by mbarriers and two tiles in flight:
//   warps 0-3  "scan":  thread r owns TMEM lane r = state row r; runs step 2 on S, writes Xin
//                       (scaled f16 pair, MN-major) to shared memory; loads Q into TMEM when
//                       the channel changes,
//   warps 4-7  "io":    thread g owns TMEM lane g = chunk g; loads u and writes its scaled f16
//                       pair (tile k+1), then reads Y1, Y2 and stores y (tile k),
//   warp 8, lane 0:     issues the MMAs, GEMM1 or GEMM2, whichever has its inputs first.
// Buffers: u operand x2, S accumulator x2 (TMEM), Xin x1, Y1/Y2 x1; Q lives in TMEM as the A
// operand of GEMM1, the Toeplitz block and G in shared memory (one bulk copy per channel).
// Units of work: a tile holds floor(128 / C) whole rows when a row has C <= 128 chunks
// (several batch rows of one channel), otherwise one row walks its tiles in order and carries
// its state from tile to tile. A CTA takes a contiguous range of units; at a change of channel
// the pipeline drains and the next channel's tables are copied in.
//
// Every wait is bounded (global timer, 1 s); a wait that runs out sets a CTA-wide abort flag,
// all roles leave their loops at the next wait or role barrier, and the kernel records
// DLR_ERR_TIMEOUT in the library's status word.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
namespace {

constexpr int kT = 64;        // steps per chunk
constexpr int kCols = 128;    // chunks per tile
constexpr int kNMax = 64;     // complex states (2N real rows of the state GEMM)
constexpr int kPw = kT + 1;   // powers lambda^0 .. lambda^64
constexpr int kThreads = 288; // warps 0-3 scan, 4-7 io, 8 mma
constexpr int kScanBar = 1, kIoBar = 2;  // named barriers of the scan and io warps

// TMEM columns (512 allocated): Q hi/lo (A operand of GEMM1, 2 f16 per column), S x2, Y1, Y2
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTQHi = 0, kTQLo = 32, kTS = 64, kTY1 = 320, kTY2 = 384;

// shared memory (bytes from a 1024-byte aligned base). K-major f16 tiles use the 128-byte
// swizzled layout: rows of 64 elements (128 bytes), 8-row atoms of 1024 bytes, 16-byte chunk
// index XOR (row & 7); K = 128 operands are two such tiles ("K-blocks") one after the other.
// Xin is MN-major: atoms of 8 K-rows (state rows) x 64 chunks (128 bytes per K-row, chunk
// index XOR (K-row & 7)); atom (K-group kg, M-half ma) at kg * 2048 + ma * 1024.
constexpr uint32_t kU = 0;              // u operand [128 chunks x 64], 2 buffers of hi + lo
constexpr uint32_t kUBuf = 32768, kULo = 16384;
constexpr uint32_t kXHi = 65536, kXLo = 98304;      // Xin [128 chunks x 128 rows], MN-major
constexpr uint32_t kTkHi = 131072, kTkLo = 139264;  // Toeplitz [64 t x 64 s], K-major
constexpr uint32_t kGHi = 147456, kGLo = 163840;    // G [64 t x 128 rows], K-major
constexpr uint32_t kInvU = 180224;   // float[2][128] 2^-14 / (u scale of chunk g), by parity
constexpr uint32_t kInvSu = kInvU + 1024;   // float[2][128] 1 / (u scale of chunk g)
constexpr uint32_t kColSx = kInvSu + 1024;  // float[2][128] Xin scale of chunk g
constexpr uint32_t kBy = kColSx + 1024;     // float[2][128] 1 / (Xin scale * G scale)
constexpr uint32_t kRowMax = kBy + 1024;    // float[128][4] per-row, per-warp max |Xin|
constexpr uint32_t kSig = kRowMax + 2048;   // float[4] K scale, G scale of the channel
constexpr uint32_t kBars = kSig + 16;       // mbarriers
// A waiter may trail the phase it waits for by at most one completed phase (the parity test
// cannot tell phase j from phase j + 2), so every wait below is on a barrier that cannot
// complete twice more before the waiter has passed: the u buffers get their own "free"
// barriers instead of sharing the GEMM2 one.
constexpr int kBarUFull = 0, kBarSFull = 2, kBarSFree = 4, kBarXFull = 6, kBarG2 = 7,
              kBarYFree = 8, kBarTab = 9, kBarScale = 10, kBarUFree = 12, kBarTabLoad = 14,
              kNumBars = 15;
constexpr uint32_t kSlot = kBars + 8 * kNumBars;  // TMEM base address
constexpr uint32_t kAbort = kSlot + 4;            // abort flag
constexpr uint32_t kEnd = kAbort + 4;
constexpr size_t kSmemBytes = kEnd + 1024;        // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Per-channel table blob in the workspace (bytes). Its first 48 KB are the shared-memory image
// of the Toeplitz and G operands (kTkHi .. kGLo + 16 KB), copied in one piece.
constexpr uint32_t kBlobSmem = kGLo + 16384 - kTkHi;  // 49152
constexpr uint32_t kBlobQ = kBlobSmem;       // uint32 [128 rows][64]: 32 hi then 32 lo words
constexpr uint32_t kBlobMu = kBlobQ + 32768;  // float4 [64]: lambda^64 (re, im), correction
constexpr uint32_t kBlobSig = kBlobMu + 1024; // float [4]: K scale, G scale
constexpr uint32_t kBlobBytes = kBlobSig + 1024;  // 83968, a multiple of 1024
static_assert(kBlobSmem == 49152 && kBlobBytes % 1024 == 0, "blob layout");

// Shared memory of the tables kernel.
constexpr uint32_t kTbKp = 0;                  // float [64 states][65] Re(W_n lambda_n^j)
constexpr uint32_t kTbK = kTbKp + 64 * 65 * 4; // float [64] K_0..K_63
constexpr uint32_t kTbRed = kTbK + 256;        // float [32]
constexpr uint32_t kTbBytes = kTbRed + 128;

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
  const uint8_t* tables;  // H table blobs of kBlobBytes
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

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier over `n` threads of named barrier `id` that also ANDs a predicate across them.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
  int r;
  asm volatile(
      "{\n"
      "  .reg .pred p, q;\n"
      "  setp.ne.s32 p, %1, 0;\n"
      "  bar.red.and.pred q, %2, %3, p;\n"
      "  selp.s32 %0, 1, 0, q;\n"
      "}\n"
      : "=r"(r)
      : "r"((int)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// Bounded wait on an mbarrier phase (one thread) that also gives up when another role has
// aborted. Each try may suspend the thread for a few microseconds.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_timer_ns();
  while (true) {
    if (tc::mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (tc::global_timer_ns() - t0 > tc::kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
}
// The same for a whole warp: lane 0 waits, the other lanes are held at the shuffle.
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity,
                                                volatile int* abort) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_phase(bar, parity, abort);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
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

// Where tile k of this CTA lies: channel, first batch row and row count, segment of the row.
struct TileInfo {
  int h, b0, nrows, seg;
};
__device__ __forceinline__ TileInfo tile_info(const TcScanArgs& a, int u0, int segs, int k) {
  const int unit = u0 + k / segs;
  TileInfo t;
  t.seg = k - (k / segs) * segs;
  if (a.R > 0) {
    t.h = unit / a.tiles_per_h;
    t.b0 = (unit - t.h * a.tiles_per_h) * a.R;
    t.nrows = min(a.R, a.B - t.b0);
  } else {
    t.h = unit / a.B;
    t.b0 = unit - t.h * a.B;
    t.nrows = 1;
  }
  return t;
}

// Column g of a tile: its batch row offset (elements) and first step, and whether it is used.
struct ColInfo {
  size_t rowoff;
  int k0;
  bool valid;
};
__device__ __forceinline__ ColInfo col_info(const TcScanArgs& a, const TileInfo& t, int g) {
  int rl, c;
  if (a.R > 0) {
    rl = g / a.C;
    c = g - rl * a.C;
  } else {
    rl = 0;
    c = t.seg * kCols + g;
  }
  ColInfo ci;
  ci.valid = (a.R > 0) ? (rl < t.nrows) : (c < a.C);
  ci.rowoff = ((size_t)(t.b0 + (ci.valid ? rl : 0)) * a.H + t.h) * (size_t)a.L;
  ci.k0 = c * kT;
  return ci;
}

// Max over the 256 threads of the tables kernel; `slot` picks 8 floats of `red`.
__device__ __forceinline__ float block_max256(float v, float* red, int slot) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[slot * 8 + (threadIdx.x >> 5)] = v;
  __syncthreads();
  float m = red[slot * 8];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[slot * 8 + i]);
  return m;
}

// Eight values of one K-major row of an f16 operand tile pair (16-byte chunk `chunk`), at a
// shared or global address.
__device__ __forceinline__ void store_chunk8(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                             int chunk, const float* v) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) split2(v[2 * q], v[2 * q + 1], h[q], l[q]);
  const uint32_t off = uint32_t(row) * 128u + ((uint32_t(chunk) ^ uint32_t(row & 7)) << 4);
  *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Per-channel tables (one CTA of 256 threads per channel h) into the channel's blob: the
// Toeplitz block of K_0..K_63 and G (scaled f16 pairs, swizzled exactly as in the main
// kernel's shared memory), Q (scaled f16 pairs as TMEM words), lambda^64 and the re-anchoring
// correction lambda^2048 - (lambda^64)^32 of every state, the scales of K and G.
// Thread (n, q) = (tid >> 2, tid & 3) owns state n and exponents j = 16q .. 16q + 16, held in
// registers: lambda^{16q + 4c} (c <= 4) and lambda^d (d < 4) evaluated directly, the others
// as one product of two of them.
__global__ void __launch_bounds__(256) dlr_scan_tc_tables(const TcScanArgs a, uint8_t* ws) {
  extern __shared__ __align__(16) uint8_t tsm[];
  const int tid = threadIdx.x;
  const int h = blockIdx.x;
  uint8_t* blob = ws + (size_t)h * kBlobBytes;
  float* sKp = reinterpret_cast<float*>(tsm + kTbKp);  // [64 states][65] Re(W_n lambda_n^j)
  float* sK = reinterpret_cast<float*>(tsm + kTbK);
  float* sRed = reinterpret_cast<float*>(tsm + kTbRed);
  const int N = a.N;
  const int n = tid >> 2, q = tid & 3;
  const bool on = n < N;
  const lam_param p = on ? make_lam_param(a.log_re[(size_t)h * N + n], a.log_im[(size_t)h * N + n])
                         : lam_param{0.f, 0.f, 0.f};
  const float2 w = on ? __ldg(&a.W[(size_t)h * N + n]) : make_float2(0.f, 0.f);
  const float sig_g = exp2i(scale_exp(block_max256(fmaxf(fabsf(w.x), fabsf(w.y)), sRed, 0)));

  // pw[i] = lambda^{16q + i}, i = 0..16
  cf pw[17];
  {
    cf base[5], small[4];
#pragma unroll
    for (int c = 0; c < 5; ++c) base[c] = on ? lam_pow(p, 16 * q + 4 * c) : cf{0.f, 0.f};
#pragma unroll
    for (int d = 0; d < 4; ++d) small[d] = on ? lam_pow(p, d) : cf{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 17; ++i) pw[i] = (i & 3) ? cmul(base[i >> 2], small[i & 3]) : base[i >> 2];
  }
  // Q rows 2n (Re) and 2n+1 (Im) at steps t = 63 - j, j in [16q, 16q + 16): TMEM words
  // (lower step in the low half) 24 - 8q .. 31 - 8q of each row
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const cf p0 = pw[15 - 2 * m], p1 = pw[14 - 2 * m];  // steps t0 = 48 - 16q + 2m, t0 + 1
      split2((c ? p0.im : p0.re) * 16384.f, (c ? p1.im : p1.re) * 16384.f, hi[m], lo[m]);
    }
    uint4* row = reinterpret_cast<uint4*>(blob + kBlobQ + (2 * n + c) * 256);
    row[6 - 2 * q] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    row[7 - 2 * q] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    row[14 - 2 * q] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    row[15 - 2 * q] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
  // G rows t = 16q .. 16q + 15, columns 2n, 2n+1: Re, -Im of W_n lambda_n^{t+1}; and the
  // products' real parts for the tap sums
  {
    const int kb = n >> 5;
    const uint32_t colb = uint32_t(((2 * n) & 7) * 2);  // byte offset of the pair in its chunk
    const uint32_t chunk = uint32_t((n & 31) >> 2);
    uint8_t* gh = blob + (kGHi - kTkHi) + kb * 8192;
    uint8_t* gl = blob + (kGLo - kTkHi) + kb * 8192;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = 16 * q + i;
      const cf g = cmul({w.x, w.y}, pw[i + 1]);
      uint32_t hb, lb;
      split2(g.re * sig_g, -g.im * sig_g, hb, lb);
      const uint32_t off = uint32_t(t) * 128u + ((chunk ^ uint32_t(t & 7)) << 4) + colb;
      *reinterpret_cast<uint32_t*>(gh + off) = hb;
      *reinterpret_cast<uint32_t*>(gl + off) = lb;
      sKp[n * 65 + 16 * q + i] = cmul({w.x, w.y}, pw[i]).re;  // Re(W lambda^j), j = 16q + i
    }
  }
  // lambda^64 and the re-anchoring correction (state n, thread q = 3 holds lambda^64)
  if (q == 3) {
    float2 d = make_float2(0.f, 0.f);
    const cf m = pw[16];
    if (on) {
      cff pp = {{m.re, 0.f}, {m.im, 0.f}};
#pragma unroll 1
      for (int i = 0; i < 5; ++i) pp = cff_fma(pp, pp, cff{{0.f, 0.f}, {0.f, 0.f}});
      const cf a32 = lam_pow(p, 32 * kT);
      const ff dr = ff_add(ff{a32.re, 0.f}, ff_neg(pp.re));
      const ff di = ff_add(ff{a32.im, 0.f}, ff_neg(pp.im));
      d = make_float2(dr.hi + dr.lo, di.hi + di.lo);
    }
    reinterpret_cast<float4*>(blob + kBlobMu)[n] = make_float4(m.re, m.im, d.x, d.y);
  }
  __syncthreads();
  // K_j = sum_n Re(W_n lambda_n^j): thread (j, part) = (tid >> 2, tid & 3) sums 16 states
  const int j = tid >> 2, part = tid & 3;
  float ks = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ks += sKp[(16 * part + i) * 65 + j];
  ks += __shfl_xor_sync(0xffffffffu, ks, 1);
  ks += __shfl_xor_sync(0xffffffffu, ks, 2);
  if (part == 0) sK[j] = ks;
  const float sig_k = exp2i(scale_exp(block_max256(part == 0 ? fabsf(ks) : 0.f, sRed, 1)));
  if (tid == 0) {
    reinterpret_cast<float*>(blob + kBlobSig)[0] = sig_k;
    reinterpret_cast<float*>(blob + kBlobSig)[1] = sig_g;
  }
  // Toeplitz row t = j, s in [16 part, 16 part + 16): K_{t-s} for s <= t (sK complete after the
  // barrier inside block_max256)
  float tv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int ss = 16 * part + i;
    tv[i] = (ss <= j) ? sK[j - ss] * sig_k : 0.f;
  }
  store_chunk8(blob, blob + (kTkLo - kTkHi), j, 2 * part, tv);
  store_chunk8(blob, blob + (kTkLo - kTkHi), j, 2 * part + 1, tv + 8);
}

// Scan warps at the start of a channel: Q from the blob into TMEM (thread r = lane r), this
// thread's lambda^64 and correction, the scales; thread 0 starts the bulk copy of the
// Toeplitz and G operands into shared memory (completing on kBarTabLoad).
__device__ __forceinline__ void load_tables(const uint8_t* blob, uint8_t* sm, uint32_t tmem,
                                            float& mu_re, float& mu_im_signed, float& dl_re,
                                            float& dl_im_signed, float& sig_g) {
  const int tid = threadIdx.x, warp = tid >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&bars[kBarTabLoad], kBlobSmem);
    tc::bulk_load(sm + kTkHi, blob, kBlobSmem, &bars[kBarTabLoad]);
  }
  const uint4* q = reinterpret_cast<const uint4*>(blob + kBlobQ + tid * 256);
  float hi[32], lo[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 a = __ldg(q + i), b = __ldg(q + 8 + i);
    hi[4 * i] = __uint_as_float(a.x); hi[4 * i + 1] = __uint_as_float(a.y);
    hi[4 * i + 2] = __uint_as_float(a.z); hi[4 * i + 3] = __uint_as_float(a.w);
    lo[4 * i] = __uint_as_float(b.x); lo[4 * i + 1] = __uint_as_float(b.y);
    lo[4 * i + 2] = __uint_as_float(b.z); lo[4 * i + 3] = __uint_as_float(b.w);
  }
  const uint32_t tl = tmem + (uint32_t(warp * 32) << 16);
  tc::tmem_st32(tl + kTQHi, hi);
  tc::tmem_st32(tl + kTQLo, lo);
  const float4 m = __ldg(reinterpret_cast<const float4*>(blob + kBlobMu) + (tid >> 1));
  mu_re = m.x;
  dl_re = m.z;
  // the state recurrence keeps (own, other) components; the Im row runs it with the sign of
  // the imaginary parts flipped
  mu_im_signed = (tid & 1) ? -m.y : m.y;
  dl_im_signed = (tid & 1) ? -m.w : m.w;
  const float sk = __ldg(reinterpret_cast<const float*>(blob + kBlobSig));
  sig_g = __ldg(reinterpret_cast<const float*>(blob + kBlobSig) + 1);
  if (tid == 0) reinterpret_cast<float*>(sm + kSig)[0] = sk;
  tc::tmem_wait_st();
  tc::fence_before_sync();
}

// ---- the three roles ------------------------------------------------------------------

// Scan warps, one tile: carries along the chunks, then Xin as a scaled f16 pair.
__device__ __forceinline__ bool scan_tile(const TcScanArgs& a, uint8_t* sm, uint32_t tmem,
                                          int k, bool new_row, float mu_re, float mu_im,
                                          float dl_re, float dl_im, float sig_g, float& xo,
                                          float& xt, float& ao, float& at,
                                          volatile int* abort) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int par = k & 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const float* sInvU = reinterpret_cast<const float*>(sm + kInvU) + par * 128;
  float* sColSx = reinterpret_cast<float*>(sm + kColSx) + par * 128;
  float* sBy = reinterpret_cast<float*>(sm + kBy) + par * 128;
  float* sRowMax = reinterpret_cast<float*>(sm + kRowMax);
  const uint32_t tS = tmem + (uint32_t(warp * 32) << 16) + kTS + uint32_t(par) * 128;

  // S of this tile, and (for the per-chunk u scales) the io threads' release of tile k
  bool ok = warp_wait_phase(&bars[kBarSFull + par], (k >> 1) & 1, abort) &&
            warp_wait_phase(&bars[kBarUFull + par], (k >> 1) & 1, abort);
  if (!named_bar_and(kScanBar, 128, ok)) return false;
  tc::fence_after_sync();

  if (new_row) xo = xt = ao = at = 0.f;
  const int C = a.C;
  if (a.R > 0 && (C == 32 || C == 64)) {
    // two independent chains: columns [0, 64) and [64, 128) (whole rows of 32 or 64 chunks);
    // row starts and anchors fall on 32-column block starts
    float xoB = 0.f, xtB = 0.f, aoB = 0.f, atB = 0.f, lA = 0.f, lB = 0.f;
#pragma unroll 1
    for (int bb = 0; bb < 2; ++bb) {
      const int cA = bb * 32, cB = 64 + bb * 32;
      if (cA % C == 0) {
        xo = xt = ao = at = 0.f;
        xoB = xtB = aoB = atB = 0.f;
      } else {
        xo = fmaf(dl_re, ao, fmaf(-dl_im, at, xo));
        xt = fmaf(dl_re, at, fmaf(dl_im, ao, xt));
        ao = xo;
        at = xt;
        xoB = fmaf(dl_re, aoB, fmaf(-dl_im, atB, xoB));
        xtB = fmaf(dl_re, atB, fmaf(dl_im, aoB, xtB));
        aoB = xoB;
        atB = xtB;
      }
      float sA[32], sB[32];
      tc::tmem_ld32(tS + cA, sA);
      tc::tmem_ld32(tS + cB, sB);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float ivA = sInvU[cA + j], ivB = sInvU[cB + j];
        const float pA = __shfl_xor_sync(0xffffffffu, sA[j], 1);
        const float pB = __shfl_xor_sync(0xffffffffu, sB[j], 1);
        const float oA = xo, oB = xoB;
        lA = fmaxf(lA, fabsf(oA));
        lB = fmaxf(lB, fabsf(oB));
        const float noA = fmaf(mu_re, xo, fmaf(-mu_im, xt, sA[j] * ivA));
        const float ntA = fmaf(mu_re, xt, fmaf(mu_im, xo, pA * ivA));
        const float noB = fmaf(mu_re, xoB, fmaf(-mu_im, xtB, sB[j] * ivB));
        const float ntB = fmaf(mu_re, xtB, fmaf(mu_im, xoB, pB * ivB));
        sA[j] = oA;
        sB[j] = oB;
        xo = noA;
        xt = ntA;
        xoB = noB;
        xtB = ntB;
      }
      tc::tmem_st32(tS + cA, sA);
      tc::tmem_st32(tS + cB, sB);
      if ((cA + 32) % C == 0) {  // rows end with this block
        const unsigned mA = __reduce_max_sync(0xffffffffu, __float_as_uint(lA));
        const unsigned mB = __reduce_max_sync(0xffffffffu, __float_as_uint(lB));
        if (lane == 0) {
          sRowMax[(cA / C) * 4 + warp] = __uint_as_float(mA);
          sRowMax[(cB / C) * 4 + warp] = __uint_as_float(mB);
        }
        lA = lB = 0.f;
      }
    }
    tc::tmem_wait_st();
  } else if (a.R == 0 || C % 32 == 0) {
    // one chain (one row per tile): a row start at column 0 when new_row, anchors at every
    // other 32-column block start
    float l = 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      const int c0 = blk * 32;
      if (a.R > 0 && c0 % C == 0) {
        xo = xt = ao = at = 0.f;
      } else {
        xo = fmaf(dl_re, ao, fmaf(-dl_im, at, xo));
        xt = fmaf(dl_re, at, fmaf(dl_im, ao, xt));
        ao = xo;
        at = xt;
      }
      float sv[32];
      tc::tmem_ld32(tS + c0, sv);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float iv = sInvU[c0 + j];
        const float p = __shfl_xor_sync(0xffffffffu, sv[j], 1);
        const float o = xo;
        l = fmaxf(l, fabsf(o));
        const float no = fmaf(mu_re, xo, fmaf(-mu_im, xt, sv[j] * iv));
        const float nt = fmaf(mu_re, xt, fmaf(mu_im, xo, p * iv));
        sv[j] = o;
        xo = no;
        xt = nt;
      }
      tc::tmem_st32(tS + c0, sv);
    }
    tc::tmem_wait_st();
    const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(l));
    if (lane == 0) sRowMax[warp] = __uint_as_float(m);
  } else {
    // any other row length: row starts and anchors checked column by column
    int next_reset = 0;
    int next_anchor = 0;
    float lmax = 0.f;
    int row_i = 0;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      float sv[32], o[32];
      tc::tmem_ld32(tS + blk * 32, sv);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int g = blk * 32 + j;
        const float iv = sInvU[g];
        const float sother = __shfl_xor_sync(0xffffffffu, sv[j], 1);
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
          next_reset += C;
          next_anchor = g + 32;
        }
        o[j] = xo;
        lmax = fmaxf(lmax, fabsf(xo));
        const float no = fmaf(mu_re, xo, fmaf(-mu_im, xt, sv[j] * iv));
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
  named_bar(kScanBar, 128);
  // Xin scale of chunk column tid (the scale of its batch row)
  {
    const int row = (a.R > 0) ? tid / a.C : 0;
    const float xmax = fmaxf(fmaxf(sRowMax[row * 4], sRowMax[row * 4 + 1]),
                             fmaxf(sRowMax[row * 4 + 2], sRowMax[row * 4 + 3]));
    const int ex = scale_exp(xmax);
    sColSx[tid] = exp2i(ex);
    sBy[tid] = exp2i(-ex) / sig_g;
  }
  mbar_arrive(&bars[kBarScale + par]);  // releases sBy (and the channel scales) to the io warps
  // the Xin buffer is free once GEMM2 of the previous tile has completed
  ok = (k == 0) || warp_wait_phase(&bars[kBarG2], (k - 1) & 1, abort);
  if (!named_bar_and(kScanBar, 128, ok)) return false;
  // Xin -> scaled f16 pair, MN-major: this thread writes state row r = tid, 8 chunks per
  // 16-byte store
  {
    const int r = tid;
    const uint32_t kbase = uint32_t(r >> 3) * 2048u + uint32_t(r & 7) * 128u;
    const uint32_t kr = uint32_t(r & 7);
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      float v[32];
      tc::tmem_ld32(tS + blk * 32, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int g0 = blk * 32 + q * 8;
        const float4 c0 = *reinterpret_cast<const float4*>(sColSx + g0);
        const float4 c1 = *reinterpret_cast<const float4*>(sColSx + g0 + 4);
        const float sc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          split2(v[q * 8 + 2 * p] * sc[2 * p], v[q * 8 + 2 * p + 1] * sc[2 * p + 1], h[p], l[p]);
        const uint32_t cg = uint32_t(g0 >> 3);  // 16-byte chunk index along the chunks
        const uint32_t off = kbase + (cg >> 3) * 1024u + (((cg & 7u) ^ kr) << 4);
        *reinterpret_cast<uint4*>(sm + kXHi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(sm + kXLo + off) = make_uint4(l[0], l[1], l[2], l[3]);
      }
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  mbar_arrive(&bars[kBarXFull]);
  mbar_arrive(&bars[kBarSFree + par]);
  return true;
}

// IO warps: u chunks of tile k -> scaled f16 pair (thread = chunk column g).
template <bool kRev>
__device__ __forceinline__ bool load_tile(const TcScanArgs& a, uint8_t* sm, int u0, int segs,
                                          int k, volatile int* abort) {
  const int g = threadIdx.x - 128;
  const int par = k & 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  // the u buffer is free once GEMM2 of tile k-2 has completed
  const bool ok =
      (k < 2) || warp_wait_phase(&bars[kBarUFree + par], ((k - 2) >> 1) & 1, abort);
  if (!named_bar_and(kIoBar, 128, ok)) return false;
  const TileInfo ti = tile_info(a, u0, segs, k);
  const ColInfo ci = col_info(a, ti, g);
  float v[64];
  load_chunk<kRev>(a.u + ci.rowoff, a.L, ci.k0, ci.valid, v);
  float m = 0.f;
#pragma unroll
  for (int t = 0; t < kT; ++t) m = fmaxf(m, fabsf(v[t]));
  const int es = scale_exp(m);
  const float su = exp2i(es);
#pragma unroll
  for (int t = 0; t < kT; ++t) v[t] *= su;
  uint8_t* ubuf = sm + kU + par * kUBuf;
  store_row64(ubuf, ubuf + kULo, g, v);
  const float inv_su = exp2i(-es);
  reinterpret_cast<float*>(sm + kInvU)[par * 128 + g] = inv_su * (1.f / 16384.f);
  reinterpret_cast<float*>(sm + kInvSu)[par * 128 + g] = inv_su;
  tc::fence_proxy_async_smem();
  mbar_arrive(&bars[kBarUFull + par]);
  return true;
}

// IO warps: outputs of tile k (thread = chunk column g = TMEM lane).
template <bool kRev>
__device__ __forceinline__ bool store_tile(const TcScanArgs& a, uint8_t* sm, uint32_t tmem,
                                           int u0, int segs, int k, volatile int* abort) {
  const int g = threadIdx.x - 128, warp = threadIdx.x >> 5;
  const int par = k & 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const bool ok = warp_wait_phase(&bars[kBarG2], k & 1, abort) &&
                  warp_wait_phase(&bars[kBarScale + par], (k >> 1) & 1, abort);
  if (!named_bar_and(kIoBar, 128, ok)) return false;
  tc::fence_after_sync();
  const float sig_k = reinterpret_cast<const float*>(sm + kSig)[0];
  const float ay = reinterpret_cast<const float*>(sm + kInvSu)[par * 128 + g] / sig_k;
  const float by = reinterpret_cast<const float*>(sm + kBy)[par * 128 + g];
  const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
  float y[64];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float y1[32], y2[32];
    tc::tmem_ld32(lane_base + kTY1 + half * 32, y1);
    tc::tmem_ld32(lane_base + kTY2 + half * 32, y2);
#pragma unroll
    for (int j = 0; j < 32; ++j) y[half * 32 + j] = fmaf(y1[j], ay, y2[j] * by);
  }
  tc::fence_before_sync();
  mbar_arrive(&bars[kBarYFree]);
  const TileInfo ti = tile_info(a, u0, segs, k);
  const ColInfo ci = col_info(a, ti, g);
  if (ci.valid) {
    float* yrow = a.y + ci.rowoff;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float o[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = y[half * 32 + j];
      store_part<kRev>(yrow, a.L, ci.k0 + half * 32, o);
    }
  }
  return true;
}

// MMA thread: are the inputs of GEMM1 of tile k in place? (u operand written, S buffer k & 1
// released by the scan of tile k-2, the channel's tables loaded for the first tile of a channel)
__device__ __forceinline__ bool gemm1_ready(uint64_t* bars, int k, bool first_of_group,
                                            uint32_t group) {
  const int par = k & 1;
  if (first_of_group && !(tc::mbar_try_wait(&bars[kBarTab], group & 1) &&
                          tc::mbar_try_wait(&bars[kBarTabLoad], group & 1)))
    return false;
  if (!tc::mbar_try_wait(&bars[kBarUFull + par], (k >> 1) & 1)) return false;
  return k < 2 || tc::mbar_try_wait(&bars[kBarSFree + par], ((k - 2) >> 1) & 1);
}

// GEMM1 of tile k: S = Q u^T into S buffer k & 1 (A = Q from TMEM, B = u operand).
__device__ __forceinline__ void gemm1(uint8_t* sm, uint32_t tmem, int k) {
  const int par = k & 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  tc::fence_after_sync();
  constexpr uint32_t id1 = tc::idesc_f16_f32(128, 128);
  const uint8_t* ubuf = sm + kU + par * kUBuf;
  const uint64_t uh = tc::smem_desc_k_sw128(ubuf), ul = tc::smem_desc_k_sw128(ubuf + kULo);
  const uint32_t dS = tmem + kTS + uint32_t(par) * 128;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t qh = tmem + kTQHi + kk * 8, ql = tmem + kTQLo + kk * 8;
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  setp.ne.b32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %3, 1;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %2, %3, 1;\n"
        "}\n" ::"r"(dS),
        "r"(qh), "l"(uh + 2 * kk), "r"(id1), "r"(kk), "l"(ul + 2 * kk), "r"(ql)
        : "memory");
  }
  tc::mma_commit(&bars[kBarSFull + par]);
}

// MMA thread: are the inputs of GEMM2 of tile k in place? (Xin written, Y read out for k-1)
__device__ __forceinline__ bool gemm2_ready(uint64_t* bars, int k) {
  if (!tc::mbar_try_wait(&bars[kBarXFull], k & 1)) return false;
  return k < 1 || tc::mbar_try_wait(&bars[kBarYFree], (k - 1) & 1);
}

// GEMM2 of tile k: Y1 = u Tk^T, Y2 = Xin G^T; its completion also frees u buffer k & 1.
__device__ __forceinline__ void gemm2(uint8_t* sm, uint32_t tmem, int k) {
  const int par = k & 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  tc::fence_after_sync();
  constexpr uint32_t idk = tc::idesc_f16_f32(128, 64);
  constexpr uint32_t idm = idk | (1u << 15);  // A (Xin) MN-major
  const uint8_t* ubuf = sm + kU + par * kUBuf;
  const uint64_t uh = tc::smem_desc_k_sw128(ubuf), ul = tc::smem_desc_k_sw128(ubuf + kULo);
  const uint64_t th = tc::smem_desc_k_sw128(sm + kTkHi), tl = tc::smem_desc_k_sw128(sm + kTkLo);
  const uint64_t gh = tc::smem_desc_k_sw128(sm + kGHi), gl = tc::smem_desc_k_sw128(sm + kGLo);
  const uint64_t xh = tc::smem_desc_mn_sw128(sm + kXHi, 1024, 2048);
  const uint64_t xl = tc::smem_desc_mn_sw128(sm + kXLo, 1024, 2048);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    tc::mma_kind_f16(tmem + kTY1, uh + 2 * kk, th + 2 * kk, idk, kk != 0);
    tc::mma_kind_f16(tmem + kTY1, uh + 2 * kk, tl + 2 * kk, idk, 1);
    tc::mma_kind_f16(tmem + kTY1, ul + 2 * kk, th + 2 * kk, idk, 1);
  }
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint64_t ao = uint64_t(s) * (4096 >> 4);                     // 16 rows = 2 K-groups
    const uint64_t bo = uint64_t(s >> 2) * (8192 >> 4) + 2 * (s & 3);  // K-block, 32 bytes
    tc::mma_kind_f16(tmem + kTY2, xh + ao, gh + bo, idm, s != 0);
    tc::mma_kind_f16(tmem + kTY2, xh + ao, gl + bo, idm, 1);
    tc::mma_kind_f16(tmem + kTY2, xl + ao, gh + bo, idm, 1);
  }
  tc::mma_commit(&bars[kBarG2]);
  tc::mma_commit(&bars[kBarUFree + par]);
}

// MMA thread, tiles [k0, k1) of one channel: issues GEMM2 of the oldest tile whose Xin is
// ready, else GEMM1 of the next tile whose u is ready. Gives up (abort flag) after the wait
// limit without progress.
__device__ __forceinline__ void mma_role(uint8_t* sm, uint32_t tmem, int k0, int k1,
                                         uint32_t group, volatile int* abort) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  int n1 = k0, n2 = k0;
  uint64_t t_last = tc::global_timer_ns();
  while (n2 < k1) {
    bool did = false;
    if (n2 < n1 && gemm2_ready(bars, n2)) {
      gemm2(sm, tmem, n2++);
      did = true;
    } else if (n1 < k1 && gemm1_ready(bars, n1, n1 == k0, group)) {
      gemm1(sm, tmem, n1++);
      did = true;
    }
    if (did) {
      t_last = tc::global_timer_ns();
    } else {
      if (*abort) return;
      if (tc::global_timer_ns() - t_last > tc::kWaitLimitNs) {
        *abort = 1;
        return;
      }
      __nanosleep(32);
    }
  }
}

template <bool kRev>
__global__ void __launch_bounds__(kThreads, 1) dlr_scan_tc_kernel(const TcScanArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kAbort);

  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    tc::mbar_init(&bars[kBarUFull], 128);
    tc::mbar_init(&bars[kBarUFull + 1], 128);
    tc::mbar_init(&bars[kBarSFull], 1);
    tc::mbar_init(&bars[kBarSFull + 1], 1);
    tc::mbar_init(&bars[kBarSFree], 128);
    tc::mbar_init(&bars[kBarSFree + 1], 128);
    tc::mbar_init(&bars[kBarXFull], 128);
    tc::mbar_init(&bars[kBarG2], 1);
    tc::mbar_init(&bars[kBarYFree], 128);
    tc::mbar_init(&bars[kBarTab], 128);
    tc::mbar_init(&bars[kBarScale], 128);
    tc::mbar_init(&bars[kBarScale + 1], 128);
    tc::mbar_init(&bars[kBarUFree], 1);
    tc::mbar_init(&bars[kBarUFree + 1], 1);
    tc::mbar_init(&bars[kBarTabLoad], 1);
    *abort = 0;
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

  const int u0 = (int)((long long)blockIdx.x * a.units / gridDim.x);
  const int u1 = (int)((long long)(blockIdx.x + 1) * a.units / gridDim.x);
  const int segs = (a.R > 0) ? 1 : (a.C + kCols - 1) / kCols;
  const int ntiles = (u1 - u0) * segs;

  // scan-thread state
  float mu_re = 0.f, mu_im = 0.f, dl_re = 0.f, dl_im = 0.f, sig_g = 1.f;
  float xo = 0.f, xt = 0.f, ao = 0.f, at = 0.f;
  uint32_t group = 0;

  for (int k0 = 0; k0 < ntiles; ++group) {
    // the tiles [k0, k1) share one channel
    const int h = tile_info(a, u0, segs, k0).h;
    const int u_end = min(u1, (a.R > 0) ? (h + 1) * a.tiles_per_h : (h + 1) * a.B);
    const int k1 = (u_end - u0) * segs;

    if (warp < 4) {
      load_tables(a.tables + (size_t)h * kBlobBytes, sm, tmem, mu_re, mu_im, dl_re, dl_im,
                  sig_g);
      mbar_arrive(&bars[kBarTab]);
      for (int k = k0; k < k1; ++k) {
        const TileInfo ti = tile_info(a, u0, segs, k);
        if (!scan_tile(a, sm, tmem, k, ti.seg == 0, mu_re, mu_im, dl_re, dl_im, sig_g, xo, xt,
                       ao, at, abort))
          break;
      }
    } else if (warp < 8) {
      bool ok = true;
      for (int k = k0; k < k1 && ok; ++k) {
        ok = load_tile<kRev>(a, sm, u0, segs, k, abort);
        if (ok && k > k0) ok = store_tile<kRev>(a, sm, tmem, u0, segs, k - 1, abort);
      }
      if (ok) store_tile<kRev>(a, sm, tmem, u0, segs, k1 - 1, abort);
    } else if ((tid & 31) == 0) {
      mma_role(sm, tmem, k0, k1, group, abort);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (*abort) break;
    k0 = k1;
  }
  if (*abort) report_status(a.status, DLR_ERR_TIMEOUT);
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
cudaError_t launch_one(const TcScanArgs& a, uint8_t* ws, cudaStream_t s) {
  cudaError_t e = max_smem_once<dlr_scan_tc_kernel<kRev>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorUnknown;
  dlr_scan_tc_tables<<<a.H, 256, kTbBytes, s>>>(a, ws);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = std::min(a.units, sms);
  dlr_scan_tc_kernel<kRev><<<grid, kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t scan_tc_workspace_bytes(int64_t H) { return (size_t)H * kBlobBytes; }

// N <= 64 complex states; u, y [B, H, L]; bidirectional adds the reversed pass (run after the
// forward one, reusing the workspace for its tables).
cudaError_t launch_dlr_scan_tc(const float* u, const float* lr, const float* li, const float* W,
                               const float* lr2, const float* li2, const float* W2, bool bidir,
                               int B, int H, int N, int L, float* y, void* ws, int* status,
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
  a.tables = static_cast<const uint8_t*>(ws);
  a.log_re = lr;
  a.log_im = li;
  a.W = reinterpret_cast<const float2*>(W);
  cudaError_t e = launch_one<false>(a, static_cast<uint8_t*>(ws), s);
  if (e != cudaSuccess || !bidir) return e;
  a.log_re = lr2;
  a.log_im = li2;
  a.W = reinterpret_cast<const float2*>(W2);
  return launch_one<true>(a, static_cast<uint8_t*>(ws), s);
}

}  // namespace dlr
