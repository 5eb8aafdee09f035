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
// split every operand is scaled by a power of two: u per batch row and tile so that its
// largest |u| lies in [2^13, 2^14) (one row's scale never depends on another row's
// magnitude), K and G per channel the same way, Q by 2^14 (|Q| <= 1), and Xin by the fixed
// 2^-27 of its tile's S units (raised for a state carried in from the previous tile; see
// kXinShift). The scalings are exact and undone in fp32 when y is written (the carries run on
// S in its scaled units; a row continued into the next tile is rescaled to that tile's units).
// Powers lambda^j are evaluated from an exactly reduced phase (lam_pow) for j = 8q + 4c and
// j < 4 and combined by one complex product, so no power carries a long multiplication chain.
//
// Two kernels. dlr_scan_tc_tables (one CTA per channel) evaluates the per-channel tables --
// Q, the Toeplitz block of K_0..K_63 and G as scaled f16 pairs in the exact byte layout the
// MMAs read, lambda^64, the re-anchoring correction and the two scales -- into a workspace
// blob per channel. dlr_scan_tc_kernel then runs one persistent CTA per SM with three roles
// joined by mbarriers, two tiles in flight:
//   warps 0-7 "main" (two warps per TMEM lane quarter, half h = warp >> 2). Iteration k:
//     - the u operand of tile k+1: thread = chunk g, steps 32h .. 32h + 31; the float32 tile
//       the producer landed in the tile's operand buffer is converted in place into its
//       scaled f16 pair (K-major), or loaded directly when the rows are not whole chunks; Q
//       into TMEM for a new channel;
//     - the outputs of tile k-1: thread = chunk g = TMEM lane, steps 32h .. 32h + 31: Y1, Y2
//       scaled, written through a per-warp staging image and a TMA store (plain stores when
//       the rows are not whole chunks);
//     - step 2 of tile k: thread r = TMEM lane r = state row r; the carries along the chunks
//       of S written straight into the Xin operand (MN-major f16 pair), half h writing the
//       columns 64h .. 64h + 63;
//   warp 8, lane 0: issues the MMAs: GEMM1 (with the Toeplitz part) of tile k+1, then GEMM2
//     of tile k,
//   warp 9, lane 0: the producer: every bulk copy (u tiles, the Toeplitz and G operands of a
//     new channel), in the order the MMA groups complete.
// One role for the per-element work keeps the instruction stream small and lets the stages
// of one tile follow each other without hand-offs between warps.
// Buffers: u operand x2, Xin x1, Toeplitz and G x1, y staging (shared memory); Q, S x2,
// Y1 x2, Y2 (TMEM).
// Units of work: a tile holds floor(128 / C) whole rows when a row has C <= 128 chunks
// (several batch rows of one channel), otherwise one row walks its tiles in order and carries
// its state from tile to tile. A CTA takes a contiguous range of units.
//
// Every wait is bounded (global timer, 1 s); a wait that runs out sets a CTA-wide abort flag,
// all roles leave their loops at the next wait or role barrier, and the kernel records
// DLR_ERR_TIMEOUT in the library's status word.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 10;

// Timeline hooks of profiling builds (compiled with DLR_SCAN_TRACE: CTA 0 records the global
// timer at fixed points into a device buffer the caller provides); no code otherwise.
#ifdef DLR_SCAN_TRACE
__device__ long long* g_scan_trace;
#define SCAN_TRACE(slot)                                                        \
  do {                                                                          \
    if (blockIdx.x == 0 && (slot) >= 0 && (slot) < 4096) {                      \
      unsigned long long t_;                                                    \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                    \
      g_scan_trace[(slot)] = (long long)t_;                                     \
    }                                                                           \
  } while (0)
// every CTA (its start and end times)
#define SCAN_TRACE_ALL(slot)                                                    \
  do {                                                                          \
    unsigned long long t_;                                                      \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                      \
    g_scan_trace[(slot)] = (long long)t_;                                       \
  } while (0)
#else
#define SCAN_TRACE(slot) \
  do {                   \
  } while (0)
#define SCAN_TRACE_ALL(slot) \
  do {                       \
  } while (0)
#endif

namespace {

constexpr int kT = 64;          // steps per chunk
constexpr int kCols = 128;      // chunks per tile
constexpr int kThreads = 320;   // warps 0-7 main, 8 mma, 9 producer
constexpr int kMainBar = 1;     // named barrier of the 256 main threads

// TMEM columns (512 allocated): Q (hi 32 + lo 32 columns: A operand of GEMM1, two f16 per
// column), S x2, Y1 x2, Y2
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTQ = 0, kTS = 64, kTY1 = 320, kTY2 = 448;

// Shared memory (bytes from a 1024-byte aligned base). f16 operand tiles use 128-byte
// swizzling. K-major (Toeplitz, G): rows of 64 elements (128 bytes), 8-row atoms of 1024
// bytes, 16-byte chunk index XOR (row & 7); K = 128 operands are two such tiles one after the
// other. MN-major (u operand, Xin): atoms of 8 K-rows x 64 MN-elements (128 bytes per K-row,
// chunk index XOR (K-row & 7)); atom (K-group kg, MN-half ma) at kg * 2048 + ma * 1024.
constexpr uint32_t kU = 0;                          // u operand [128 chunks x 64], x2 (hi, lo)
constexpr uint32_t kUBuf = 32768, kULo = 16384;
constexpr uint32_t kXHi = 65536, kXLo = 98304;      // Xin [128 chunks x 128 rows]
constexpr uint32_t kTkHi = 131072, kTkLo = 139264;  // Toeplitz [64 t x 64 s], K-major
constexpr uint32_t kGHi = 147456, kGLo = 163840;    // G [64 t x 128 rows], K-major
constexpr uint32_t kYStage = 180224;  // y staging, one 4 KB image per main warp:
                                      // [32 lines][32 floats], swizzled
constexpr uint32_t kRowEs = kYStage + 32768;  // int[4][128] u scale exponent of each row
constexpr uint32_t kRowMaxU = kRowEs + 2048;  // uint[128] max |u| of each row (scratch)
constexpr uint32_t kAy = kRowMaxU + 512;      // float[4][128] 1 / (u scale * K scale)
constexpr uint32_t kBy = kAy + 2048;          // float[4][128] 1 / (Xin scale * G scale)
constexpr uint32_t kScanRed = kBy + 2048;     // uint[4] per-warp max |carried state|
constexpr uint32_t kBars = kScanRed + 16;     // mbarriers
// A waiter may trail the phase it waits for by at most one completed phase (the parity test
// cannot tell phase j from phase j + 2): every wait below is on a barrier that cannot
// complete twice more before the waiter has passed it.
constexpr int kBarStage = 0,   // [2] u tile (float32) landed in its operand buffer (TMA bytes)
    kBarUFull = 2,             // [2] u operand and its scales written (main, 256)
    kBarG1 = 4,                // [2] GEMM1 + Toeplitz done: S, Y1 ready, u buffer free (commit)
    kBarXFull = 6,             // Xin operand written, S read (main, 256)
    kBarG2 = 7,                // GEMM2 (state part) done: Y2 ready, Xin buffer free (commit)
    kBarY1Free = 8,            // [2] Y1 read out of TMEM (main, 256)
    kBarY2Free = 10,           // Y2 read out of TMEM (main, 256)
    kBarTabTk = 11,            // Toeplitz operand copied (bytes)
    kBarTabG = 12,             // G operand copied (bytes)
    kNumBars = 13;
constexpr uint32_t kSlot = kBars + 8 * kNumBars;  // TMEM base address
constexpr uint32_t kAbort = kSlot + 4;            // abort flag
constexpr uint32_t kEnd = kAbort + 4;
constexpr size_t kSmemBytes = kEnd + 1024;        // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// Per-channel table blob in the workspace (bytes). Its first 48 KB are the shared-memory image
// of the Toeplitz and G operands (kTkHi .. kGLo + 16 KB), copied in one piece.
constexpr uint32_t kBlobSmem = kGLo + 16384 - kTkHi;  // 49152
constexpr uint32_t kBlobQ = kBlobSmem;        // uint32 [128 rows][64]: 32 hi then 32 lo words
constexpr uint32_t kBlobMu = kBlobQ + 32768;  // float4 [64]: lambda^64 (re, im), correction
constexpr uint32_t kBlobSig = kBlobMu + 1024; // float [4]: K scale, G scale
constexpr uint32_t kBlobBytes = kBlobSig + 1024;  // 83968, a multiple of 1024
static_assert(kBlobSmem == 49152 && kBlobBytes % 1024 == 0, "blob layout");

// Shared memory of the tables kernel: the blob image, then scratch.
constexpr uint32_t kTbKp = kBlobBytes;         // float [64 states][65] Re(W_n lambda_n^j)
constexpr uint32_t kTbK = kTbKp + 64 * 65 * 4; // float [64] K_0..K_63
constexpr uint32_t kTbRed = kTbK + 256;        // float [2][16]
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
  int tma;          // u tiles by TMA (L % 64 == 0 and C in {32, 64, 128} or C > 128, C % 64 == 0)
  int bc;           // chunks per TMA box (32 or 64)
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

// a, b -> f16 pairs: hi = a and b rounded to 11 significant bits (to nearest, ties away from
// zero, by an integer add at the 13th mantissa bit and a mask: exact in f16 for |a| >= 2^-14),
// lo = the f16 rounding of the remainder (|lo| <= 2^-11 |a|). The pair carries a to 2^-22 of
// |a| (and to 2^-24 absolute below the f16 normal range); every operand is scaled so that its
// largest magnitude lies near 2^14, which keeps the absolute floor far below what the products
// need. No conversion result feeds another conversion.
__device__ __forceinline__ float round11(float a) {
  return __uint_as_float((__float_as_uint(a) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const float ah = round11(a), bh = round11(b);
  const __half2 h = __floats2half2_rn(ah, bh);
  const __half2 l = __floats2half2_rn(a - ah, b - bh);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// The same for a * s and b * s, the scaling and the remainders in two-wide float instructions
// (each lane of a pair rounds as the scalar operation would: the results are identical).
__device__ __forceinline__ void split2s(float a, float b, float s, uint32_t& hi, uint32_t& lo) {
  const float2 v = __fmul2_rn(make_float2(a, b), make_float2(s, s));
  const float ah = round11(v.x), bh = round11(v.y);
  const float2 r = __ffma2_rn(make_float2(ah, bh), make_float2(-1.f, -1.f), v);  // v - (ah, bh)
  const __half2 h = __floats2half2_rn(ah, bh);
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Programmatic dependent launch: the table kernel lets the scan kernel launch early; the scan
// kernel waits for the table kernel's completion (and memory) before it reads the tables. Both
// are no-ops when the launch is not programmatic.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_wait_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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
// The main warps' wait for a phase: every lane waits (and so acquires what the phase
// published). A wait that gives up leaves the abort flag set and returns; the warp then carries
// on through its schedule (every later wait returns at once), so all main warps still reach
// every named barrier and the kernel ends; the caller reports DLR_ERR_TIMEOUT.
__device__ __forceinline__ bool lanes_wait_phase(uint64_t* bar, uint32_t parity,
                                                 volatile int* abort) {
  return wait_phase(bar, parity, abort);
}

constexpr int kTbThreads = 512;  // threads of the tables kernel

// Max over the kTbThreads threads of the tables kernel; `slot` picks 16 floats of `red`.
__device__ __forceinline__ float block_max_tb(float v, float* red, int slot) {
  constexpr int kWarps = kTbThreads / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[slot * kWarps + (threadIdx.x >> 5)] = v;
  __syncthreads();
  float m = red[slot * kWarps];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) m = fmaxf(m, red[slot * kWarps + i]);
  return m;
}

// Eight values of one K-major row of an f16 operand tile pair (16-byte chunk `chunk`), at a
// shared or global address.
__device__ __forceinline__ void store_chunk8(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                             int chunk, const float* v, int rows) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) split2(v[2 * q], v[2 * q + 1], h[q], l[q]);
  const uint32_t off = uint32_t(row) * 128u + ((uint32_t(chunk) ^ uint32_t(row & 7)) << 4);
  if (DLR_IN(row, rows) && DLR_IN(chunk, 8)) {
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// store_chunk8 of v * s (the scaling in two-wide float instructions).
__device__ __forceinline__ void store_chunk8s(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                              int chunk, const float* v, float s, int rows) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) split2s(v[2 * q], v[2 * q + 1], s, h[q], l[q]);
  const uint32_t off = uint32_t(row) * 128u + ((uint32_t(chunk) ^ uint32_t(row & 7)) << 4);
  if (DLR_IN(row, rows) && DLR_IN(chunk, 8)) {
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
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

// The tiles of a CTA in order, without a division after the first: the channel, the group of
// batch rows (row mode) or batch row (long rows) within it, and the segment of the row.
struct TileIter {
  TileInfo t;
  int bt;  // group of rows (row mode) or batch row (long rows) within the channel
};
__device__ __forceinline__ TileIter tile_iter_begin(const TcScanArgs& a, int u0) {
  TileIter it;
  it.t.seg = 0;
  if (a.R > 0) {
    it.t.h = u0 / a.tiles_per_h;
    it.bt = u0 - it.t.h * a.tiles_per_h;
    it.t.b0 = it.bt * a.R;
    it.t.nrows = min(a.R, a.B - it.t.b0);
  } else {
    it.t.h = u0 / a.B;
    it.bt = u0 - it.t.h * a.B;
    it.t.b0 = it.bt;
    it.t.nrows = 1;
  }
  return it;
}
__device__ __forceinline__ void tile_iter_next(const TcScanArgs& a, int segs, TileIter& it) {
  if (++it.t.seg < segs) return;
  it.t.seg = 0;
  if (++it.bt == ((a.R > 0) ? a.tiles_per_h : a.B)) {
    it.bt = 0;
    ++it.t.h;
  }
  if (a.R > 0) {
    it.t.b0 = it.bt * a.R;
    it.t.nrows = min(a.R, a.B - it.t.b0);
  } else {
    it.t.b0 = it.bt;
  }
}

// Column g of a tile: its row within the tile, chunk index within its row, batch row offset
// (elements) and first step, and whether it is used. In row mode the row and chunk of a column
// are the same in every tile (`rc` = (g / C, g % C), computed once).
struct ColInfo {
  size_t rowoff;
  int rl, c, k0;
  bool valid;
};
__device__ __forceinline__ int2 col_rows(const TcScanArgs& a, int g) {
  if (a.R > 0) {
    const int rl = g / a.C;
    return make_int2(rl, g - rl * a.C);
  }
  return make_int2(0, g);
}
__device__ __forceinline__ ColInfo col_info(const TcScanArgs& a, const TileInfo& t, int2 rc) {
  ColInfo ci;
  ci.rl = rc.x;
  ci.c = (a.R > 0) ? rc.y : t.seg * kCols + rc.y;
  ci.valid = (a.R > 0) ? (ci.rl < t.nrows) : (ci.c < a.C);
  ci.rowoff = ((size_t)(t.b0 + (ci.valid ? ci.rl : 0)) * a.H + t.h) * (size_t)a.L;
  ci.k0 = ci.c * kT;
  return ci;
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

// Per-channel tables (one CTA of 512 threads per channel h) into the channel's blob: the
// Toeplitz block of K_0..K_63 and G (scaled f16 pairs, swizzled exactly as in the main
// kernel's shared memory), Q (scaled f16 pairs as TMEM words), lambda^64 and the re-anchoring
// correction lambda^2048 - (lambda^64)^32 of every state, the scales of K and G. The blob is
// assembled in shared memory and leaves in bulk copies.
// Thread (n, q) = (tid & 63, tid >> 6) owns state n and exponents j = 8q .. 8q + 8, held in
// registers (lambda and lambda^{8q} evaluated directly, the rest by short products); warps 14
// and 15 (q = 7) also form the re-anchoring correction.
__global__ void __launch_bounds__(kTbThreads, 2)
    dlr_scan_tc_tables(const TcScanArgs a, uint8_t* ws) {
  extern __shared__ __align__(1024) uint8_t tsm[];
  const int tid = threadIdx.x;
  const int h = blockIdx.x;
  uint8_t* img = tsm;  // the blob image
  float* sKp = reinterpret_cast<float*>(tsm + kTbKp);  // [64 states][65] Re(W_n lambda_n^j)
  float* sK = reinterpret_cast<float*>(tsm + kTbK);
  float* sRed = reinterpret_cast<float*>(tsm + kTbRed);
  const int N = a.N;
  const int n = tid & 63, q = tid >> 6;
  const bool on = n < N;
  grid_launch_dependents();
  if (tid == 0) SCAN_TRACE(3900);
  const lam_param p = on ? make_lam_param(a.log_re[(size_t)h * N + n], a.log_im[(size_t)h * N + n])
                         : lam_param{0.f, 0.f, 0.f};
  const float2 w = on ? __ldg(&a.W[(size_t)h * N + n]) : make_float2(0.f, 0.f);
  const float sig_g = exp2i(scale_exp(block_max_tb(fmaxf(fabsf(w.x), fabsf(w.y)), sRed, 0)));
  if (tid == 0) SCAN_TRACE(3901);

  // pw[i] = lambda^{8q + i}, i = 0..8: lambda and lambda^{8q} evaluated directly, lambda^i
  // (i <= 8) by products of depth at most three, then one product with lambda^{8q}; each power
  // carries at most a few roundings, never a chain that grows with the exponent. The table
  // entries enter y once each, so a few roundings stay far below the tolerance.
  cf pw[9];
  {
    cf sm_[9];
    sm_[0] = cf{1.f, 0.f};
    sm_[1] = on ? lam_pow(p, 1) : cf{0.f, 0.f};
    sm_[2] = cmul(sm_[1], sm_[1]);
    sm_[3] = cmul(sm_[2], sm_[1]);
    sm_[4] = cmul(sm_[2], sm_[2]);
    sm_[5] = cmul(sm_[4], sm_[1]);
    sm_[6] = cmul(sm_[4], sm_[2]);
    sm_[7] = cmul(sm_[4], sm_[3]);
    sm_[8] = cmul(sm_[4], sm_[4]);
    const cf base = on ? lam_pow(p, 8 * q) : cf{0.f, 0.f};
    pw[0] = base;
#pragma unroll
    for (int i = 1; i < 9; ++i) pw[i] = (q == 0) ? sm_[i] : cmul(base, sm_[i]);
    // lambda^64 = mu, whose rounding the chunk recurrence compounds between re-anchors:
    // evaluated directly
    if (q == 7 && on) pw[8] = lam_pow(p, 64);
  }
  // Q rows 2n (Re) and 2n+1 (Im) at steps t = 63 - j, j in [8q, 8q + 8): TMEM words (lower step
  // in the low half) 28 - 4q .. 31 - 4q of each row
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const cf p0 = pw[7 - 2 * m], p1 = pw[6 - 2 * m];  // steps t0 = 56 - 8q + 2m, t0 + 1
      split2((c ? p0.im : p0.re) * 16384.f, (c ? p1.im : p1.re) * 16384.f, hi[m], lo[m]);
    }
    uint4* row = reinterpret_cast<uint4*>(img + kBlobQ + (2 * n + c) * 256);
    if (DLR_IN(2 * n + c, 128) && DLR_IN(15 - q, 16) && DLR_IN(7 - q, 8)) {
      row[7 - q] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      row[15 - q] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  // G rows t = 8q .. 8q + 7, columns 2n, 2n+1: Re, -Im of W_n lambda_n^{t+1}; and the products'
  // real parts for the tap sums
  {
    const int kb = n >> 5;
    const uint32_t colb = uint32_t(((2 * n) & 7) * 2);  // byte offset of the pair in its chunk
    const uint32_t chunk = uint32_t((n & 31) >> 2);
    uint8_t* gh = img + (kGHi - kTkHi) + kb * 8192;
    uint8_t* gl = img + (kGLo - kTkHi) + kb * 8192;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = 8 * q + i;
      const cf g = cmul({w.x, w.y}, pw[i + 1]);
      uint32_t hb, lb;
      split2(g.re * sig_g, -g.im * sig_g, hb, lb);
      const uint32_t off = uint32_t(t) * 128u + ((chunk ^ uint32_t(t & 7)) << 4) + colb;
      if (DLR_IN(kb * 8192 + off + 3, 16384)) {
        *reinterpret_cast<uint32_t*>(gh + off) = hb;
        *reinterpret_cast<uint32_t*>(gl + off) = lb;
      }
      if (DLR_IN(n * 65 + 8 * q + i, 64 * 65))
        sKp[n * 65 + 8 * q + i] = cmul({w.x, w.y}, pw[i]).re;  // Re(W lambda^j), j = 8q + i
    }
  }
  // lambda^64 and the re-anchoring correction (warps 14 and 15: q = 7 holds lambda^64)
  if (q == 7) {
    float2 d = make_float2(0.f, 0.f);
    const cf m = pw[8];
    if (on) {
      cff pp = {{m.re, 0.f}, {m.im, 0.f}};
#pragma unroll 1
      for (int i = 0; i < 5; ++i) pp = cff_fma(pp, pp, cff{{0.f, 0.f}, {0.f, 0.f}});
      const cf a32 = lam_pow(p, 32 * kT);
      const ff dr = ff_add(ff{a32.re, 0.f}, ff_neg(pp.re));
      const ff di = ff_add(ff{a32.im, 0.f}, ff_neg(pp.im));
      d = make_float2(dr.hi + dr.lo, di.hi + di.lo);
    }
    if (DLR_IN(n, 64))
      reinterpret_cast<float4*>(img + kBlobMu)[n] = make_float4(m.re, m.im, d.x, d.y);
  }
  if (tid == 0) SCAN_TRACE(3902);
  __syncthreads();
  if (tid == 0) SCAN_TRACE(3903);
  // K_j = sum_n Re(W_n lambda_n^j): thread (j, part) = (tid >> 3, tid & 7) sums 8 states
  const int j = tid >> 3, part = tid & 7;
  float ks = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (DLR_IN((8 * part + i) * 65 + j, 64 * 65)) ks += sKp[(8 * part + i) * 65 + j];
  ks += __shfl_xor_sync(0xffffffffu, ks, 1);
  ks += __shfl_xor_sync(0xffffffffu, ks, 2);
  ks += __shfl_xor_sync(0xffffffffu, ks, 4);
  if (part == 0 && DLR_IN(j, 64)) sK[j] = ks;
  const float sig_k = exp2i(scale_exp(block_max_tb(part == 0 ? fabsf(ks) : 0.f, sRed, 1)));
  if (tid == 0) {
    reinterpret_cast<float*>(img + kBlobSig)[0] = sig_k;
    reinterpret_cast<float*>(img + kBlobSig)[1] = sig_g;
  }
  // Toeplitz row t = j, s in [8 part, 8 part + 8): K_{t-s} for s <= t (sK complete after the
  // barrier inside block_max_tb)
  float tv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ss = 8 * part + i;
    tv[i] = (ss <= j && DLR_IN(j - ss, 64)) ? sK[j - ss] * sig_k : 0.f;
  }
  store_chunk8(img, img + (kTkLo - kTkHi), j, part, tv, 64);
  // the image to the channel's blob
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) SCAN_TRACE(3904);
  if (tid == 0) {
    uint8_t* blob = ws + (size_t)h * kBlobBytes;
    constexpr uint32_t kPart = kBlobBytes / 4;  // 20992, a multiple of 16
#pragma unroll
    for (int i = 0; i < 4; ++i) tc::bulk_store(blob + i * kPart, img + i * kPart, kPart);
    tc::bulk_commit_group();
    tc::bulk_wait_group0();
    SCAN_TRACE(3905);
  }
}

// ---- the roles ----------------------------------------------------------------------------

// producer thread: the TMA tiles of u for tile k, as float32, into the tile's operand buffer
// (k & 1) -- forward chunk order, one 128-byte line per chunk and half, 128-byte swizzle --
// completing on kBarStage + (k & 1). The main warps convert them in place. Row mode: boxes of
// bc chunks of each valid row; one-row mode: two boxes of 64 chunks. Chunks past the row (or
// before it, reversed) read as zero.
template <bool kRev>
__device__ __forceinline__ void issue_u_tma(const TcScanArgs& a, const CUtensorMap* map,
                                            uint8_t* sm, int u0, int segs, int k) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const TileInfo ti = tile_info(a, u0, segs, k);
  const int bc = a.bc;
  const int nrows = (a.R > 0) ? ti.nrows : 1;
  const int nblk = (a.R > 0) ? a.C / bc : kCols / bc;
  uint64_t* bar = &bars[kBarStage + (k & 1)];
  uint8_t* buf = sm + kU + (k & 1) * kUBuf;
  tc::mbar_arrive_expect_tx(bar, uint32_t(nrows * nblk * 2 * bc * 128));
  for (int rl = 0; rl < nrows; ++rl)
    for (int cb = 0; cb < nblk; ++cb) {
      const int line0 = ((a.R > 0) ? rl * a.C : 0) + cb * bc;
      const int c0 = ((a.R > 0) ? 0 : ti.seg * kCols) + cb * bc;  // first (reversed) chunk
      const int y = kRev ? (a.C - c0 - bc) : c0;
      const int z = (ti.b0 + rl) * a.H + ti.h;
#pragma unroll
      for (int half = 0; half < 2; ++half)
        tc::tma_load_3d(buf + half * 16384 + line0 * 128, map, half * 32, y, z, bar);
    }
}

// Staging line holding column g's chunk when the staging is in forward chunk order and the
// columns count reversed chunks (TMA path, reversed pass).
__device__ __forceinline__ int mirrored_line(const TcScanArgs& a, int g) {
  const int bc = a.bc;
  const int base = (a.R > 0) ? (g / a.C) * a.C : 0;
  const int c = g - base, cb = c / bc, j = c - cb * bc;
  return base + cb * bc + (bc - 1 - j);
}

// u at steps kb .. kb + 31 of the chunk that starts at step k0 of a row (the reversed row when
// kRev); zero past the end of the row or for an unused column.
template <bool kRev>
__device__ __forceinline__ void load_part32(const float* __restrict__ row, int L, int kb,
                                            bool valid, float (&v)[32]) {
  const int len = valid ? min(32, L - kb) : 0;
  if (len == 32 && (L & 3) == 0) {
    if (!kRev) {
      const float4* p = reinterpret_cast<const float4*>(row + kb);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = __ldg(p + q);
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(row + (L - kb - 32));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = __ldg(p + q);
        v[31 - 4 * q] = x.x; v[30 - 4 * q] = x.y; v[29 - 4 * q] = x.z; v[28 - 4 * q] = x.w;
      }
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      v[t] = (t < len) ? __ldg(row + (kRev ? (L - 1 - kb - t) : (kb + t))) : 0.f;
  }
}

// main warps, at the first tile of a channel: half h of Q of the channel (the hi words for
// h = 0, the lo words for h = 1) from its blob into TMEM (thread = lane r of its quarter).
__device__ __forceinline__ void load_q_half(const uint8_t* blob, uint32_t tmem, int r, int h) {
  const uint4* q = reinterpret_cast<const uint4*>(blob + kBlobQ + (DLR_IN(r, 128) ? r : 0) * 256) + 8 * h;
  const uint32_t tl = tmem + (uint32_t(r & ~31) << 16) + kTQ + 32 * h;
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = __ldg(q + 4 * part + i);
      w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
    }
    tc::tmem_st16(tl + 16 * part, w);
  }
}

// main warps, tile j: u -> the scaled f16 pair operand (K-major). Thread = chunk column g (lane
// of its quarter), half h = steps 32h .. 32h + 31 of the chunk; the float32 tile the TMA wrote
// into the same buffer is read by every thread before the barrier inside and overwritten only
// after it. Also the row scales of the tile (ring slot j & 3) and, at a new channel, Q.
template <bool kRev>
__device__ __forceinline__ bool conv_tile(const TcScanArgs& a, uint8_t* sm, uint32_t tmem,
                                          const TileInfo& ti, int2 rc, int j, int& cur_h,
                                          float& sig_k, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = warp >> 2, g = (warp & 3) * 32 + lane;
  const int par = j & 1, slot = j & 3;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const bool new_channel = ti.h != cur_h;
  // the u buffer released by GEMM1 of tile j-2; at a new channel also GEMM1 of tile j-1 done
  // (Q is reloaded); the u tile landed
  bool ok = true;
  if (j >= 2) ok = lanes_wait_phase(&bars[kBarG1 + par], ((j - 2) >> 1) & 1, abort);
  if (new_channel && j >= 1)
    ok &= lanes_wait_phase(&bars[kBarG1 + (par ^ 1)], ((j - 1) >> 1) & 1, abort);
  if (a.tma) ok &= lanes_wait_phase(&bars[kBarStage + par], (j >> 1) & 1, abort);
  if (threadIdx.x == 0) SCAN_TRACE(1000 + j * 8 + 1);
  const uint8_t* blob = a.tables + (size_t)ti.h * kBlobBytes;
  const ColInfo ci = col_info(a, ti, rc);
  uint8_t* ubuf = sm + kU + par * kUBuf;
  float v[32];
  if (a.tma) {
    const int line = kRev ? mirrored_line(a, g) : g;
    const uint32_t sw = uint32_t(line & 7);
    const uint8_t* src = ubuf + (kRev ? 1 - h : h) * 16384 + line * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 x = DLR_IN(line, 128)
                           ? *reinterpret_cast<const float4*>(src + ((uint32_t(q) ^ sw) << 4))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      if (!kRev) {
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
      } else {
        v[31 - 4 * q] = x.x; v[30 - 4 * q] = x.y; v[29 - 4 * q] = x.z; v[28 - 4 * q] = x.w;
      }
    }
    if (!ci.valid) {
#pragma unroll
      for (int t = 0; t < 32; ++t) v[t] = 0.f;
    }
  } else {
    load_part32<kRev>(a.u + ci.rowoff, a.L, ci.k0 + 32 * h, ci.valid, v);
  }
  // the row's largest |u| in this tile: a warp reduction when the warp's 32 chunks share a
  // row, else one shared-memory atomic per thread (non-negative floats order as their bits)
  float m = 0.f;
#pragma unroll
  for (int t = 0; t < 32; ++t) m = fmaxf(m, fabsf(v[t]));
  unsigned* rmax = reinterpret_cast<unsigned*>(sm + kRowMaxU);
  const int rl = ci.rl;
  const bool warp_row = __shfl_sync(0xffffffffu, rl, 0) == __shfl_sync(0xffffffffu, rl, 31);
  if (warp_row) {
    const unsigned mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
    if (lane == 0 && DLR_IN(rl, 128)) atomicMax(&rmax[rl], mw);
  } else {
    if (DLR_IN(rl, 128)) atomicMax(&rmax[rl], __float_as_uint(m));
  }
  named_bar(kMainBar, 256);
  const int es = scale_exp(__uint_as_float(DLR_IN(rl, 128) ? rmax[rl] : 0u));
  const float su = exp2i(es);
#pragma unroll
  for (int p = 0; p < 4; ++p) store_chunk8s(ubuf, ubuf + kULo, g, 4 * h + p, v + 8 * p, su, 128);
  if (new_channel) {
    // the first read of the tables: at the CTA's first tile, wait here for the table kernel
    // (programmatic dependent launch), so the conversion above overlaps its end
    if (cur_h < 0) grid_wait_prerequisites();
    cur_h = ti.h;
    sig_k = __ldg(reinterpret_cast<const float*>(blob + kBlobSig));
  }
  if (h == 0) {
    if ((ci.c == 0 || g == 0) && DLR_IN(slot * 128 + rl, 512))
      reinterpret_cast<int*>(sm + kRowEs)[slot * 128 + rl] = es;
    if (DLR_IN(slot * 128 + g, 512))
      reinterpret_cast<float*>(sm + kAy)[slot * 128 + g] = exp2i(-es) / sig_k;
  }
  tc::fence_proxy_async_smem();
  if (new_channel) {
    load_q_half(blob, tmem, g, h);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  if (threadIdx.x == 0) SCAN_TRACE(1000 + j * 8 + 2);
  tc::mbar_arrive(&bars[kBarUFull + par]);
  named_bar(kMainBar, 256);  // every thread has read the row maxima of this tile
  if (h == 0) rmax[g] = 0u;
  return true;
}

// producer (warp 9, lane 0): every bulk copy into shared memory, taken in the order the MMA
// groups complete (GEMM1 of tile 0, then GEMM1 of tile k+1 and GEMM2 of tile k for k = 0, 1,
// ...): u of tile k into operand buffer k & 1 once GEMM1 of tile k-2 has read that buffer;
// the Toeplitz operand of a new channel once GEMM1 of the previous tile is done, its G operand
// once GEMM2 of the previous tile is done. A thread blocked while the TMA unit takes a copy's
// requests holds up nobody else.
template <bool kRev>
__device__ __forceinline__ void producer_role(const TcScanArgs& a, const CUtensorMap* map,
                                              uint8_t* sm, int u0, int segs, int ntiles,
                                              volatile int* abort) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  if (ntiles == 0) return;
  auto channel = [&](int k) { return tile_info(a, u0, segs, k).h; };
  auto copy_tk = [&](int h) {
    tc::mbar_arrive_expect_tx(&bars[kBarTabTk], kGHi - kTkHi);
    tc::bulk_load(sm + kTkHi, a.tables + (size_t)h * kBlobBytes, kGHi - kTkHi, &bars[kBarTabTk]);
  };
  auto copy_g = [&](int h) {
    tc::mbar_arrive_expect_tx(&bars[kBarTabG], kGLo + 16384 - kGHi);
    tc::bulk_load(sm + kGHi, a.tables + (size_t)h * kBlobBytes + (kGHi - kTkHi),
                  kGLo + 16384 - kGHi, &bars[kBarTabG]);
  };
  if (a.tma) {
    SCAN_TRACE(1100);
    issue_u_tma<kRev>(a, map, sm, u0, segs, 0);
    SCAN_TRACE(1101);
    if (ntiles > 1) issue_u_tma<kRev>(a, map, sm, u0, segs, 1);
    SCAN_TRACE(1102);
  }
  grid_wait_prerequisites();  // the tables are written
  int h = channel(0);
  copy_tk(h);
  copy_g(h);
  for (int k = -1; k < ntiles; ++k) {
    // GEMM1 of tile j = k + 1 done: u of tile j + 2; the Toeplitz operand of tile j + 1
    const int j = k + 1;
    if (j < ntiles) {
      const bool u_next = a.tma && j + 2 < ntiles;
      const bool tk_next = j + 1 < ntiles && channel(j + 1) != channel(j);
      if (u_next || tk_next) {
        if (!wait_phase(&bars[kBarG1 + (j & 1)], (j >> 1) & 1, abort)) return;
        SCAN_TRACE(1000 + (j + 2) * 8 + 5);
        if (u_next) issue_u_tma<kRev>(a, map, sm, u0, segs, j + 2);
        if (tk_next) copy_tk(channel(j + 1));
      }
    }
    // GEMM2 of tile k done: the G operand of tile k + 1 at a new channel. G2 is one barrier
    // whose parity test cannot tell phase k from phase k +- 2, so every completion is waited
    // for in order (free: GEMM2 of tile k completes before GEMM1 of tile k + 2, the next
    // completion this thread waits for). This thread is then never a phase ahead of G2, and
    // the skipped GEMM1 waits above stay exact. It can fall a phase behind only where GEMM2
    // does not depend on it; such a wait just returns at a later completion (everything the
    // later GEMM2s need from this thread -- u copies -- was issued before it), and at a channel
    // change it is exact again: GEMM2 of the new channel's first tile needs the copy below.
    if (k >= 0 && k + 1 < ntiles) {
      if (!wait_phase(&bars[kBarG2], k & 1, abort)) return;
      if (channel(k + 1) != channel(k)) copy_g(channel(k + 1));
    }
  }
}

// main warps: y of tile j once GEMM2 of the tile is done (thread = chunk column g = TMEM lane
// of its quarter, half h = steps 32h .. 32h + 31): y = Y1 / (u scale * K scale) + Y2 / (Xin
// scale * G scale). With whole-chunk rows (the TMA shapes) each warp writes its 32 chunks x 32
// steps into its staging image and one lane stores them as one TMA tile (added, at the
// mirrored chunks and steps, when kRev); otherwise each thread stores its 32 steps itself.
template <bool kRev>
__device__ __forceinline__ bool epi_tile(const TcScanArgs& a, const CUtensorMap* ymap,
                                         uint8_t* sm, uint32_t tmem, const TileInfo& ti,
                                         int2 rc, int j, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = warp >> 2, quarter = warp & 3, g = quarter * 32 + lane;
  const int par = j & 1, slot = j & 3;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const bool ok = lanes_wait_phase(&bars[kBarG2], j & 1, abort);
  if (threadIdx.x == 0) SCAN_TRACE(2000 + j * 8 + 1);
  tc::fence_after_sync();
  const uint32_t lane_base = tmem + (uint32_t(quarter * 32) << 16);
  float y1[32], y2[32];
  // (the TMEM column ranges are uniform over the warp: a failed check skips the warp's loads)
  if (DLR_IN(kTY1 + par * 64 + 32 * h + 31, kTmemCols) && DLR_IN(kTY2 + 32 * h + 31, kTmemCols)) {
    tc::tmem_ld32(lane_base + kTY1 + par * 64 + 32 * h, y1);
    tc::tmem_ld32(lane_base + kTY2 + 32 * h, y2);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) y1[i] = y2[i] = 0.f;
  }
  tc::fence_before_sync();
  tc::mbar_arrive(&bars[kBarY1Free + par]);
  tc::mbar_arrive(&bars[kBarY2Free]);
  const bool sc_in = DLR_IN(slot * 128 + g, 512);
  const float ay = sc_in ? reinterpret_cast<const float*>(sm + kAy)[slot * 128 + g] : 0.f;
  const float by = sc_in ? reinterpret_cast<const float*>(sm + kBy)[slot * 128 + g] : 0.f;
  float y[32];  // y1 * ay + y2 * by, two outputs per instruction
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 t = __fmul2_rn(make_float2(y2[i], y2[i + 1]), make_float2(by, by));
    const float2 r = __ffma2_rn(make_float2(y1[i], y1[i + 1]), make_float2(ay, ay), t);
    y[i] = r.x;
    y[i + 1] = r.y;
  }
  const ColInfo ci = col_info(a, ti, rc);
  if (a.tma) {
    uint8_t* stg = sm + kYStage + warp * 4096;
    if (lane == 0) tc::bulk_wait_group_read0();  // this warp's previous tile left the image
    __syncwarp();
    const int line = kRev ? 31 - lane : lane;
    const uint32_t sw = uint32_t(line & 7);
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // steps 4q .. 4q + 3 of the half (reversed when kRev)
      const float4 v = kRev ? make_float4(y[31 - 4 * q], y[30 - 4 * q], y[29 - 4 * q],
                                          y[28 - 4 * q])
                            : make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
      if (DLR_IN(warp * 4096 + line * 128 + 127, 8 * 4096))
        *reinterpret_cast<float4*>(stg + line * 128 + ((uint32_t(q) ^ sw) << 4)) = v;
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && ci.valid) {
      // 32 chunks of one row, chunks ci.c .. ci.c + 31 (reversed: forward chunks from C-32-c),
      // steps 32h .. 32h + 31 (reversed: forward steps 32(1-h) .. 32(1-h) + 31)
      const int z = (ti.b0 + ci.rl) * a.H + ti.h;
      const int yc = kRev ? a.C - 32 - ci.c : ci.c;
      const int x = kRev ? 32 * (1 - h) : 32 * h;
      if (kRev) tc::tma_reduce_add_3d(ymap, stg, x, yc, z);
      else tc::tma_store_3d(ymap, stg, x, yc, z);
      tc::bulk_commit_group();
    }
  } else if (ci.valid) {
    store_part<kRev>(a.y + ci.rowoff, a.L, ci.k0 + 32 * h, y);
  }
  if (threadIdx.x == 0) SCAN_TRACE(2000 + j * 8 + 2);
  return true;
}

// GEMM1 of tile k with the Toeplitz part of GEMM2 (both need only the u operand):
// S = Q u^T into S buffer k & 1 (A = Q from TMEM), Y1 = u Tk^T into Y1 buffer k & 1.
__device__ __forceinline__ void gemm1(uint8_t* sm, uint32_t tmem, int k) {
  const int par = k & 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  SCAN_TRACE(3000 + k * 4 + 0);
  tc::fence_after_sync();
  constexpr uint32_t id1 = tc::idesc_f16_f32(128, 128);
  constexpr uint32_t idk = tc::idesc_f16_f32(128, 64);
  const uint8_t* ubuf = sm + kU + par * kUBuf;
  const uint64_t uh = tc::smem_desc_k_sw128(ubuf), ul = tc::smem_desc_k_sw128(ubuf + kULo);
  const uint64_t th = tc::smem_desc_k_sw128(sm + kTkHi), tl = tc::smem_desc_k_sw128(sm + kTkLo);
  const uint32_t dS = tmem + kTS + uint32_t(par) * 128;
  const uint32_t dY1 = tmem + kTY1 + uint32_t(par) * 64;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t qh = tmem + kTQ + kk * 8, ql = tmem + kTQ + 32 + kk * 8;
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
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    tc::mma_kind_f16(dY1, uh + 2 * kk, th + 2 * kk, idk, kk != 0);
    tc::mma_kind_f16(dY1, uh + 2 * kk, tl + 2 * kk, idk, 1);
    tc::mma_kind_f16(dY1, ul + 2 * kk, th + 2 * kk, idk, 1);
  }
  tc::mma_commit(&bars[kBarG1 + par]);
}

// GEMM2 (state part) of tile k: Y2 = Xin G^T.
__device__ __forceinline__ void gemm2(uint8_t* sm, uint32_t tmem, int k) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  SCAN_TRACE(3000 + k * 4 + 1);
  tc::fence_after_sync();
  constexpr uint32_t idm = tc::idesc_f16_f32(128, 64) | (1u << 15);  // A (Xin) MN-major
  const uint64_t gh = tc::smem_desc_k_sw128(sm + kGHi), gl = tc::smem_desc_k_sw128(sm + kGLo);
  const uint64_t xh = tc::smem_desc_mn_sw128(sm + kXHi, 1024, 2048);
  const uint64_t xl = tc::smem_desc_mn_sw128(sm + kXLo, 1024, 2048);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint64_t ao = uint64_t(s) * (4096 >> 4);                     // 16 rows = 2 K-groups
    const uint64_t bo = uint64_t(s >> 2) * (8192 >> 4) + 2 * (s & 3);  // K-block, 32 bytes
    tc::mma_kind_f16(tmem + kTY2, xh + ao, gh + bo, idm, s != 0);
    tc::mma_kind_f16(tmem + kTY2, xh + ao, gl + bo, idm, 1);
    tc::mma_kind_f16(tmem + kTY2, xl + ao, gh + bo, idm, 1);
  }
  tc::mma_commit(&bars[kBarG2]);
}

// MMA thread over all tiles of the CTA, in the order GEMM1 of tile k+1, GEMM2 of tile k. At a
// change of channel GEMM1 waits for the producer's copy of the Toeplitz operand and GEMM2 for
// its copy of G. Returns false on abort.
__device__ __forceinline__ bool mma_g1(uint8_t* sm, uint32_t tmem, int h, int k, int& tk_h,
                                       uint32_t& tk_n, volatile int* abort) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const int par = k & 1;
  if (h != tk_h) {  // the Toeplitz operand of a new channel (copied by the producer)
    if (!wait_phase(&bars[kBarTabTk], tk_n & 1, abort)) return false;
    ++tk_n;
    tk_h = h;
  }
  // u of tile k written; the Y1 buffer read out (tile k-2). The S buffer of tile k-2 was read
  // by the chain before it released Xin of that tile, which this thread waited for before
  // issuing GEMM2 of tile k-2 (program order: GEMM1 k, GEMM2 k-1, GEMM1 k+1, ...).
  if (!wait_phase(&bars[kBarUFull + par], (k >> 1) & 1, abort)) return false;
  if (k >= 2 && !wait_phase(&bars[kBarY1Free + par], ((k - 2) >> 1) & 1, abort)) return false;
  gemm1(sm, tmem, k);
  return true;
}

__device__ __forceinline__ bool mma_g2(uint8_t* sm, uint32_t tmem, int h, int k, int& g_h,
                                       uint32_t& g_n, volatile int* abort) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  if (h != g_h) {  // the G operand of a new channel (copied by the producer)
    if (!wait_phase(&bars[kBarTabG], g_n & 1, abort)) return false;
    ++g_n;
    g_h = h;
  }
  SCAN_TRACE(3000 + k * 4 + 2);
  if (!wait_phase(&bars[kBarXFull], k & 1, abort)) return false;
  if (k >= 1 && !wait_phase(&bars[kBarY2Free], (k - 1) & 1, abort)) return false;
  gemm2(sm, tmem, k);
  return true;
}

// MMA thread over all tiles of the CTA, in the order GEMM1 of tile k+1, GEMM2 of tile k. At a
// change of channel GEMM1 waits for the producer's copy of the Toeplitz operand and GEMM2 for
// its copy of G.
__device__ __forceinline__ void mma_role(const TcScanArgs& a, uint8_t* sm, uint32_t tmem,
                                         int u0, int segs, int ntiles, volatile int* abort) {
  int tk_h = -1, g_h = -1;
  uint32_t tk_n = 0, g_n = 0;
  if (ntiles == 0) return;
  TileIter it1 = tile_iter_begin(a, u0), it2 = it1;
  if (!mma_g1(sm, tmem, it1.t.h, 0, tk_h, tk_n, abort)) return;
  for (int k = 0; k < ntiles; ++k) {
    if (k + 1 < ntiles) {
      tile_iter_next(a, segs, it1);
      if (!mma_g1(sm, tmem, it1.t.h, k + 1, tk_h, tk_n, abort)) return;
    }
    if (!mma_g2(sm, tmem, it2.t.h, k, g_h, g_n, abort)) return;
    tile_iter_next(a, segs, it2);
  }
}

// ---- the chain ---------------------------------------------------------------------------
// Xin leaves the scan as X * 2^-xs, X in the S units of its tile (true state * 2^(es + 14)).
// Within a tile |S| <= 64 * 2^14 * 2^14 per component, so a state that starts the tile at zero
// stays below 127 * 2^34.5 < 2^41.5 and xs = 27 keeps Xin below 2^14.5, inside the f16 range
// with room for the rounding of the split; a state carried in from the previous tile of a long
// row raises xs by the excess of its bound over 2^41. Values far below the bound lose nothing
// that matters: the f16 pair resolves 2^-24 absolute, i.e. 2^-24 of the row's largest |u|.
constexpr int kXinShift = 27;

// lambda^64 and the re-anchoring correction of the thread's state in (own, other) components:
// the Im thread of a state pair runs the recurrence with the imaginary parts negated.
struct ChainConst {
  float mu_re, mu_im, dl_re, dl_im;
};
// state (xo, xt) <- mu * state + (s_own, s_oth)
__device__ __forceinline__ void chain_step(const ChainConst& q, float s_own, float s_oth,
                                           float& xo, float& xt) {
  const float no = fmaf(q.mu_re, xo, fmaf(-q.mu_im, xt, s_own));
  const float nt = fmaf(q.mu_re, xt, fmaf(q.mu_im, xo, s_oth));
  xo = no;
  xt = nt;
}
// re-anchoring at a 32-chunk boundary: state += (lambda^2048 - mu^32) * (state at the last
// anchor); the corrected state becomes the new anchor
__device__ __forceinline__ void chain_anchor(const ChainConst& q, float& xo, float& xt,
                                             float& ao, float& at) {
  xo = fmaf(q.dl_re, ao, fmaf(-q.dl_im, at, xo));
  xt = fmaf(q.dl_re, at, fmaf(q.dl_im, ao, xt));
  ao = xo;
  at = xt;
}

// Byte offset of the 16-byte chunk of an Xin buffer holding K-row r, columns g0 .. g0 + 7
// (g0 a multiple of 8): MN-major, 128-byte swizzle, atom (K-group r >> 3, MN-half g0 >> 6) at
// (r >> 3) * 2048 + (g0 >> 6) * 1024, line r & 7, chunk ((g0 >> 3) & 7) XOR (r & 7).
__device__ __forceinline__ uint32_t xin_chunk(int r, int g0) {
  const uint32_t cg = uint32_t(g0 >> 3);
  return uint32_t(r >> 3) * 2048u + (cg >> 3) * 1024u + uint32_t(r & 7) * 128u +
         (((cg & 7u) ^ uint32_t(r & 7)) << 4);
}
// Eight Xin values of K-row r, columns g0 .. g0 + 7, times `s`, as the f16 pair.
__device__ __forceinline__ void store_xin8(uint8_t* sm, int r, int g0, const float* v, float s) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) split2s(v[2 * q], v[2 * q + 1], s, h[q], l[q]);
  const uint32_t off = xin_chunk(r, g0);
  if (DLR_IN(off + 15, kXLo - kXHi)) {
    *reinterpret_cast<uint4*>(sm + kXHi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(sm + kXLo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// main warps, chain of tile k. Thread r owns TMEM lane r = state row r (lane quarter warp & 3)
// and runs the complex recurrence of its state pair (the other component of S comes from the
// partner lane r ^ 1; both threads of a pair run the same recurrence and each writes its own
// Xin K-row). Half h writes the Xin columns 64h .. 64h + 63. When the rows start at both
// halves (C divides 64) each half runs only its own columns; otherwise half 1 starts at the
// last row start at or before column 64 (its earlier columns are recomputed, not stored) and
// in long-row mode both halves run all 128 columns, so both carry the state into the next
// tile. Row mode resets the state at every row start (multiples of C) and re-anchors every 32
// chunks from it; long rows re-anchor every 32 chunks from the tile start. kStep: row starts
// checked at every column (C not a multiple of 16); otherwise only where a piece of 16 columns
// begins. S is read one piece ahead. The Xin buffer is free: the outputs of the previous tile,
// taken earlier in the same iteration, waited for its GEMM2.
template <bool kStep>
__device__ __forceinline__ void chain_run(const TcScanArgs& a, uint8_t* sm, uint32_t tS, int r,
                                          const ChainConst& q, float xscale, int c_begin,
                                          int c_store, int c_end, float& xo, float& xt,
                                          float& ao, float& at) {
  // the S columns read lie in TMEM (uniform over the warp; a failed check skips the chain)
  if (!DLR_IN(int(tS & 0xFFFFu) + c_end - 1, int(kTmemCols))) return;
  const int c_store_end = c_store + 64;
  int next_reset, next_anchor;
  if (a.R > 0) {
    next_reset = ((c_begin + a.C - 1) / a.C) * a.C;  // the first row start at or after c_begin
    next_anchor = next_reset;
  } else {
    next_reset = 1 << 30;
    next_anchor = 0;
  }
  uint32_t cur[16], nxt[16];
  tc::tmem_ld16_issue(tS + c_begin, cur);
  tc::tmem_wait_ld16(cur);
#pragma unroll 1
  for (int c = c_begin; c < c_end; c += 16) {
    const bool more = c + 16 < c_end;
    if (more) tc::tmem_ld16_issue(tS + c + 16, nxt);
    if (!kStep) {
      if (c == next_anchor) {
        chain_anchor(q, xo, xt, ao, at);
        next_anchor += 32;
      }
      if (c == next_reset) {
        xo = xt = ao = at = 0.f;
        next_reset += a.C;
        next_anchor = c + 32;
      }
    }
    // the partner's components of the whole piece first: the exchanges do not depend on the
    // recurrence, so their latency overlaps instead of adding to every step
    float oth[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) oth[j] = __shfl_xor_sync(0xffffffffu, __uint_as_float(cur[j]), 1);
    float oo[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float own = __uint_as_float(cur[j]);
      if (kStep) {
        const int g = c + j;
        if (g == next_anchor) {
          chain_anchor(q, xo, xt, ao, at);
          next_anchor += 32;
        }
        if (g == next_reset) {
          xo = xt = ao = at = 0.f;
          next_reset += a.C;
          next_anchor = g + 32;
        }
      }
      oo[j] = xo;
      chain_step(q, own, oth[j], xo, xt);
    }
    if (c >= c_store && c < c_store_end) {
      store_xin8(sm, r, c, oo, xscale);
      store_xin8(sm, r, c + 8, oo + 8, xscale);
    }
    if (more) {
      tc::tmem_wait_ld16(nxt);
#pragma unroll
      for (int j = 0; j < 16; ++j) cur[j] = nxt[j];
    }
  }
}

// The same for a half of the tile that is 64 columns from a row start with rows of C in
// {16, 32, 64} chunks (row starts and anchors at multiples of 16 columns): the whole half in
// registers, fully unrolled, so the conversion and stores of the first columns overlap the
// recurrence of the later ones.
__device__ __forceinline__ void chain64(uint8_t* sm, uint32_t tS, int r, int C,
                                        const ChainConst& q, float xscale, int c0) {
  if (!DLR_IN(int(tS & 0xFFFFu) + c0 + 63, int(kTmemCols))) return;
  uint32_t s0[16], s1[16], s2[16], s3[16];
  tc::tmem_ld16_issue(tS + c0, s0);
  tc::tmem_ld16_issue(tS + c0 + 16, s1);
  tc::tmem_ld16_issue(tS + c0 + 32, s2);
  tc::tmem_ld16_issue(tS + c0 + 48, s3);
  tc::tmem_wait_ld16(s0);
  tc::tmem_wait_ld16(s1);
  tc::tmem_wait_ld16(s2);
  tc::tmem_wait_ld16(s3);
  float xo = 0.f, xt = 0.f, ao = 0.f, at = 0.f;
  float out[64];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t* sp = p == 0 ? s0 : p == 1 ? s1 : p == 2 ? s2 : s3;
    float oth[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) oth[j] = __shfl_xor_sync(0xffffffffu, __uint_as_float(sp[j]), 1);
    const int cr = (16 * p) & (C - 1);  // column within the row
    if (p > 0 && cr == 0) xo = xt = ao = at = 0.f;
    if (cr == 32) chain_anchor(q, xo, xt, ao, at);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      out[16 * p + j] = xo;
      chain_step(q, __uint_as_float(sp[j]), oth[j], xo, xt);
    }
  }
#pragma unroll
  for (int g8 = 0; g8 < 8; ++g8) store_xin8(sm, r, c0 + 8 * g8, out + 8 * g8, xscale);
}

__device__ __forceinline__ bool chain_tile(const TcScanArgs& a, uint8_t* sm, uint32_t tmem,
                                           int k, bool new_row, const ChainConst& q,
                                           float sig_g, float& xo, float& xt, float& ao,
                                           float& at, int& es_prev, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = warp >> 2, quarter = warp & 3, r = quarter * 32 + lane;
  const int par = k & 1, slot = k & 3;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  const int* sRowEs = reinterpret_cast<const int*>(sm + kRowEs) + slot * 128;
  unsigned* sRed = reinterpret_cast<unsigned*>(sm + kScanRed);
  const uint32_t tS = tmem + (uint32_t(quarter * 32) << 16) + kTS + uint32_t(par) * 128;

  // S of this tile
  const bool ok = lanes_wait_phase(&bars[kBarG1 + par], (k >> 1) & 1, abort);
  tc::fence_after_sync();
  if (threadIdx.x == 0) SCAN_TRACE(k * 8 + 0);
#ifdef DLR_SCAN_TRACE
  if (threadIdx.x == 0 && blockIdx.x == 0 && k < 8) g_scan_trace[3800 + 2 * k] = clock64();
#endif

  int xs = kXinShift;
  if (a.R == 0) {
    // one row walked tile by tile: the carried state and anchor move from the previous tile's
    // S units to this tile's (times 2^(es - es_prev), in two exact steps); the Xin scale makes
    // room for the carried state's magnitude (both halves carry the same state)
    const int es = sRowEs[0];
    if (new_row) {
      xo = xt = ao = at = 0.f;
    } else {
      const int d = max(-252, min(252, es - es_prev));
      const float f = exp2i(d / 2) * exp2i(d - d / 2);
      xo *= f; xt *= f; ao *= f; at *= f;
    }
    es_prev = es;
    const unsigned mw = __reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(fabsf(xo), fabsf(xt))));
    if (lane == 0 && h == 0 && DLR_IN(quarter, 4)) sRed[quarter] = mw;
    named_bar(kMainBar, 256);
    const unsigned m = max(max(sRed[0], sRed[1]), max(sRed[2], sRed[3]));
    const int e = int((m >> 23) & 0xFFu) - 126;  // carried |state| < 2^e
    xs += max(0, e - 41);
  } else {
    xo = xt = ao = at = 0.f;
  }
  if (h == 0) {
    // y = Y2 * 2^(xs - 14 - es) / sig_g for the column's row
    const int row = (a.R > 0) ? r / a.C : 0;
    if (DLR_IN(slot * 128 + r, 512)) reinterpret_cast<float*>(sm + kBy)[slot * 128 + r] =
        exp2i(xs - kXinShift) * exp2i(kXinShift - 14 - sRowEs[row]) / sig_g;
  }
  const float xscale = exp2i(-xs);
  int c_begin, c_end;
  if (a.R > 0 && (64 % a.C) == 0) {
    c_begin = 64 * h;
    c_end = 64 * h + 64;
  } else if (a.R > 0) {
    c_begin = h ? ((64 / a.C) * a.C) & ~15 : 0;
    c_end = 64 * h + 64;
  } else {
    c_begin = 0;
    c_end = kCols;
  }
  if (a.R > 0 && (a.C == 16 || a.C == 32 || a.C == 64))
    chain64(sm, tS, r, a.C, q, xscale, 64 * h);
  else if (a.R > 0 && (a.C & 15) != 0)
    chain_run<true>(a, sm, tS, r, q, xscale, c_begin, 64 * h, c_end, xo, xt, ao, at);
  else
    chain_run<false>(a, sm, tS, r, q, xscale, c_begin, 64 * h, c_end, xo, xt, ao, at);
  if (threadIdx.x == 0) SCAN_TRACE(k * 8 + 3);
#ifdef DLR_SCAN_TRACE
  if (threadIdx.x == 0 && blockIdx.x == 0 && k < 8) g_scan_trace[3801 + 2 * k] = clock64();
#endif
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  tc::mbar_arrive(&bars[kBarXFull]);
  return true;
}

// The main warps (0-7) over all tiles of the CTA. Iteration k: the u operand of tile k+1, the
// outputs of tile k-1 (once its GEMM2 is done), the chain of tile k. The scale slots are rings
// of four tiles, so tile k+1's u scales never overwrite those tile k-1's outputs still read.
// Each warp takes its waits on its own (lanes_wait_phase); the warps meet only at the named
// barriers of the u conversion and at the top of each iteration.
template <bool kRev>
__device__ __forceinline__ void main_role(const TcScanArgs& a, const CUtensorMap* ymap,
                                          uint8_t* sm, uint32_t tmem, int u0, int segs,
                                          int ntiles, volatile int* abort) {
  const int r = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);  // lane = chunk or row
  const int2 rc = col_rows(a, r);
  int conv_h = -1;
  float sig_k = 1.f;
  ChainConst q{0.f, 0.f, 0.f, 0.f};
  float sig_g = 1.f;
  float xo = 0.f, xt = 0.f, ao = 0.f, at = 0.f;
  int es_prev = 0;
  int chain_h = -1;
  if (ntiles == 0) return;
  TileIter it_conv = tile_iter_begin(a, u0), it_epi = it_conv, it_chain = it_conv;
  conv_tile<kRev>(a, sm, tmem, it_conv.t, rc, 0, conv_h, sig_k, abort);
  tile_iter_next(a, segs, it_conv);
  // Every warp runs the whole schedule even after an abort (its waits then return at once), so
  // the named barriers below are always reached by all 256 threads.
  for (int k = 0; k < ntiles; ++k) {
    named_bar(kMainBar, 256);  // the previous stages' shared-memory writes are visible
    if (k + 1 < ntiles) {
      conv_tile<kRev>(a, sm, tmem, it_conv.t, rc, k + 1, conv_h, sig_k, abort);
      tile_iter_next(a, segs, it_conv);
    }
    if (k >= 1) {
      epi_tile<kRev>(a, ymap, sm, tmem, it_epi.t, rc, k - 1, abort);
      tile_iter_next(a, segs, it_epi);
    }
    const TileInfo& ti = it_chain.t;
    if (ti.h != chain_h) {
      // this thread's lambda^64 and re-anchoring correction; the G scale of the channel. The
      // state recurrence keeps (own, other) components; the Im row runs it with the sign of the
      // imaginary parts flipped.
      chain_h = ti.h;
      const uint8_t* blob = a.tables + (size_t)ti.h * kBlobBytes;
      const float4 m =
          __ldg(reinterpret_cast<const float4*>(blob + kBlobMu) + (DLR_IN(r >> 1, 64) ? r >> 1 : 0));
      q.mu_re = m.x;
      q.dl_re = m.z;
      q.mu_im = (r & 1) ? -m.y : m.y;
      q.dl_im = (r & 1) ? -m.w : m.w;
      sig_g = __ldg(reinterpret_cast<const float*>(blob + kBlobSig) + 1);
    }
    chain_tile(a, sm, tmem, k, ti.seg == 0, q, sig_g, xo, xt, ao, at, es_prev, abort);
    tile_iter_next(a, segs, it_chain);
  }
  named_bar(kMainBar, 256);
  epi_tile<kRev>(a, ymap, sm, tmem, it_epi.t, rc, ntiles - 1, abort);
  if (a.tma && (threadIdx.x & 31) == 0) tc::bulk_wait_group0();  // y stores done
}

template <bool kRev>
__global__ void __launch_bounds__(kThreads, 1)
    dlr_scan_tc_kernel(const TcScanArgs a, const __grid_constant__ CUtensorMap umap,
                       const __grid_constant__ CUtensorMap ymap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kAbort);

  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) SCAN_TRACE(3999);
  if (tid == 0 && blockIdx.x < 192) SCAN_TRACE_ALL(3600 + blockIdx.x);
  if (tid == 0) {
    tc::mbar_init(&bars[kBarTabTk], 1);
    tc::mbar_init(&bars[kBarTabG], 1);
    tc::mbar_init(&bars[kBarG2], 1);
    tc::mbar_init(&bars[kBarXFull], 256);
    tc::mbar_init(&bars[kBarY2Free], 256);
    for (int p = 0; p < 2; ++p) {
      tc::mbar_init(&bars[kBarStage + p], 1);
      tc::mbar_init(&bars[kBarUFull + p], 256);
      tc::mbar_init(&bars[kBarG1 + p], 1);
      tc::mbar_init(&bars[kBarY1Free + p], 256);
    }
    *abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid < 128) reinterpret_cast<unsigned*>(sm + kRowMaxU)[tid] = 0u;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  const int u0 = (int)((long long)blockIdx.x * a.units / gridDim.x);
  const int u1 = (int)((long long)(blockIdx.x + 1) * a.units / gridDim.x);
  const int segs = (a.R > 0) ? 1 : (a.C + kCols - 1) / kCols;
  const int ntiles = (u1 - u0) * segs;

  // The tables written by the table kernel are read by the producer's copies (it waits for the
  // table kernel after issuing its first u copies) and by the main warps (they wait at their
  // first read, in conv_tile); the MMA thread reads only what those two produce.
  if (warp < 8) {
    main_role<kRev>(a, &ymap, sm, tmem, u0, segs, ntiles, abort);
  } else if (warp == 8) {
    if ((tid & 31) == 0) mma_role(a, sm, tmem, u0, segs, ntiles, abort);
  } else if ((tid & 31) == 0) {
    producer_role<kRev>(a, &umap, sm, u0, segs, ntiles, abort);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) SCAN_TRACE(3997);
  if (tid == 0 && blockIdx.x < 192) SCAN_TRACE_ALL(3400 + blockIdx.x);
  if (*abort) report_status(a.status, DLR_ERR_TIMEOUT);
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

// 3D view of u (or y) for the TMA copies: [64 steps][C chunks][B*H rows], boxes of 32 steps x
// bc chunks x 1 row, 128-byte swizzle (one 128-byte line per chunk and half).
bool make_u_map(CUtensorMap* m, const float* u, int B, int H, int L, int bc) {
  auto fn = tc::tensor_map_encoder();
  if (!fn) return false;
  const int C = L / kT;
  cuuint64_t dims[3] = {(cuuint64_t)kT, (cuuint64_t)C, (cuuint64_t)B * (cuuint64_t)H};
  cuuint64_t strides[2] = {(cuuint64_t)kT * 4, (cuuint64_t)L * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)bc, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(u), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <bool kRev>
cudaError_t launch_main(const TcScanArgs& a, const CUtensorMap& umap, const CUtensorMap& ymap,
                        bool after_tables, cudaStream_t s) {
  cudaError_t e = max_smem_once<dlr_scan_tc_kernel<kRev>>(kSmemBytes);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorUnknown;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)std::min(a.units, sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  // Right after this library's table kernel (which writes only the tables and started after all
  // earlier work, so u is final) the scan kernel is launched as its programmatic dependent: its
  // prologue and first u copies overlap the table kernel's tail, and it waits for the tables
  // in the kernel. After anything else it is launched normally.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_tables ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, dlr_scan_tc_kernel<kRev>, a, umap, ymap);
}

}  // namespace

size_t scan_tc_workspace_bytes(int64_t H) { return (size_t)H * kBlobBytes; }

// The channel tables of one parameter set (N <= 64 states) into the workspace.
cudaError_t launch_scan_tc_tables(const float* lr, const float* li, const float* W, int H, int N,
                                  void* ws, cudaStream_t s) {
  TcScanArgs a{};
  a.H = H;
  a.N = N;
  a.log_re = lr;
  a.log_im = li;
  a.W = reinterpret_cast<const float2*>(W);
  cudaError_t e = max_smem_once<dlr_scan_tc_tables>(kTbBytes);
  if (e != cudaSuccess) return e;
  dlr_scan_tc_tables<<<H, kTbThreads, kTbBytes, s>>>(a, static_cast<uint8_t*>(ws));
  return cudaGetLastError();
}

// The layer on u [B, H, L] with the tables in the workspace: y = DLR(u), or (reverse) y +=
// rev(DLR(rev(u))).
cudaError_t launch_scan_tc_apply(const float* u, int B, int H, int L, bool reverse, float* y,
                                 const void* ws, int* status, cudaStream_t s,
                                 bool after_tables) {
  TcScanArgs a{};
  a.u = u;
  a.y = y;
  a.B = B;
  a.H = H;
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
  // u tiles by TMA when every row is whole chunks and a tile's rows are whole boxes
  const bool tma_shape = (L % kT == 0) && ((a.R > 0) ? (a.C == 32 || a.C == 64 || a.C == 128)
                                                      : (a.C % 64 == 0));
  a.bc = (a.C == 32) ? 32 : 64;
  CUtensorMap umap, ymap;
  std::memset(&umap, 0, sizeof(umap));
  std::memset(&ymap, 0, sizeof(ymap));
  a.tma = tma_shape && make_u_map(&umap, u, B, H, L, a.bc) && make_u_map(&ymap, y, B, H, L, 32)
              ? 1
              : 0;
  return reverse ? launch_main<true>(a, umap, ymap, after_tables, s)
                 : launch_main<false>(a, umap, ymap, after_tables, s);
}

// N <= 64 complex states; u, y [B, H, L]; bidirectional adds the reversed pass (run after the
// forward one, reusing the workspace for its tables).
cudaError_t launch_dlr_scan_tc(const float* u, const float* lr, const float* li, const float* W,
                               const float* lr2, const float* li2, const float* W2, bool bidir,
                               int B, int H, int N, int L, float* y, void* ws, int* status,
                               cudaStream_t s) {
  cudaError_t e = launch_scan_tc_tables(lr, li, W, H, N, ws, s);
  if (e == cudaSuccess) e = launch_scan_tc_apply(u, B, H, L, false, y, ws, status, s, true);
  if (e != cudaSuccess || !bidir) return e;
  e = launch_scan_tc_tables(lr2, li2, W2, H, N, ws, s);
  if (e == cudaSuccess) e = launch_scan_tc_apply(u, B, H, L, true, y, ws, status, s, true);
  return e;
}

}  // namespace dlr
