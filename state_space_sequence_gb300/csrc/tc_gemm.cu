// tc_gemm.cu -- C[M, N] (f32 or bf16) = A[M, K] * B[N, K]^T (+ D[n] * E[m, n]) on 5th-generation
// tensor cores: bf16 operands in shared memory (TMA tile loads, 128-byte swizzle; a float32 A
// is converted to bf16 in the kernel), f32 accumulators in tensor memory, tcgen05.mma
// (kind::f16) issued by one thread, tcgen05.ld epilogue with TMA tile stores.
//
// Persistent: one CTA per SM walks the 128 x 256 output tiles t = blockIdx.x, + gridDim.x, ...
// with the N tile varying fastest (the CTAs working on the N tiles of one M tile at the same
// time share its A rows through L2). Warps:
//   warp 0 lane 0  TMA producer: K-blocks of 64 into a ring of 3-4 stages (A 16 KB + B 32 KB),
//                  running ahead across tiles. With a float32 A a stage holds A as float32
//                  (two 16 KB boxes per K-block) and B; warp 0 then loads only A, and
//   warp 3 lane 0  loads B,
//   warps 8-11     (float32 A only) convert in place: thread = row r of the tile reads the 64
//                  float32 of its row and writes them as 64 bf16 over the first 16 KB of the
//                  stage, in the operand layout (row r is read and written by thread r only),
//   warps 8-13     (A = the S5 scan's V only) turn the A tile of each ring stage in place into
//                  the scan's states, two warps per stage (one per chunk of 64 rows), lane =
//                  state,
//   warp 1 lane 0  MMA issuer: four K=16 MMAs per K-block, a commit that frees the stage, and
//                  per tile a commit that hands one of two TMEM accumulators to the epilogue,
//   warp 2         allocates / frees the 512 TMEM columns (two 256-column accumulators),
//   warps 4-7      epilogue: warp 4+q owns TMEM lanes 32q..32q+31 (rows of the tile). Per slice
//                  of 128 output bytes per row (32 f32 or 64 bf16 columns): tcgen05.ld, + D (.) E
//                  with the E box brought in by TMA, into a 4 KB staging box (128-byte swizzle),
//                  out by one TMA store per warp. The boxes of a warp rotate: the E loads of the
//                  next two slices and the stores of the last one or two are in flight while the
//                  current slice is worked on.
// While the epilogue drains one accumulator the MMAs of the next tile fill the other.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 14;
namespace {

constexpr int kBM = 128, kBN = 256;
constexpr int kRowBytes = 128;  // K bytes of one operand row per stage (the swizzle span)
constexpr uint32_t kABytes = kBM * kRowBytes, kBBytes = kBN * kRowBytes;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kBoxBytes = 32 * 128;  // 32 rows x 128 bytes

// Operand modes, all kind::f16 with bf16 operands in shared memory:
//   kOpBf16   A and B bf16 in global memory;
//   kOpCvtA   A float32 in global memory, converted to bf16 by four converter warps;
//   kOpApply  A = the chunked scan's per-step input V (bf16), turned in place into the states
//             x_t = lambda x_{t-1} + V_t (restarting from the carried state at every chunk of
//             64 steps) by two converter warps per ring stage (one per chunk) before the MMAs
//             read it.
enum OpMode { kOpBf16 = 0, kOpCvtA = 1, kOpApply = 2 };

// Shared-memory plan. With E the epilogue keeps four boxes per warp (two E loads ahead) and
// the ring three stages; without E two boxes suffice and the ring gets a fourth stage. With a
// float32 A a stage is 64 KB (A as float32, later bf16 in its first half, then B) and the ring
// has three.
template <bool kWithE, int kOp>
struct Plan {
  static constexpr bool kCvt = kOp == kOpCvtA;
  static constexpr int kStages = kCvt ? 3 : (kWithE ? 3 : 4);
  static constexpr uint32_t kFBytes = kBM * 2 * kRowBytes;  // 128 rows x 64 float32
  static constexpr uint32_t kBOff = kCvt ? kFBytes : kABytes;  // B within a stage
  static constexpr uint32_t kStride = kBOff + kBBytes;        // stage size
  static constexpr int kBoxes = kWithE ? 4 : 2;
  static constexpr uint32_t kEpiOff = kStages * kStride;
  static constexpr uint32_t kBarOff = kEpiOff + 4 * kBoxes * kBoxBytes;
  static constexpr size_t kSmemBytes = 1024 + kBarOff + 256;
  static constexpr int kThreads = kOp == kOpBf16 ? 256 : (kOp == kOpCvtA ? 384 : 448);
  static_assert(kSmemBytes <= 232448, "shared memory");
};
constexpr uint32_t kTmemCols = 512;

struct GemmArgs {
  int M, N, K;
  const float* D;  // [N] or null (then E is not read)
  int* status;
  // kOpApply: lambda per state, the state entering each chunk [B][NC][P], sequence length
  // (a multiple of 64), states P (A has K = 2P columns: Re, Im per state), chunks per row.
  // With `sums` (bf16 output, N = 2P, L a multiple of 64) the epilogue also writes, per 32-row
  // block of each chunk, sum_i lambda^(31-i) C[row i] of the bf16-rounded outputs:
  // sums[b][c][half][p].
  const float2* lam;
  const float2* xin;
  int L, P, NC;
  float2* sums;
};

// Bounded wait by a whole warp with one verdict for all its lanes.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity)) != 0;
}

template <int kOp, bool kWithE, bool kBf16Out>
__global__ void __launch_bounds__(Plan<kWithE, kOp>::kThreads, 1)
tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmE,
             GemmArgs g) {
  static_assert(!(kWithE && kBf16Out), "D (.) E is added to f32 outputs only");
  static_assert(!(kWithE && kOp == kOpCvtA), "no plan for E with a converted A");
  constexpr bool kCvt = kOp == kOpCvtA, kApply = kOp == kOpApply;
  using PL = Plan<kWithE, kOp>;
  constexpr int kStages = PL::kStages, kBoxes = PL::kBoxes;
  constexpr int kSlice = kBf16Out ? 64 : 32;  // output columns per slice (128 bytes per row)
  constexpr int kSlices = kBN / kSlice;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + PL::kBarOff);
  uint64_t* full = bars;                       // [kStages]  operands (B only with kCvt) landed
  uint64_t* empty = bars + kStages;            // [kStages]  operands consumed by the MMAs
  uint64_t* acc_full = bars + 2 * kStages;     // [2]        accumulator complete
  uint64_t* acc_empty = acc_full + 2;          // [2]        accumulator read out (4 arrivals)
  uint64_t* e_full = acc_empty + 2;            // [4][kBoxes] E box landed
  uint64_t* a_ready = e_full + 4 * kBoxes;     // [kStages]  converted A written (4 arrivals)
  uint64_t* f_full = a_ready + kStages;        // [kStages]  float32 A landed (kCvt)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(f_full + kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (g.N + kBN - 1) / kBN;
  const int tiles = n_tiles * ((g.M + kBM - 1) / kBM);
  constexpr int kBK = kRowBytes / 2;  // K elements (bf16) per stage
  const int nk = (g.K + kBK - 1) / kBK;
  constexpr bool with_e = kWithE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);
    }
    for (int i = 0; i < 4 * kBoxes; ++i) tc::mbar_init(&e_full[i], 1);
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&a_ready[s], kCvt ? 4 : 2);
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&f_full[s], 1);
    tc::mbar_fence_init();
  }
  if (warp == 2) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    if constexpr (!kCvt) {
      uint32_t it = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (t / n_tiles) * kBM, n0 = (t % n_tiles) * kBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !(ok = tc::mbar_wait(&empty[s], ((it / kStages) - 1) & 1))) break;
          uint8_t* a = base + s * PL::kStride;
          tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
          tc::tma_load_2d(a, &tmA, kb * kBK, m0, &full[s]);
          tc::tma_load_2d(a + PL::kBOff, &tmB, kb * kBK, n0, &full[s]);
        }
      }
      // before the CTA may exit, every copy it issued has landed (normally long since consumed)
      for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
        ok &= tc::mbar_wait(&full[j % kStages], (j / kStages) & 1);
    } else {
      // converted A: float32 K-blocks of 64 (two 128-byte boxes) into the stage
      uint32_t it = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (t / n_tiles) * kBM;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !(ok = tc::mbar_wait(&empty[s], ((it / kStages) - 1) & 1))) break;
          uint8_t* f = base + s * PL::kStride;
          tc::mbar_arrive_expect_tx(&f_full[s], PL::kFBytes);
          tc::tma_load_2d(f, &tmA, kb * kBK, m0, &f_full[s]);
          tc::tma_load_2d(f + PL::kFBytes / 2, &tmA, kb * kBK + kBK / 2, m0, &f_full[s]);
        }
      }
      for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
        ok &= tc::mbar_wait(&f_full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == 3 && lane == 0) {
    if constexpr (kCvt) {
      // converted A: the B operand into the ring
      uint32_t it = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int n0 = (t % n_tiles) * kBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !(ok = tc::mbar_wait(&empty[s], ((it / kStages) - 1) & 1))) break;
          tc::mbar_arrive_expect_tx(&full[s], kBBytes);
          tc::tma_load_2d(base + s * PL::kStride + PL::kBOff, &tmB, kb * kBK, n0, &full[s]);
        }
      }
      for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
        ok &= tc::mbar_wait(&full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp >= 8) {
    if constexpr (kCvt) {
      // converters: thread = row r of the tile; 64 float32 of row r -> 64 bf16 in the K-major
      // 128-byte-swizzled layout the MMA reads (16-byte chunk c of row r at (c ^ (r & 7)) << 4),
      // written over row r of the first float32 box (read by this thread alone)
      const int r = (warp - 8) * 32 + lane;
      const uint32_t sw = uint32_t(r & 7);
      uint32_t it = 0;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < nk && ok; ++kb, ++it) {
          const int s = it % kStages;
          if (!(ok = warp_wait(&f_full[s], (it / kStages) & 1))) break;
          uint8_t* f = base + s * PL::kStride + r * kRowBytes;
          float4 v[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            v[c] = *reinterpret_cast<const float4*>(f + (c >> 3) * (PL::kFBytes / 2) +
                                                    (((uint32_t(c) & 7u) ^ sw) << 4));
          uint4 h[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(v[2 * c].x, v[2 * c].y);
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(v[2 * c].z, v[2 * c].w);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * c + 1].x, v[2 * c + 1].y);
            const __nv_bfloat162 b3 = __floats2bfloat162_rn(v[2 * c + 1].z, v[2 * c + 1].w);
            h[c] = make_uint4(*reinterpret_cast<const uint32_t*>(&b0),
                              *reinterpret_cast<const uint32_t*>(&b1),
                              *reinterpret_cast<const uint32_t*>(&b2),
                              *reinterpret_cast<const uint32_t*>(&b3));
          }
          if (DLR_IN(r, kBM)) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(f + ((uint32_t(c) ^ sw) << 4)) = h[c];
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&a_ready[s]);
        }
      }
    } else if constexpr (kApply) {
      // warps 8 + 2s and 9 + 2s own ring stage s (so each waits every phase of its barriers in
      // order), one chunk of 64 rows each: tiles start on chunk starts (L a multiple of 64), so
      // rows 0 and 64 of a tile begin chunks and take the carried state. Lane j holds state
      // p = 32 kb + j: the 4 bytes (Re, Im in bf16) at byte 4 (j & 3) of 16-byte chunk j >> 2
      // of every row. The carried state and lambda of the warp's next stage are fetched while
      // it works on the current one.
      const int s = (warp - 8) >> 1, h = (warp - 8) & 1;
      if (s < kStages) {
        const uint32_t sub = uint32_t(lane & 3) * 4u, chunk = uint32_t(lane >> 2);
        // carried state and lambda for ring iteration it (zero where the rows or states end)
        auto fetch = [&](uint32_t it, cf& lam, cf& x) {
          lam = {0.f, 0.f};
          x = {0.f, 0.f};
          const int tt = blockIdx.x + int(it / nk) * gridDim.x, kb = int(it % nk);
          if (tt >= tiles) return;
          const int m = (tt / n_tiles) * kBM + h * 64, p = kb * 32 + lane;
          if (m >= g.M || p >= g.P) return;
          const int b = m / g.L, t = m - b * g.L;
          const float2 l = g.lam[p], v = g.xin[((size_t)b * g.NC + (t >> 6)) * g.P + p];
          lam = {l.x, l.y};
          x = {v.x, v.y};
        };
        const uint32_t total = uint32_t((tiles - int(blockIdx.x) + int(gridDim.x) - 1) /
                                        int(gridDim.x)) * uint32_t(nk);
        cf lam, x, lam_n, x_n;
        fetch(uint32_t(s), lam, x);
        for (uint32_t it = uint32_t(s); it < total && ok; it += kStages) {
          fetch(it + kStages, lam_n, x_n);
          if (!(ok = warp_wait(&full[s], (it / kStages) & 1))) break;
          const int m0 = (blockIdx.x + int(it / nk) * gridDim.x) / n_tiles * kBM + h * 64;
          const int rows = min(64, g.M - m0);
          uint8_t* a = base + s * PL::kStride;
#pragma unroll 1
          for (int i0 = h * 64; i0 < h * 64 + rows; i0 += 16) {
            uint32_t* ptr[16];
            uint32_t v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int i = DLR_IN(i0 + j, kBM) ? i0 + j : 0;
              ptr[j] = reinterpret_cast<uint32_t*>(a + i * kRowBytes +
                                                   ((chunk ^ uint32_t(i & 7)) << 4) + sub);
              v[j] = *ptr[j];
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 vf =
                  __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v[j]));
              x = cfma(lam, x, {vf.x, vf.y});
              const __nv_bfloat162 hx = __floats2bfloat162_rn(x.re, x.im);
              if (i0 + j < h * 64 + rows) *ptr[j] = *reinterpret_cast<const uint32_t*>(&hx);
            }
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&a_ready[s]);
          lam = lam_n;
          x = x_n;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
    uint32_t it = 0, local = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
      const uint32_t acc = local & 1;
      if (local >= 2 && !(ok = tc::mbar_wait(&acc_empty[acc], ((local >> 1) - 1) & 1))) break;
      tc::fence_after_sync();
      const uint32_t d = tmem + acc * kBN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = it % kStages;
        if (!(ok = tc::mbar_wait(&full[s], (it / kStages) & 1))) break;
        if ((kCvt || kApply) && !(ok = tc::mbar_wait(&a_ready[s], (it / kStages) & 1))) break;
        tc::fence_after_sync();
        const uint8_t* a = base + s * PL::kStride;
        const uint64_t ad = tc::smem_desc_k_sw128(a);
        const uint64_t bd = tc::smem_desc_k_sw128(a + PL::kBOff);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // advance 16 bf16 = 32 bytes = 2 descriptor units
          tc::mma_kind_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(&acc_full[acc]);
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    uint8_t* boxes = base + PL::kEpiOff + q * kBoxes * kBoxBytes;
    uint64_t* ebar = e_full + q * kBoxes;
    const uint32_t sw = uint32_t(lane & 7);
    // the slices this warp walks: (tile, column block), tiles in the CTA's order
    int t = blockIdx.x, c = 0;
    auto n_slices = [&](int tt) {
      return min(kSlices, (g.N - (tt % n_tiles) * kBN + kSlice - 1) / kSlice);
    };
    auto issue_e = [&](int tt, int cc, uint32_t sc) {
      const int j = sc % kBoxes;
      tc::mbar_arrive_expect_tx(&ebar[j], kBoxBytes);
      tc::tma_load_2d(boxes + j * kBoxBytes, &tmE, (tt % n_tiles) * kBN + cc * kSlice,
                      (tt / n_tiles) * kBM + q * 32, &ebar[j]);
    };
    // advances (tt, cc) to the next slice of the walk over the CTA's tiles
    auto ahead = [&](int& tt, int& cc) {
      if (++cc == n_slices(tt)) { tt += gridDim.x; cc = 0; }
    };
    uint32_t sc = 0, local = 0, e_issued = 0;
    int tp = t, cp = 0;  // the next slice whose E box is not yet requested
    if (with_e && lane == 0)
      for (int i = 0; i < 2 && tp < tiles; ++i, ahead(tp, cp)) issue_e(tp, cp, e_issued++);
    for (; t < tiles && ok; t += gridDim.x, ++local) {
      const uint32_t acc = local & 1;
      if (!(ok = warp_wait(&acc_full[acc], (local >> 1) & 1))) break;
      tc::fence_after_sync();
      const int m0 = (t / n_tiles) * kBM, n0 = (t % n_tiles) * kBN;
      const int ns = n_slices(t);
      for (c = 0; c < ns; ++c, ++sc) {
        const int j = sc % kBoxes;
        uint8_t* box = boxes + j * kBoxBytes;
        if (lane == 0) {
          // with E the box of slice sc + 2 held slice sc - 2, without E the box of slice sc
          // did: that store must have read it
          tc::bulk_wait_group_read<1>();
          if (with_e && tp < tiles) {
            issue_e(tp, cp, e_issued++);
            ahead(tp, cp);
          }
        }
        __syncwarp();
        const uint32_t tcol = tmem + acc * kBN + (uint32_t(q * 32) << 16) + uint32_t(c * kSlice);
        float v[32], v2[32];
        tc::tmem_ld32(tcol, v);
        if constexpr (kBf16Out) tc::tmem_ld32(tcol + 32, v2);  // the other 32 of 64 columns
        if (c == ns - 1) {  // accumulator read out: the MMAs of tile local + 2 may start
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
        }
        if constexpr (kBf16Out) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float* src = k < 4 ? v + 8 * k : v2 + 8 * (k - 4);
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(src[2 * i], src[2 * i + 1]);
              h[i] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(box + lane * 128 + ((uint32_t(k) ^ sw) << 4)) =
                make_uint4(h[0], h[1], h[2], h[3]);
          }
          if (g.sums) {
            // lane j: state p = (n0 + 64 c) / 2 + j, the 4 bytes at byte 4 (j & 3) of 16-byte
            // chunk j >> 2 of each of the warp's 32 rows; Horner over the rows
            __syncwarp();
            const int p = (n0 + c * kSlice) / 2 + lane, m = m0 + q * 32;
            if (p < g.P && m < g.M) {
              const float2 l = g.lam[p];
              const cf lam = {l.x, l.y};
              cf acc = {0.f, 0.f};
              const uint32_t sub = uint32_t(lane & 3) * 4u, ck = uint32_t(lane >> 2);
#pragma unroll 8
              for (int i = 0; i < 32; ++i) {
                const uint32_t wv = *reinterpret_cast<const uint32_t*>(
                    box + i * 128 + ((ck ^ uint32_t(i & 7)) << 4) + sub);
                const float2 vf =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv));
                acc = cfma(lam, acc, {vf.x, vf.y});
              }
              const int b = m / g.L, t = m - b * g.L;
              const size_t si = (((size_t)b * g.NC + (t >> 6)) * 2 + ((t >> 5) & 1)) * g.P + p;
              if (DLR_IN(si, (size_t)(g.M / g.L) * g.NC * 2 * g.P))
                g.sums[si] = make_float2(acc.re, acc.im);
            }
          }
        } else if (with_e) {
          if (!(ok = warp_wait(&ebar[j], (sc / kBoxes) & 1))) break;
          const int nc = n0 + c * kSlice;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4* p = reinterpret_cast<float4*>(box + lane * 128 + ((uint32_t(k) ^ sw) << 4));
            const float4 e = *p;
            float4 dk = make_float4(0.f, 0.f, 0.f, 0.f);
            if (nc + 4 * k < g.N) dk = __ldg(reinterpret_cast<const float4*>(g.D + nc + 4 * k));
            *p = make_float4(fmaf(dk.x, e.x, v[4 * k]), fmaf(dk.y, e.y, v[4 * k + 1]),
                             fmaf(dk.z, e.z, v[4 * k + 2]), fmaf(dk.w, e.w, v[4 * k + 3]));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(box + lane * 128 + ((uint32_t(k) ^ sw) << 4)) =
                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_store_2d(&tmC, box, n0 + c * kSlice, m0 + q * 32);
          tc::bulk_commit_group();
        }
      }
    }
    if (lane == 0) {
      // E boxes issued but never consumed (only after a failed wait) land before the CTA exits
      for (uint32_t s2 = sc; s2 < e_issued; ++s2)
        ok &= tc::mbar_wait(&ebar[s2 % kBoxes], (s2 / kBoxes) & 1);
      tc::bulk_wait_group0();
    }
  }
  if (!ok) report_status(g.status, DLR_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---- float32 GEMM from three tf32 products ----------------------------------------------
// C[M, N] = A[M, K] * B[N, K]^T (+ D[n] * E[m, n]) with float32 A, B, C. Each operand x is
// split into x_hi = x with the 13 low mantissa bits cleared (exactly a tf32 value) and
// x_lo = x - x_hi (exact in float32; the MMA uses its 11 leading significant bits), and the
// product is A_hi B_hi + A_hi B_lo + A_lo B_hi (three kind::tf32 MMAs into one f32 TMEM
// accumulator). The dropped A_lo B_lo term and the truncation of the lo parts are below
// 2^-21 of |A||B| per term; tf32 keeps float32's exponent range, so no operand scaling is
// needed. B comes split (B_hi, B_lo: two float32 arrays); A is split in the kernel.
//
// Persistent, one CTA per SM over 128 x 256 output tiles (N tile fastest). K-blocks of 32
// (128 bytes of float32 per row, the swizzle span) in a 2-stage ring of 96 KB stages:
//   warp 0 lane 0  TMA: A (float32, into the stage's A_hi slot), B_hi, B_lo;
//   warps 8-11     split A in place: thread = row r reads its 32 floats, writes x_hi over them
//                  and x_lo into the A_lo slot (same swizzled layout);
//   warp 1 lane 0  per K-block 4 K-steps x 3 MMAs of 128 x 256 x 8, a commit that frees the
//                  stage, per tile a commit that hands one of two 256-column accumulators over;
//   warp 2         TMEM allocation (512 columns);
//   warps 4-7      epilogue: slices of 32 columns, tcgen05.ld, + D (.) E (E read with plain
//                  loads one slice ahead), a 4 KB staging box per slice, TMA store.
namespace x3 {
constexpr int kBM = 128, kBN = 256, kBK = 32;
constexpr int kStages = 2;
constexpr uint32_t kAB = kBM * 128, kBB = kBN * 128;  // one operand half of a stage
constexpr uint32_t kOffALo = kAB, kOffBHi = 2 * kAB, kOffBLo = 2 * kAB + kBB;
constexpr uint32_t kStride = 2 * kAB + 2 * kBB;  // 96 KB
constexpr int kBoxes = 2;
constexpr uint32_t kEpiOff = kStages * kStride;
constexpr uint32_t kBarOff = kEpiOff + 4 * kBoxes * kBoxBytes;
constexpr size_t kSmemBytes = 1024 + kBarOff + 256;
constexpr int kThreads = 384;
static_assert(kSmemBytes <= 232448, "shared memory");
}  // namespace x3

struct X3Args {
  int M, N, K;
  const float* D;  // [N] or null
  const float* E;  // [M, N] (read when D is given)
  int* status;
};

template <bool kWithE>
__global__ void __launch_bounds__(x3::kThreads, 1)
tc_gemm_x3(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBh,
           const __grid_constant__ CUtensorMap tmBl, const __grid_constant__ CUtensorMap tmC,
           X3Args g) {
  constexpr int kBM = x3::kBM, kBN = x3::kBN, kBK = x3::kBK, kStages = x3::kStages;
  constexpr int kBoxes = x3::kBoxes;
  constexpr uint32_t kAB = x3::kAB, kBB = x3::kBB, kStride = x3::kStride;
  constexpr uint32_t kOffALo = x3::kOffALo, kOffBHi = x3::kOffBHi, kOffBLo = x3::kOffBLo;
  constexpr uint32_t kEpiOff = x3::kEpiOff, kBarOff = x3::kBarOff;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kBarOff);
  uint64_t* full = bars;                    // [kStages] A (float32), B_hi, B_lo landed
  uint64_t* empty = bars + kStages;         // [kStages] the MMAs have read the stage
  uint64_t* a_ready = bars + 2 * kStages;   // [kStages] A split (4 arrivals)
  uint64_t* acc_full = bars + 3 * kStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2] (4 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (g.N + kBN - 1) / kBN;
  const int tiles = n_tiles * ((g.M + kBM - 1) / kBM);
  const int nk = g.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
      tc::mbar_init(&a_ready[s], 4);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);
    }
    tc::mbar_fence_init();
  }
  if (warp == 2) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    uint32_t it = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const int m0 = (t / n_tiles) * kBM, n0 = (t % n_tiles) * kBN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = it % kStages;
        if (it >= kStages && !(ok = tc::mbar_wait(&empty[s], ((it / kStages) - 1) & 1))) break;
        uint8_t* st = base + s * kStride;
        tc::mbar_arrive_expect_tx(&full[s], kAB + 2 * kBB);
        tc::tma_load_2d(st, &tmA, kb * kBK, m0, &full[s]);
        tc::tma_load_2d(st + kOffBHi, &tmBh, kb * kBK, n0, &full[s]);
        tc::tma_load_2d(st + kOffBLo, &tmBl, kb * kBK, n0, &full[s]);
      }
    }
    // every copy issued has landed before the CTA may exit
    for (uint32_t j = it > kStages ? it - kStages : 0; j < it; ++j)
      ok &= tc::mbar_wait(&full[j % kStages], (j / kStages) & 1);
  } else if (warp >= 8) {
    // thread = row r of the tile: its 32 floats (8 chunks of 16 bytes at (c ^ (r & 7)) << 4)
    const int r = (warp - 8) * 32 + lane;
    const uint32_t sw = uint32_t(r & 7);
    uint32_t it = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < nk && ok; ++kb, ++it) {
        const int s = it % kStages;
        if (!(ok = warp_wait(&full[s], (it / kStages) & 1))) break;
        uint8_t* row = base + s * kStride + (DLR_IN(r, kBM) ? r : 0) * 128;
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          v[c] = *reinterpret_cast<const uint4*>(row + ((uint32_t(c) ^ sw) << 4));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 hi = make_uint4(v[c].x & 0xFFFFE000u, v[c].y & 0xFFFFE000u,
                                      v[c].z & 0xFFFFE000u, v[c].w & 0xFFFFE000u);
          const uint4 lo = make_uint4(
              __float_as_uint(__uint_as_float(v[c].x) - __uint_as_float(hi.x)),
              __float_as_uint(__uint_as_float(v[c].y) - __uint_as_float(hi.y)),
              __float_as_uint(__uint_as_float(v[c].z) - __uint_as_float(hi.z)),
              __float_as_uint(__uint_as_float(v[c].w) - __uint_as_float(hi.w)));
          const uint32_t o = (uint32_t(c) ^ sw) << 4;
          *reinterpret_cast<uint4*>(row + o) = hi;
          *reinterpret_cast<uint4*>(row + kOffALo + o) = lo;
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&a_ready[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::idesc_tf32_f32(kBM, kBN);
    uint32_t it = 0, local = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
      const uint32_t acc = local & 1;
      if (local >= 2 && !(ok = tc::mbar_wait(&acc_empty[acc], ((local >> 1) - 1) & 1))) break;
      tc::fence_after_sync();
      const uint32_t d = tmem + acc * kBN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = it % kStages;
        if (!(ok = tc::mbar_wait(&full[s], (it / kStages) & 1))) break;
        if (!(ok = tc::mbar_wait(&a_ready[s], (it / kStages) & 1))) break;
        tc::fence_after_sync();
        const uint8_t* st = base + s * kStride;
        const uint64_t ah = tc::smem_desc_k_sw128(st), al = tc::smem_desc_k_sw128(st + kOffALo);
        const uint64_t bh = tc::smem_desc_k_sw128(st + kOffBHi);
        const uint64_t bl = tc::smem_desc_k_sw128(st + kOffBLo);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 8 tf32 = 32 bytes = 2 descriptor units per K-step
          tc::mma_kind_tf32(d, ah + 2 * kk, bh + 2 * kk, idesc, (kb | kk) != 0);
          tc::mma_kind_tf32(d, ah + 2 * kk, bl + 2 * kk, idesc, 1);
          tc::mma_kind_tf32(d, al + 2 * kk, bh + 2 * kk, idesc, 1);
        }
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(&acc_full[acc]);
    }
  } else if (warp >= 4 && warp < 8) {
    const int q = warp - 4;
    uint8_t* boxes = base + kEpiOff + q * kBoxes * kBoxBytes;
    const uint32_t sw = uint32_t(lane & 7);
    uint32_t sc = 0, local = 0;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
      const uint32_t acc = local & 1;
      const int m0 = (t / n_tiles) * kBM, n0 = (t % n_tiles) * kBN;
      const int ns = min(kBN, g.N - n0) / 32;  // N is a multiple of 32
      const int m = m0 + q * 32 + lane;         // this thread's row
      // E of the first slice, loaded before the accumulator is ready
      float4 e[8], en[8];
      auto load_e = [&](int c, float4 (&dst)[8]) {
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kWithE && m < g.M && c < ns &&
            DLR_IN((size_t)m * g.N + n0 + 32 * c + 31, (size_t)g.M * g.N)) {
          const float4* src =
              reinterpret_cast<const float4*>(g.E + (size_t)m * g.N + n0 + 32 * c);
#pragma unroll
          for (int k = 0; k < 8; ++k) dst[k] = __ldg(src + k);
        }
      };
      load_e(0, e);
      if (!(ok = warp_wait(&acc_full[acc], (local >> 1) & 1))) break;
      tc::fence_after_sync();
      for (int c = 0; c < ns; ++c, ++sc) {
        uint8_t* box = boxes + (sc % kBoxes) * kBoxBytes;
        if (lane == 0) tc::bulk_wait_group_read<kBoxes - 1>();  // the box's last store read it
        __syncwarp();
        float v[32];
        tc::tmem_ld32(tmem + acc * kBN + (uint32_t(q * 32) << 16) + uint32_t(c * 32), v);
        if (c == ns - 1) {  // accumulator read out: the MMAs of tile local + 2 may start
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
        }
        load_e(c + 1, en);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
          if (kWithE) {
            const float4 dk =
                DLR_IN(n0 + 32 * c + 4 * k + 3, g.N)
                    ? __ldg(reinterpret_cast<const float4*>(g.D + n0 + 32 * c + 4 * k))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
            o.x = fmaf(dk.x, e[k].x, o.x);
            o.y = fmaf(dk.y, e[k].y, o.y);
            o.z = fmaf(dk.z, e[k].z, o.z);
            o.w = fmaf(dk.w, e[k].w, o.w);
          }
          *reinterpret_cast<float4*>(box + lane * 128 + ((uint32_t(k) ^ sw) << 4)) = o;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = en[k];
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_store_2d(&tmC, box, n0 + c * 32, m0 + q * 32);
          tc::bulk_commit_group();
        }
      }
    }
    if (lane == 0) tc::bulk_wait_group0();
  }
  if (!ok) report_status(g.status, DLR_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, kTmemCols);
}

#ifdef DLR_BOUNDS_CHECK
// Bounds-check self-test: thread t of one warp reads element t + 1 of a 32-element shared
// buffer through the check, so thread 31's read (one past the end) is skipped and reported.
__global__ void selftest_bounds_kernel(float* sink) {
  __shared__ float buf[32];
  const int t = threadIdx.x;
  buf[t] = (float)t;
  __syncwarp();
  float v = 0.f;
  if (DLR_IN(t + 1, 32)) v = buf[t + 1];
  if (v < 0.f) *sink = v;  // never true; keeps the read
}
#endif

// Failure-reporting self-test: one thread waits on a barrier that nothing completes.
__global__ void selftest_wait_timeout(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
    if (!tc::mbar_wait(&bar, 0, limit_ns)) report_status(status, DLR_ERR_TIMEOUT);
  }
}

// Row-major [rows, cols] tensor of 2-byte (bf16) or 4-byte (f32) elements, boxes of
// box_rows x box_cols elements with a 128-byte swizzle (box_cols * element size = 128).
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
              bool f32) {
  auto fn = tc::tensor_map_encoder();
  if (!fn) return false;
  const uint64_t esz = f32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols * esz) % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {uint32_t(128 / esz), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kOp, bool kWithE, bool kBf16Out>
cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                     const CUtensorMap& me, const GemmArgs& g, int grid, cudaStream_t s) {
  using PL = Plan<kWithE, kOp>;
  constexpr size_t smem = PL::kSmemBytes;
  cudaError_t e = max_smem_once<tc_gemm<kOp, kWithE, kBf16Out>>(smem);
  if (e != cudaSuccess) return e;
  tc_gemm<kOp, kWithE, kBf16Out><<<grid, PL::kThreads, smem, s>>>(ma, mb, mc, me, g);
  return cudaGetLastError();
}

int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
  });
  return n;
}

}  // namespace

cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s) {
  selftest_wait_timeout<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

#ifdef DLR_BOUNDS_CHECK
cudaError_t launch_selftest_bounds(cudaStream_t s) {
  selftest_bounds_kernel<<<1, 32, 0, s>>>(nullptr);
  return cudaGetLastError();
}
#endif

// A: [M, K] row-major, bf16 (a_f32 false) or float32 (a_f32, converted to bf16 in the
// kernel); B: bf16 [N, K] row-major. C: [M, N], f32 or (c_bf16, no D) bf16; D: f32 [N] or
// null; E: f32 [M, N] (read only when D is given; not with a float32 A). With `sums` (bf16 C,
// N = 2P, rows = B sequences of length L, L a multiple of 64): the per-32-row partial chunk
// states of C, sums[b][c][half][p] = sum_i lam[p]^(31-i) C[b L + 64 c + 32 half + i][2p, 2p+1].
cudaError_t launch_tc_gemm(const void* A, bool a_f32, const void* B, void* C, bool c_bf16,
                           int M, int N, int K, const float* D, const float* E, int* status,
                           cudaStream_t s, const float2* lam, float2* sums, int L, int NC) {
  if (M < 1 || N < 1 || K < 1 || (c_bf16 && D) || (a_f32 && D)) return cudaErrorInvalidValue;
  if (sums && (!c_bf16 || N % 2 || L % 64 || !lam)) return cudaErrorInvalidValue;
  CUtensorMap ma, mb, mc, me;
  if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, kBM, a_f32)) return cudaErrorInvalidValue;
  if (!make_map(&mb, B, (uint64_t)N, (uint64_t)K, kBN, false)) return cudaErrorInvalidValue;
  if (!make_map(&mc, C, (uint64_t)M, (uint64_t)N, 32, !c_bf16)) return cudaErrorInvalidValue;
  if (D && !make_map(&me, E, (uint64_t)M, (uint64_t)N, 32, true)) return cudaErrorInvalidValue;
  if (!D) me = mc;  // not read
  GemmArgs g{M, N, K, D, status, lam, nullptr, L, N / 2, NC, sums};
  const long long tiles = (long long)((N + kBN - 1) / kBN) * ((M + kBM - 1) / kBM);
  const int grid = (int)std::min<long long>(tiles, sm_count());
  if (D) return run_gemm<kOpBf16, true, false>(ma, mb, mc, me, g, grid, s);
  if (c_bf16)
    return a_f32 ? run_gemm<kOpCvtA, false, true>(ma, mb, mc, me, g, grid, s)
                 : run_gemm<kOpBf16, false, true>(ma, mb, mc, me, g, grid, s);
  return a_f32 ? run_gemm<kOpCvtA, false, false>(ma, mb, mc, me, g, grid, s)
               : run_gemm<kOpBf16, false, false>(ma, mb, mc, me, g, grid, s);
}

// The S5 output projection with the chunked scan's last step fused in: V bf16 [M = B L, K = 2P]
// (Re, Im per state), L a multiple of 64; x_t = lambda x_{t-1} + V_t inside each chunk of 64
// steps, starting from xin[b][c][p] (the state entering the chunk); y = x C^T + D (.) E with C
// bf16 [N, K] and E, y float32 [M, N].
cudaError_t launch_tc_gemm_apply(const void* V, const void* C, float* y, int M, int N, int K,
                                 const float* D, const float* E, const float2* lam,
                                 const float2* xin, int L, int P, int NC, int* status,
                                 cudaStream_t s) {
  if (M < 1 || N < 1 || K != 2 * P || L % 64 || !D || !E) return cudaErrorInvalidValue;
  CUtensorMap ma, mb, mc, me;
  if (!make_map(&ma, V, (uint64_t)M, (uint64_t)K, kBM, false)) return cudaErrorInvalidValue;
  if (!make_map(&mb, C, (uint64_t)N, (uint64_t)K, kBN, false)) return cudaErrorInvalidValue;
  if (!make_map(&mc, y, (uint64_t)M, (uint64_t)N, 32, true)) return cudaErrorInvalidValue;
  if (!make_map(&me, E, (uint64_t)M, (uint64_t)N, 32, true)) return cudaErrorInvalidValue;
  GemmArgs g{M, N, K, D, status, lam, xin, L, P, NC, nullptr};
  const long long tiles = (long long)((N + kBN - 1) / kBN) * ((M + kBM - 1) / kBM);
  const int grid = (int)std::min<long long>(tiles, sm_count());
  return run_gemm<kOpApply, true, false>(ma, mb, mc, me, g, grid, s);
}


// C[M, N] = A[M, K] B[N, K]^T (+ D (.) E) in float32 from three tf32 products (tc_gemm_x3). A,
// Bh, Bl, C, E: row-major float32, 16-byte aligned; Bh = B with the 13 low mantissa bits
// cleared, Bl = B - Bh; K and N multiples of 32; D [N] or null.
cudaError_t launch_tc_gemm_x3(const float* A, const float* Bh, const float* Bl, float* C, int M,
                              int N, int K, const float* D, const float* E, int* status,
                              cudaStream_t s) {
  if (M < 1 || N < 1 || K < 1 || K % 32 || N % 32 || (D && !E)) return cudaErrorInvalidValue;
  if (D && ((reinterpret_cast<uintptr_t>(D) | reinterpret_cast<uintptr_t>(E)) & 15))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mbh, mbl, mc;
  if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, x3::kBM, true) ||
      !make_map(&mbh, Bh, (uint64_t)N, (uint64_t)K, x3::kBN, true) ||
      !make_map(&mbl, Bl, (uint64_t)N, (uint64_t)K, x3::kBN, true) ||
      !make_map(&mc, C, (uint64_t)M, (uint64_t)N, 32, true))
    return cudaErrorInvalidValue;
  X3Args g{M, N, K, D, E, status};
  const long long tiles = (long long)((N + x3::kBN - 1) / x3::kBN) * ((M + x3::kBM - 1) / x3::kBM);
  const int grid = (int)std::min<long long>(tiles, sm_count());
  cudaError_t e;
  if (D) {
    if ((e = max_smem_once<tc_gemm_x3<true>>(x3::kSmemBytes)) != cudaSuccess) return e;
    tc_gemm_x3<true><<<grid, x3::kThreads, x3::kSmemBytes, s>>>(ma, mbh, mbl, mc, g);
  } else {
    if ((e = max_smem_once<tc_gemm_x3<false>>(x3::kSmemBytes)) != cudaSuccess) return e;
    tc_gemm_x3<false><<<grid, x3::kThreads, x3::kSmemBytes, s>>>(ma, mbh, mbl, mc, g);
  }
  return cudaGetLastError();
}

}  // namespace dlr
