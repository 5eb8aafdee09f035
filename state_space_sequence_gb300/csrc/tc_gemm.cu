// tc_gemm.cu -- C[M, N] (f32) = A[M, K] * B[N, K]^T (+ D[n] * E[m, n]) on 5th-generation tensor
// cores: bf16 operands in shared memory (TMA tile loads, 128-byte swizzle), f32 accumulator in
// tensor memory, tcgen05.mma issued by one thread, tcgen05.ld epilogue.
//
// One CTA computes one 128 x 256 tile with 4 warps:
//   warp 0 lane 0  TMA producer: K-blocks of 64 into a 2-stage ring (A 16 KB + B 32 KB),
//   warp 1 lane 0  MMA issuer: four K=16 MMAs per K-block, then a commit that frees the stage;
//                  a final commit marks the accumulator complete,
//   warp 2         allocates / frees 256 TMEM columns,
//   warps 0-3      epilogue: warp w reads TMEM lanes 32w..32w+31 (rows of the tile).
// Two CTAs fit on an SM (96 KB shared memory, 256 TMEM columns each), so one CTA's epilogue
// overlaps the other's main loop.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "dlr_common.cuh"
#include "tc_ptx.cuh"

namespace dlr {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 2;
constexpr uint32_t kABytes = kBM * kBK * 2, kBBytes = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 256;
constexpr uint32_t kTmemCols = 256;

struct GemmArgs {
  int M, N, K;
  float* C;
  const float* D;  // [N] or null
  const float* E;  // [M, N] or null
  int* status;
};

__global__ void __launch_bounds__(128, 1)
tc_gemm_bf16(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* full = bars;                 // [kStages]
  uint64_t* empty = bars + kStages;      // [kStages]
  uint64_t* acc_full = bars + 2 * kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  const int nk = (g.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(acc_full, 1);
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
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % kStages;
      const uint32_t round = kb / kStages;
      if (kb >= kStages) ok = tc::mbar_wait(&empty[s], (round - 1) & 1);
      if (!ok) break;
      uint8_t* a = base + s * kStageBytes;
      uint8_t* b = a + kABytes;
      tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
      tc::tma_load_2d(a, &tmA, kb * kBK, m0, &full[s]);
      tc::tma_load_2d(b, &tmB, kb * kBK, n0, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % kStages;
      ok = tc::mbar_wait(&full[s], (kb / kStages) & 1);
      if (!ok) break;
      tc::fence_after_sync();
      const uint8_t* a = base + s * kStageBytes;
      const uint64_t ad = tc::smem_desc_k_sw128(a);
      const uint64_t bd = tc::smem_desc_k_sw128(a + kABytes);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)  // advance 16 bf16 = 32 bytes = 2 descriptor units
        tc::mma_kind_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(acc_full);
  }
  __syncwarp();

  // ---- epilogue: all four warps. Each 32-column slice of the accumulator goes TMEM ->
  // registers (thread = row) -> shared memory (the drained stages) -> row-coalesced float4
  // stores, with D (.) E added on the way out. ----
  const bool acc_ok = tc::mbar_wait(acc_full, 0);
  tc::fence_after_sync();
  float* tile = reinterpret_cast<float*>(base);  // [128][33]
  const bool vec = (g.N & 3) == 0;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    const int nc = n0 + c * 32;
    if (nc >= g.N) break;  // block-uniform
    float v[32];
    tc::tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c * 32), v);
    const int r_own = warp * 32 + lane;
#pragma unroll
    for (int j = 0; j < 32; ++j) tile[r_own * 33 + j] = v[j];
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int idx = it * 128 + threadIdx.x;  // 128 rows x 8 float4 per slice
      const int r = idx >> 3, c4 = (idx & 7) * 4;
      const int row = m0 + r, col = nc + c4;
      if (row < g.M && acc_ok) {
        float o[4] = {tile[r * 33 + c4], tile[r * 33 + c4 + 1], tile[r * 33 + c4 + 2],
                      tile[r * 33 + c4 + 3]};
        if (vec && col + 3 < g.N) {
          if (g.E) {
            const float4 e = __ldg(reinterpret_cast<const float4*>(g.E + (size_t)row * g.N + col));
            const float4 d = __ldg(reinterpret_cast<const float4*>(g.D + col));
            o[0] = fmaf(d.x, e.x, o[0]);
            o[1] = fmaf(d.y, e.y, o[1]);
            o[2] = fmaf(d.z, e.z, o[2]);
            o[3] = fmaf(d.w, e.w, o[3]);
          }
          *reinterpret_cast<float4*>(g.C + (size_t)row * g.N + col) =
              make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (col + q < g.N) {
              float val = o[q];
              if (g.E) val = fmaf(g.D[col + q], g.E[(size_t)row * g.N + col + q], val);
              g.C[(size_t)row * g.N + col + q] = val;
            }
        }
      }
    }
    __syncthreads();
  }
  if (!ok || !acc_ok) report_status(g.status, DLR_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, kTmemCols);
}

// Failure-reporting self-test: one thread waits on a barrier that nothing completes.
__global__ void selftest_wait_timeout(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
    if (!tc::mbar_wait(&bar, 0, limit_ns)) report_status(status, DLR_ERR_TIMEOUT);
  }
}

// fp32 -> bf16, same layout (n a multiple of 4, 16-byte aligned pointers)
__global__ void to_bf16(const float4* __restrict__ x, __nv_bfloat162* __restrict__ y, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = __ldg(&x[i]);
    y[2 * i] = __floats2bfloat162_rn(v.x, v.y);
    y[2 * i + 1] = __floats2bfloat162_rn(v.z, v.w);
  }
}

// fp32 [R, C] -> bf16 [C, R] (transposed), small matrices
__global__ void to_bf16_t(const float* __restrict__ x, __nv_bfloat16* __restrict__ y, int R,
                          int C) {
  __shared__ float tile[32][33];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    tile[i][threadIdx.x] = (r < R && c < C) ? x[(size_t)r * C + c] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < C && r < R) y[(size_t)c * R + r] = __float2bfloat16_rn(tile[threadIdx.x][i]);
  }
}

// Row-major bf16 [rows, cols] with boxes of box_rows x 64 columns, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = tc::tensor_map_encoder();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols * 2) % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_to_bf16(const float* x, void* y, size_t n, cudaStream_t s) {
  const size_t n4 = n / 4;
  const int blocks = (int)std::min<size_t>((n4 + 255) / 256, 152 * 16);
  to_bf16<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(x),
                                 reinterpret_cast<__nv_bfloat162*>(y), n4);
  return cudaGetLastError();
}

cudaError_t launch_to_bf16_t(const float* x, void* y, int R, int C, cudaStream_t s) {
  dim3 grid((C + 31) / 32, (R + 31) / 32);
  to_bf16_t<<<grid, dim3(32, 8), 0, s>>>(x, reinterpret_cast<__nv_bfloat16*>(y), R, C);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s) {
  selftest_wait_timeout<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

// A: bf16 [M, K] row-major; B: bf16 [N, K] row-major; C: f32 [M, N].
cudaError_t launch_tc_gemm(const void* A, const void* B, float* C, int M, int N, int K,
                           const float* D, const float* E, int* status, cudaStream_t s) {
  CUtensorMap ma, mb;
  if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, kBM)) return cudaErrorInvalidValue;
  if (!make_map(&mb, B, (uint64_t)N, (uint64_t)K, kBN)) return cudaErrorInvalidValue;
  cudaError_t e = max_smem_once<tc_gemm_bf16>(kSmemBytes);
  if (e != cudaSuccess) return e;
  GemmArgs g{M, N, K, C, D, E, status};
  dim3 grid((M + kBM - 1) / kBM, (N + kBN - 1) / kBN);
  tc_gemm_bf16<<<grid, 128, kSmemBytes, s>>>(ma, mb, g);
  return cudaGetLastError();
}

}  // namespace dlr
