// s5_layer.cu -- S5 SSM outputs ("Simplified State Space Layers for Sequence Modeling",
// section 2.2 (linear recurrence as a scan), section 3 (diagonalised MIMO system with B~, C~,
// diagonal D, one timescale per state, zero-order hold)):
//   Lbar = exp(Lambda Delta), Bbar = (Lbar - 1)/Lambda * B~,
//   x_k = Lbar x_{k-1} + Bbar u_k,   y_k = Re(C~ x_k) + D u_k.
//
// Float32 tier, as a sequence of kernels over a workspace:
//   prep   (one CTA per state p, double precision): Lbar_p, the powers Lbar_p^t (t <= T) and
//          Lbar_p^T as two floats, Bbar as the real [2P, H] operand and C~ as the real [H, 2P]
//          operand [Re C~, -Im C~], each split into its tf32 part and the float32 remainder.
//   gemm   V[B*L, 2P] = u[B*L, H] * Bbar^T in float32 from three tf32 tensor-core products
//          (tc_gemm_x3 in tc_gemm.cu)
//   chunk  S_c = sum_t Lbar^{T-1-t} V_t (end state of chunk c from a zero start)
//   carry  X_c = Lbar^T X_{c-1} + S_c in two-float arithmetic, one warp per (b, p) scanning
//          groups of chunks (the tensor-core tier: float32, one CTA per (b, 32 states) with a
//          warp per group of chunks); stores the state entering each chunk
//   apply  x_t = Lbar^{t+1} X_in + l_t, l_t = Lbar l_{t-1} + V_t, written over V in place
//   gemm   y = x * [Re C~, -Im C~]^T + D (.) u (tc_gemm_x3)
// The tensor-core tier runs the two projections on tcgen05 (tc_gemm.cu) with bf16 operands and
// float32 accumulation: the input projection converts the float32 u to bf16 in the kernel and
// writes V as bf16; the scan reads V in bf16 and computes in float32; apply writes x as bf16
// over V, the operand of the output projection. When L is a multiple of 64 (the usual case)
// the chunk and apply steps move into the projections: the input projection's epilogue writes
// the chunk end states in two 32-step halves, and the output projection turns its V operand
// tiles into x itself, so the tier is prep, input projection, carry, output projection.
#include <cuda_bf16.h>

#include "dlr_common.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 13;
namespace {

constexpr int kT = 64;   // steps per chunk

struct S5Work {
  void* bbar_t16;  // bf16 [2P][H]   (tensor-core tier only)
  void* cmat_t16;  // bf16 [H][2P]
  void* vx16;      // bf16 [B*L][2P]: V, then x (tensor-core tier)
  float* b1;       // [2][2P][H]: B_bar as the input projection's [N, K] operand, tf32 hi, lo
  float* b2;       // [2][H][2P]: [Re C~, -Im C~] as the output projection's operand, hi, lo
  float2* lbar_pw; // [T+1][P]  Lbar^t (state fastest, so a warp's loads of one power coalesce)
  float4* lbar_T;  // [P] (re.hi, re.lo, im.hi, im.lo) of Lbar^T
  float2* S;       // [B][NC][P]
  float2* S2;      // [B][NC][2][P]: the two 32-step halves of each chunk's end state (tensor-core
                   // tier, L a multiple of 64: written by the input projection)
  float2* Xin;     // [B][NC][P]
  float* xv;       // [B*L][2P]: V, then x (float32 tier)
};

// x as its tf32 part (the 13 low mantissa bits cleared) and the float32 remainder
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  lo = x - hi;
}

// The float32 tier's projection operands for state p and feature h, split into tf32 hi and lo
// halves: B_bar (br + i bi) at rows 2p, 2p + 1 of the input projection's [2P, H] operand, and
// Re C~, -Im C~ at columns 2p, 2p + 1 of row h of the output projection's [H, 2P] operand.
__device__ __forceinline__ void store_operands(const S5Work& w, int H, int P, int p, int h,
                                               float br, float bi, float2 c) {
  const size_t n1 = (size_t)2 * P * H;
  float hi, lo;
  split_tf32(br, hi, lo);
  w.b1[(size_t)(2 * p) * H + h] = hi;
  w.b1[n1 + (size_t)(2 * p) * H + h] = lo;
  split_tf32(bi, hi, lo);
  w.b1[(size_t)(2 * p + 1) * H + h] = hi;
  w.b1[n1 + (size_t)(2 * p + 1) * H + h] = lo;
  split_tf32(c.x, hi, lo);
  w.b2[(size_t)h * 2 * P + 2 * p] = hi;
  w.b2[n1 + (size_t)h * 2 * P + 2 * p] = lo;
  split_tf32(-c.y, hi, lo);
  w.b2[(size_t)h * 2 * P + 2 * p + 1] = hi;
  w.b2[n1 + (size_t)h * 2 * P + 2 * p + 1] = lo;
}

__global__ void s5_prep(const float* __restrict__ lambda, const float* __restrict__ log_delta,
                        const float2* __restrict__ Bt, const float2* __restrict__ Ct, int H, int P,
                        int bilinear, S5Work w) {
  // One thread evaluates the state's transcendental functions in double (the FP64 units are
  // few): Lbar, (Lbar - 1) / Lambda, and the powers Lbar^k, Lbar^(8k) for k = 0..8 by
  // sequential products; every power t <= T is then one product Lbar^(8(t>>3)) Lbar^(t&7).
  __shared__ double sp1[9][2], sp8[9][2];
  __shared__ float2 sq;
  const int p = blockIdx.x;
  if (threadIdx.x == 0) {
    const double lr = lambda[2 * p], li = lambda[2 * p + 1];
    const double delta = exp((double)log_delta[p]);
    const double zr = lr * delta, zi = li * delta;
    double ar, ai;
    if (!bilinear) {
      // zero-order hold: Lbar = exp(z), B_bar = (Lbar - 1) / Lambda B~
      const double er = exp(zr);
      ar = er * cos(zi);
      ai = er * sin(zi);
      const double nr = ar - 1.0, ni = ai;
      const double den = lr * lr + li * li;
      sq = make_float2((float)((nr * lr + ni * li) / den), (float)((ni * lr - nr * li) / den));
    } else {
      // bilinear transform ("The Annotated S4", part 1): Lbar = (1 + z/2) / (1 - z/2),
      // B_bar = Delta / (1 - z/2) B~
      const double dr = 1.0 - 0.5 * zr, di = -0.5 * zi;   // 1 - z/2
      const double pr = 1.0 + 0.5 * zr, pi = 0.5 * zi;    // 1 + z/2
      const double den = dr * dr + di * di;
      ar = (pr * dr + pi * di) / den;
      ai = (pi * dr - pr * di) / den;
      sq = make_float2((float)(delta * dr / den), (float)(-delta * di / den));
    }
    double re = 1.0, im = 0.0;
    for (int k = 0; k <= 8; ++k) {
      sp1[k][0] = re;
      sp1[k][1] = im;
      const double r2 = re * ar - im * ai;
      im = re * ai + im * ar;
      re = r2;
    }
    const double br = sp1[8][0], bi = sp1[8][1];
    re = 1.0, im = 0.0;
    for (int k = 0; k <= 8; ++k) {
      sp8[k][0] = re;
      sp8[k][1] = im;
      const double r2 = re * br - im * bi;
      im = re * bi + im * br;
      re = r2;
    }
  }
  __syncthreads();
  const float qr = sq.x, qi = sq.y;
  const bool tc = w.bbar_t16 != nullptr;  // tensor-core tier: bf16 operands
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float2 b = Bt[(size_t)p * H + h];
    const float br = fmaf(qr, b.x, -qi * b.y), bi = fmaf(qr, b.y, qi * b.x);
    const float2 c = Ct[(size_t)h * P + p];
    if (tc) {
      __nv_bfloat16* bt = reinterpret_cast<__nv_bfloat16*>(w.bbar_t16);
      bt[(size_t)(2 * p) * H + h] = __float2bfloat16_rn(br);
      bt[(size_t)(2 * p + 1) * H + h] = __float2bfloat16_rn(bi);
      reinterpret_cast<__nv_bfloat162*>(w.cmat_t16)[(size_t)h * P + p] =
          __floats2bfloat162_rn(c.x, -c.y);
    } else {
      store_operands(w, H, P, p, h, br, bi, c);
    }
  }
  for (int t = threadIdx.x; t <= kT; t += blockDim.x) {
    const double* a8 = sp8[t >> 3];
    const double* a1 = sp1[t & 7];
    const double re = a8[0] * a1[0] - a8[1] * a1[1], im = a8[0] * a1[1] + a8[1] * a1[0];
    w.lbar_pw[(size_t)t * P + p] = make_float2((float)re, (float)im);
    if (t == kT) {
      float rh = (float)re, ih = (float)im;
      w.lbar_T[p] = make_float4(rh, (float)(re - rh), ih, (float)(im - ih));
    }
  }
}

// grid (NC, B), one thread per state p: the chunk end state from a zero start,
// S_c = sum_t Lbar^{T-1-t} V_t with the directly computed powers. The V loads of a thread are
// issued kBatch at a time ahead of their use, so each thread keeps several in flight.
constexpr int kBatch = 16;

__global__ void __launch_bounds__(256)
s5_chunk_state(S5Work w, int L, int P, int NC) {
  const int c = blockIdx.x, b = blockIdx.y;
  const int t0 = c * kT;
  const int valid = min(kT, L - t0);
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const size_t col = ((size_t)b * L + t0) * P + p;  // in complex elements
    cf acc = {0.f, 0.f};
    for (int tb = 0; tb < valid; tb += kBatch) {
      float2 v[kBatch], a[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const bool in = tb + j < valid &&
                        DLR_IN(col + (size_t)(tb + j) * P, (size_t)gridDim.y * L * P) &&
                        DLR_IN((size_t)(kT - 1 - tb - j) * P + p, (size_t)(kT + 1) * P);
        v[j] = in ? reinterpret_cast<const float2*>(w.xv)[col + (size_t)(tb + j) * P]
                  : make_float2(0.f, 0.f);
        a[j] = in ? w.lbar_pw[(size_t)(kT - 1 - tb - j) * P + p] : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) acc = cfma({a[j].x, a[j].y}, {v[j].x, v[j].y}, acc);
    }
    if (DLR_IN(((size_t)b * NC + c) * P + p, (size_t)gridDim.y * NC * P))
      w.S[((size_t)b * NC + c) * P + p] = make_float2(acc.re, acc.im);
  }
}

__device__ __forceinline__ cff cff_mul(cff a, cff b) {
  return cff_fma(a, b, {{0.f, 0.f}, {0.f, 0.f}});
}
__device__ __forceinline__ cff cff_shfl_up(cff a, int d) {
  return {{__shfl_up_sync(0xffffffffu, a.re.hi, d), __shfl_up_sync(0xffffffffu, a.re.lo, d)},
          {__shfl_up_sync(0xffffffffu, a.im.hi, d), __shfl_up_sync(0xffffffffu, a.im.lo, d)}};
}

// One warp per (b, p): the state entering each chunk, X_0 = 0, X_{c+1} = m X_c + S_c with
// m = Lbar^T, in two-float arithmetic (float32 tier). Lane i takes G = ceil(NC / 32)
// consecutive chunks:
//   1. its group's end state from a zero start,
//   2. an inclusive Kogge-Stone scan over the lanes of the maps x -> m^G x + A_i (the step of
//      offset d multiplies by m^{G d}), so lane i - 1 holds the state entering group i,
//   3. the group's chain again from that state, storing the state entering each chunk.
// Only the last non-empty group may be short; no lane before it reads its value.
__global__ void __launch_bounds__(256)
s5_carry(S5Work w, int B, int P, int NC) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (gw >= B * P) return;  // whole warps
  const int b = gw / P, p = gw % P;
  const float4 lt = w.lbar_T[p];
  const cff m = {{lt.x, lt.y}, {lt.z, lt.w}};
  const cff zero = {{0.f, 0.f}, {0.f, 0.f}};
  const int G = (NC + 31) / 32;
  const int c0 = min(NC, lane * G), c1 = min(NC, c0 + G);
  const size_t base = (size_t)b * NC * P + p;
  auto chain = [&](cff x, bool store) {
    for (int cb = c0; cb < c1; cb += 8) {
      float2 sv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        sv[q] = (cb + q < c1) ? w.S[base + (size_t)(cb + q) * P] : make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cb + q >= c1) break;
        if (store)
          w.Xin[base + (size_t)(cb + q) * P] =
              make_float2(x.re.hi + x.re.lo, x.im.hi + x.im.lo);
        x = cff_fma(m, x, {{sv[q].x, 0.f}, {sv[q].y, 0.f}});
      }
    }
    return x;
  };
  cff a = chain(zero, false);
  // m^G by binary powering, then the scan
  cff md = {{1.f, 0.f}, {0.f, 0.f}}, sq = m;
  for (int e = G; e; e >>= 1) {
    if (e & 1) md = cff_mul(md, sq);
    if (e > 1) sq = cff_mul(sq, sq);
  }
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const cff prev = cff_shfl_up(a, d);
    if (lane >= d) a = cff_fma(md, prev, a);
    md = cff_mul(md, md);
  }
  const cff prev = cff_shfl_up(a, 1);
  chain(lane ? prev : zero, true);
}

// Tensor-core tier carry, float32: grid (P / 32, B), 1024 threads. Lane j holds state
// p = 32 blockIdx.x + j (coalesced loads and stores), warp g the chunk group
// [g G, (g + 1) G), G = ceil(NC / 32):
//   1. the group's end state from a zero start,
//   2. through shared memory, each warp's carry-in: the earlier groups' end states chained with
//      m^G (all groups before the last are full),
//   3. the group's chain again from its carry-in, storing the state entering each chunk.
// With kHalves the chunk end state is Lbar^32 h0 + h1 from its two 32-step halves.
template <bool kHalves>
__global__ void __launch_bounds__(1024)
s5_carry_groups(S5Work w, int B, int P, int NC) {
  __shared__ cf agg[32][32];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int b = blockIdx.y, p = blockIdx.x * 32 + lane;
  const float4 lt = w.lbar_T[p];
  const cf m = {lt.x, lt.z};
  const float2 l32 = w.lbar_pw[(size_t)32 * P + p];
  const int G = (NC + 31) / 32;
  const int c0 = min(NC, grp * G), c1 = min(NC, c0 + G);
  const size_t base = (size_t)b * NC * P + p;
  auto chunk_s = [&](int c) -> cf {
    if constexpr (kHalves) {
      const size_t i = ((size_t)b * NC + c) * 2 * P + p;
      const float2 h0 = w.S2[i], h1 = w.S2[i + P];
      return cfma({l32.x, l32.y}, {h0.x, h0.y}, {h1.x, h1.y});
    } else {
      const float2 v = w.S[base + (size_t)c * P];
      return {v.x, v.y};
    }
  };
  auto chain = [&](cf x, bool store) {
    for (int cb = c0; cb < c1; cb += 8) {
      cf sv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) sv[q] = (cb + q < c1) ? chunk_s(cb + q) : cf{0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cb + q >= c1) break;
        if (store && DLR_IN(base + (size_t)(cb + q) * P, (size_t)B * NC * P))
          w.Xin[base + (size_t)(cb + q) * P] = make_float2(x.re, x.im);
        x = cfma(m, x, sv[q]);
      }
    }
    return x;
  };
  agg[grp][lane] = chain({0.f, 0.f}, false);
  cf mg = {1.f, 0.f}, sq = m;  // m^G
  for (int e = G; e; e >>= 1) {
    if (e & 1) mg = cmul(mg, sq);
    if (e > 1) sq = cmul(sq, sq);
  }
  __syncthreads();
  cf x = {0.f, 0.f};
  for (int j = 0; j < grp; ++j) x = cfma(mg, x, agg[j][lane]);
  chain(x, true);
}

// grid (NC, B), one thread per state p: x_t = Lbar^{t+1} X_in + l_t with the in-chunk part
// l_t = Lbar l_{t-1} + V_t (l_{-1} = 0) run as a 64-step recurrence, written over V in place.
// The carried state enters through the directly computed power Lbar^{t+1}; only in-chunk lags
// go through the float32 product chain (at most 64 roundings).
__global__ void __launch_bounds__(256)
s5_chunk_apply(S5Work w, int L, int P, int NC) {
  constexpr int kB = 8;  // steps per batch; the loads of batch i + 1 are in flight during batch i
  const int c = blockIdx.x, b = blockIdx.y;
  const int t0 = c * kT;
  const int valid = min(kT, L - t0);
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const float2 xi = w.Xin[((size_t)b * NC + c) * P + p];
    const cf xin = {xi.x, xi.y};
    const float2 lb = w.lbar_pw[(size_t)P + p];
    const cf lam = {lb.x, lb.y};
    cf l = {0.f, 0.f};
    float2* row = reinterpret_cast<float2*>(w.xv) + ((size_t)b * L + t0) * P + p;
    float2 v[2][kB], a[2][kB];
    auto fetch = [&](int buf, int tb) {
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const bool in = tb + j < valid && DLR_IN(tb + j + 1, kT + 1) &&
                        DLR_IN(((size_t)b * L + t0 + tb + j) * P + p, (size_t)gridDim.y * L * P);
        v[buf][j] = in ? row[(size_t)(tb + j) * P] : make_float2(0.f, 0.f);
        a[buf][j] = in ? w.lbar_pw[(size_t)(tb + j + 1) * P + p] : make_float2(0.f, 0.f);
      }
    };
    fetch(0, 0);
#pragma unroll 1
    for (int tb = 0; tb < valid; tb += 2 * kB) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int tc = tb + half * kB;
        if (tc >= valid) break;
        if (tc + kB < valid) fetch(half ^ 1, tc + kB);
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          if (tc + j >= valid) break;
          l = cfma(lam, l, {v[half][j].x, v[half][j].y});
          const cf x = cfma({a[half][j].x, a[half][j].y}, xin, l);
          if (DLR_IN(((size_t)b * L + t0 + tc + j) * P + p, (size_t)gridDim.y * L * P))
            row[(size_t)(tc + j) * P] = make_float2(x.re, x.im);
        }
      }
    }
  }
}

// Tensor-core tier, V and x in bf16. One thread per (b, chunk c, four consecutive states),
// 16-byte loads and stores; both kernels run the recurrence x <- Lbar x + V_t over the chunk in
// float32 (64 roundings of the product, far below the bf16 rounding of V and x):
//   state16  from x = 0, keeping the chunk end state S_c,
//   apply16  from x = X_in (the state entering the chunk), writing x_t over V_t.
struct Quad {
  int b, c, p0;  // batch row, chunk, first of the four states
};
__device__ __forceinline__ bool quad_of(int B, int NC, int P, Quad& q) {
  const int nq = P / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * NC * nq) return false;
  q.p0 = int(i % nq) * 4;
  const long long r = i / nq;
  q.c = int(r % NC);
  q.b = int(r / NC);
  return true;
}
__device__ __forceinline__ void unpack4(uint4 v, cf (&x)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    x[k] = {f.x, f.y};
  }
}
__device__ __forceinline__ uint4 pack4(const cf (&x)[4]) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x[k].re, x[k].im);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool kApply>
__global__ void __launch_bounds__(256)
s5_chunk16(S5Work w, int B, int L, int P, int NC) {
  constexpr int kB = 8;
  Quad q;
  if (!quad_of(B, NC, P, q)) return;
  const int t0 = q.c * kT;
  const int valid = min(kT, L - t0);
  uint4* row = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat162*>(w.vx16) +
                                        ((size_t)q.b * L + t0) * P + q.p0);
  const size_t stride = (size_t)P / 4;  // uint4 per time step
  cf lam[4], x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 lb = w.lbar_pw[(size_t)P + q.p0 + k];
    lam[k] = {lb.x, lb.y};
    if (kApply) {
      const float2 xi = w.Xin[((size_t)q.b * NC + q.c) * P + q.p0 + k];
      x[k] = {xi.x, xi.y};
    } else {
      x[k] = {0.f, 0.f};
    }
  }
  uint4 v[2][kB];
  auto fetch = [&](int buf, int tb) {
#pragma unroll
    for (int j = 0; j < kB; ++j)
      v[buf][j] = (tb + j < valid &&
                   DLR_IN(((size_t)q.b * L + t0 + tb + j) * P + q.p0 + 3, (size_t)B * L * P))
                      ? row[(size_t)(tb + j) * stride]
                      : make_uint4(0, 0, 0, 0);
  };
  fetch(0, 0);
#pragma unroll 1
  for (int tb = 0; tb < valid; tb += 2 * kB) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int tc = tb + half * kB;
      if (tc >= valid) break;
      if (tc + kB < valid) fetch(half ^ 1, tc + kB);
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        if (tc + j >= valid) break;
        cf vin[4];
        unpack4(v[half][j], vin);
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = cfma(lam[k], x[k], vin[k]);
        if (kApply && DLR_IN(((size_t)q.b * L + t0 + tc + j) * P + q.p0 + 3, (size_t)B * L * P))
          row[(size_t)(tc + j) * stride] = pack4(x);
      }
    }
  }
  if (!kApply) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (DLR_IN(((size_t)q.b * NC + q.c) * P + q.p0 + k, (size_t)B * NC * P))
        w.S[((size_t)q.b * NC + q.c) * P + q.p0 + k] = make_float2(x[k].re, x[k].im);
  }
}

S5Work carve(void* ws, int64_t B, int64_t L, int64_t H, int64_t P, bool bf16, size_t* total) {
  const int64_t NC = (L + kT - 1) / kT;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~size_t(255);
    return o;
  };
  size_t o_b1 = bf16 ? 0 : take(sizeof(float) * 2 * 2 * P * H);
  size_t o_b2 = bf16 ? 0 : take(sizeof(float) * 2 * H * 2 * P);
  size_t o_pw = take(sizeof(float2) * P * (kT + 1));
  size_t o_lt = take(sizeof(float4) * P);
  size_t o_S = take(sizeof(float2) * B * NC * P);
  size_t o_X = take(sizeof(float2) * B * NC * P);
  size_t o_xv = bf16 ? 0 : take(sizeof(float) * B * L * 2 * P);
  size_t o_bt = 0, o_c16 = 0, o_vx16 = 0, o_S2 = 0;
  if (bf16) {
    o_bt = take(2 * 2 * P * H);
    o_c16 = take(2 * H * 2 * P);
    o_vx16 = take(2 * B * L * 2 * P);
    o_S2 = take(sizeof(float2) * B * NC * 2 * P);
  }
  if (total) *total = off;
  char* base = reinterpret_cast<char*>(ws);
  S5Work w;
  w.b1 = bf16 ? nullptr : reinterpret_cast<float*>(base + o_b1);
  w.b2 = bf16 ? nullptr : reinterpret_cast<float*>(base + o_b2);
  w.lbar_pw = reinterpret_cast<float2*>(base + o_pw);
  w.lbar_T = reinterpret_cast<float4*>(base + o_lt);
  w.S = reinterpret_cast<float2*>(base + o_S);
  w.Xin = reinterpret_cast<float2*>(base + o_X);
  w.xv = bf16 ? nullptr : reinterpret_cast<float*>(base + o_xv);
  w.bbar_t16 = bf16 ? base + o_bt : nullptr;
  w.cmat_t16 = bf16 ? base + o_c16 : nullptr;
  w.vx16 = bf16 ? base + o_vx16 : nullptr;
  w.S2 = bf16 ? reinterpret_cast<float2*>(base + o_S2) : nullptr;
  return w;
}

}  // namespace

// ---- S5 with a step that changes from step to step ----------------------------------------
// "Simplified State Space Layers for Sequence Modeling", section 2.2 (a different A_bar at each
// step, for irregularly sampled sequences) and section 6.3. Each batch row has observation gaps
// dt_k > 0; state p steps by Delta_p dt_k with a zero-order hold:
//   Lambda_bar_{p,k} = exp(Lambda_p Delta_p dt_k),  f_{p,k} = (Lambda_bar_{p,k} - 1) / Lambda_p,
//   x_k = Lambda_bar_k x_{k-1} + f_k (B~ u_k),      y_k = Re(C~ x_k) + D u_k.
// The float32 tier's kernels: V = u B~^T (the projection has no discretisation factor now),
// then a chunked scan whose multipliers are formed per step (exp of the real part, an exactly
// reduced phase, expm1 for Lambda_bar - 1 so that a short step loses nothing), the chunk carries
// with exp(Lambda Delta tau), tau the chunk's elapsed time summed in two-float arithmetic, and
// the output projection as before.

// per state: (Re Lambda Delta, Im Lambda Delta / pi as hi + lo), (1 / Lambda)
__global__ void s5tv_prep(const float* __restrict__ lambda, const float* __restrict__ log_delta,
                          const float2* __restrict__ Bt, const float2* __restrict__ Ct, int H,
                          int P, S5Work w, float4* __restrict__ st) {
  const int p = blockIdx.x;
  if (threadIdx.x == 0) {
    const double lr = lambda[2 * p], li = lambda[2 * p + 1];
    const double delta = exp((double)log_delta[p]);
    const double th = li * delta / 3.14159265358979323846;
    const float th_hi = (float)th;
    const double den = lr * lr + li * li;
    st[2 * p] = make_float4((float)(lr * delta), th_hi, (float)(th - (double)th_hi), 0.f);
    st[2 * p + 1] = make_float4((float)(lr / den), (float)(-li / den), 0.f, 0.f);
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float2 b = Bt[(size_t)p * H + h];
    store_operands(w, H, P, p, h, b.x, b.y, Ct[(size_t)h * P + p]);
  }
}

// Lambda_bar and (Lambda_bar - 1) / Lambda of one step of length dt
__device__ __forceinline__ void s5tv_coef(const float4 s0, const float4 s1, float dt, cf& abar,
                                          cf& f) {
  const float x = s0.x * dt;
  const float ph = reduce_halfturns(dt, s0.y, s0.z);  // (Im Lambda Delta dt) / pi mod 2
  float sh, ch;
  sincospif(0.5f * ph, &sh, &ch);
  const float sn = 2.f * sh * ch, cs = 1.f - 2.f * sh * sh;
  const float ex = expf(x), em = expm1f(x);
  abar = {ex * cs, ex * sn};
  const cf m = {fmaf(em, cs, -2.f * sh * sh), ex * sn};  // exp(z) - 1
  f = cmul(m, cf{s1.x, s1.y});
}

// chunk end states from a zero start (thread per (b, chunk, state), states fastest)
template <bool kApply>
__global__ void s5tv_chunks(float* __restrict__ xv, const float* __restrict__ dt,
                            const float4* __restrict__ st, const float2* __restrict__ Xin,
                            float2* __restrict__ S, int B, int L, int P, int NC) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)B * NC * P) return;
  const int p = (int)(i % P);
  const int64_t bc = i / P;
  const int c = (int)(bc % NC), b = (int)(bc / NC);
  const float4 s0 = st[2 * p], s1 = st[2 * p + 1];
  cf x = kApply ? cf{Xin[i].x, Xin[i].y} : cf{0.f, 0.f};
  const int k0 = c * kT, k1 = min(L, k0 + kT);
  const float* dtr = dt + (int64_t)b * L;
  float2* v = reinterpret_cast<float2*>(xv) + ((int64_t)b * L) * P + p;
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    cf a, f;
    s5tv_coef(s0, s1, __ldg(dtr + k), a, f);
    const bool in = DLR_IN(((int64_t)b * L + k) * P + p, (int64_t)B * L * P);
    const float2 vk = in ? v[(int64_t)k * P] : make_float2(0.f, 0.f);
    x = cfma(a, x, cmul(f, cf{vk.x, vk.y}));
    if (kApply && in) v[(int64_t)k * P] = make_float2(x.re, x.im);
  }
  if (!kApply) S[i] = make_float2(x.re, x.im);
}

// carries over the chunks of a row (thread per (b, state)): X_{c+1} = exp(Lambda Delta tau_c) X_c
// + S_c, tau_c the chunk's elapsed time in two-float arithmetic
__global__ void s5tv_carry(const float* __restrict__ dt, const float4* __restrict__ st,
                           const float2* __restrict__ S, float2* __restrict__ Xin, int B, int L,
                           int P, int NC) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)B * P) return;
  const int p = (int)(i % P), b = (int)(i / P);
  const float4 s0 = st[2 * p];
  const float* dtr = dt + (int64_t)b * L;
  cf X = {0.f, 0.f};
  for (int c = 0; c < NC; ++c) {
    const int64_t o = ((int64_t)b * NC + c) * P + p;
    if (!DLR_IN(o, (int64_t)B * NC * P)) break;
    Xin[o] = make_float2(X.re, X.im);
    ff tau = {0.f, 0.f};
    const int k0 = c * kT, k1 = min(L, k0 + kT);
    for (int k = k0; k < k1; ++k) tau = ff_add(tau, ff{__ldg(dtr + k), 0.f});
    // exp(Lambda Delta tau): magnitude from the real part, phase reduced exactly for tau.hi and
    // corrected by tau.lo
    const float mag = expf(s0.x * (tau.hi + tau.lo));
    float ph = reduce_halfturns(tau.hi, s0.y, s0.z) + s0.y * tau.lo;
    ph -= 2.f * rintf(0.5f * ph);
    float sn, cs;
    sincospif(ph, &sn, &cs);
    const float2 sc = S[o];
    X = cfma(cf{mag * cs, mag * sn}, X, cf{sc.x, sc.y});
  }
}

size_t s5_workspace_bytes(int64_t B, int64_t L, int64_t H, int64_t P, bool bf16) {
  size_t total = 0;
  carve(nullptr, B, L, H, P, bf16, &total);
  return total;
}

cudaError_t launch_tc_gemm(const void* A, bool a_f32, const void* B, void* C, bool c_bf16,
                           int M, int N, int K, const float* D, const float* E, int* status,
                           cudaStream_t s, const float2* lam, float2* sums, int L, int NC);
cudaError_t launch_tc_gemm_apply(const void* V, const void* C, float* y, int M, int N, int K,
                                 const float* D, const float* E, const float2* lam,
                                 const float2* xin, int L, int P, int NC, int* status,
                                 cudaStream_t s);
cudaError_t launch_tc_gemm_x3(const float* A, const float* Bh, const float* Bl, float* C, int M,
                              int N, int K, const float* D, const float* E, int* status,
                              cudaStream_t s);

// The chunked diagonal scan shared by both tiers: V -> x in place, in w.xv (float32 tier) or
// w.vx16 (tensor-core tier). `fused` (tensor-core tier, L a multiple of 64): the input
// projection has written the chunk end states in halves and the output projection runs the
// apply step on its operand tiles, so only the carries run here.
static cudaError_t s5_scan_xv(const S5Work& w, int B, int L, int P, bool bf16, bool fused,
                              cudaStream_t s) {
  const int NC = (L + kT - 1) / kT;
  const int threads = P < 256 ? P : 256;  // P is a multiple of 32
  const long long quads = (long long)B * NC * (P / 4);
  const int grid16 = (int)((quads + 255) / 256);
  if (fused) {
    s5_carry_groups<true><<<dim3(P / 32, B), 1024, 0, s>>>(w, B, P, NC);
    return cudaGetLastError();
  }
  if (bf16)
    s5_chunk16<false><<<grid16, 256, 0, s>>>(w, B, L, P, NC);
  else
    s5_chunk_state<<<dim3(NC, B), threads, 0, s>>>(w, L, P, NC);
  if (bf16)
    s5_carry_groups<false><<<dim3(P / 32, B), 1024, 0, s>>>(w, B, P, NC);
  else
    s5_carry<<<(B * P + 7) / 8, 256, 0, s>>>(w, B, P, NC);
  if (bf16)
    s5_chunk16<true><<<grid16, 256, 0, s>>>(w, B, L, P, NC);
  else
    s5_chunk_apply<<<dim3(NC, B), threads, 0, s>>>(w, L, P, NC);
  return cudaGetLastError();
}

cudaError_t launch_s5(const float* u, const float* lambda, const float* log_delta,
                      const float* Bt, const float* Ct, const float* D, int B, int L, int H, int P,
                      bool bf16, bool bilinear, float* y, void* ws, int* status,
                      cudaStream_t s) {
  S5Work w = carve(ws, B, L, H, P, bf16, nullptr);
  s5_prep<<<P, 128, 0, s>>>(lambda, log_delta, reinterpret_cast<const float2*>(Bt),
                            reinterpret_cast<const float2*>(Ct), H, P, bilinear ? 1 : 0, w);
  const int M = B * L;
  cudaError_t e;
  if (!bf16) {
    // float32 tier: both projections as three tf32 products on the tensor cores, the scan in
    // float32 between them
    const size_t n1 = (size_t)2 * P * H;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_tc_gemm_x3(u, w.b1, w.b1 + n1, w.xv, M, 2 * P, H, nullptr, nullptr, status,
                               s)) != cudaSuccess)
      return e;
    if ((e = s5_scan_xv(w, B, L, P, false, false, s)) != cudaSuccess) return e;
    return launch_tc_gemm_x3(w.xv, w.b2, w.b2 + n1, y, M, H, 2 * P, D, u, status, s);
  }
  // tensor cores with f32 accumulation: the input projection reads the float32 u (converted to
  // bf16 in the kernel) and writes bf16 V, the scan in f32 arithmetic, the output projection
  // adds D (.) u. When L is a multiple of 64 (tiles of 128 steps start on chunk starts) the
  // output projection turns V into x itself as its operand tiles arrive; otherwise the apply
  // kernel writes bf16 x over V first.
  const bool fused = L % kT == 0;
  const int NC = (L + kT - 1) / kT;
  if ((e = launch_tc_gemm(u, true, w.bbar_t16, w.vx16, true, M, 2 * P, H, nullptr, nullptr,
                          status, s, w.lbar_pw + P, fused ? w.S2 : nullptr, L, NC)) != cudaSuccess)
    return e;
  if ((e = s5_scan_xv(w, B, L, P, true, fused, s)) != cudaSuccess) return e;
  if (fused)
    return launch_tc_gemm_apply(w.vx16, w.cmat_t16, y, M, H, 2 * P, D, u, w.lbar_pw + P, w.Xin,
                                L, P, NC, status, s);
  return launch_tc_gemm(w.vx16, false, w.cmat_t16, y, false, M, H, 2 * P, D, u, status, s,
                        nullptr, nullptr, 0, 0);
}

cudaError_t launch_s5_tv(const float* u, const float* dt, const float* lambda,
                         const float* log_delta, const float* Bt, const float* Ct,
                         const float* D, int B, int L, int H, int P, float* y, void* ws,
                         int* status, cudaStream_t s) {
  S5Work w = carve(ws, B, L, H, P, false, nullptr);
  // the per-state constants in the (otherwise unused) power table: 2 float4 per state
  float4* st = reinterpret_cast<float4*>(w.lbar_pw);
  s5tv_prep<<<P, 128, 0, s>>>(lambda, log_delta, reinterpret_cast<const float2*>(Bt),
                              reinterpret_cast<const float2*>(Ct), H, P, w, st);
  const int M = B * L;
  const int NC = (L + kT - 1) / kT;
  const size_t n1 = (size_t)2 * P * H;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = launch_tc_gemm_x3(u, w.b1, w.b1 + n1, w.xv, M, 2 * P, H, nullptr, nullptr, status,
                             s)) != cudaSuccess)
    return e;
  const int64_t nchunk = (int64_t)B * NC * P;
  const unsigned gc = (unsigned)((nchunk + 255) / 256);
  s5tv_chunks<false><<<gc, 256, 0, s>>>(w.xv, dt, st, nullptr, w.S, B, L, P, NC);
  s5tv_carry<<<(unsigned)(((int64_t)B * P + 127) / 128), 128, 0, s>>>(dt, st, w.S, w.Xin, B, L,
                                                                        P, NC);
  s5tv_chunks<true><<<gc, 256, 0, s>>>(w.xv, dt, st, w.Xin, nullptr, B, L, P, NC);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_tc_gemm_x3(w.xv, w.b2, w.b2 + n1, y, M, H, 2 * P, D, u, status, s);
}

}  // namespace dlr
