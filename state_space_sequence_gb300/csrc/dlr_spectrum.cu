// dlr_spectrum.cu -- the circulant spectrum of the Re-cast DLR kernel straight from the
// parameters ("The Annotated S4", part 2: the kernel's truncated generating function evaluated
// at the roots of unity instead of the kernel itself; for a diagonal state matrix ("Simplifying
// and Understanding State Space Models with Diagonal Linear RNNs", section 2, K_j = sum_n W_n
// lambda_n^j) it is a sum of N geometric series per frequency). The result is written into the
// workspace of the FFT convolution in exactly the form dlr_conv_spectrum leaves there (twiddle
// tables, then the scaled Hermitian half of each channel's spectrum), so dlr_conv_apply runs on
// it unchanged: the layer by FFT without materialising K.
//
// With omega = exp(-2 pi i / M), M = 2n the circulant size, and
//   A(k) = sum_n W_n G(lambda_n omega^k),   G(z) = sum_{j<L} z^j = (1 - z^L) / (1 - z),
// the real kernel's column [K_0 .. K_{L-1}, 0 ..] has the spectrum C_k = (A(k) + conj(A(-k))) / 2;
// the bidirectional layer (section 2.1) adds the anti-causal column of the second parameter
// set, (A2(-k) + conj(A2(k))) / 2.
//
// Numerics. G = expm1(L l) / expm1(l) with l = log z = -a^2 + i pi phi (phi in half-turns):
//   - expm1(x + i pi f) = expm1(x) cos(pi f) - 2 sin^2(pi f / 2) + i e^x sin(pi f), from one
//     sincospif of f / 2, stays accurate as l -> 0 (no cancellation in 1 - z);
//   - phi = theta / pi -/+ k / n is formed from the two-float reduced theta / pi with the
//     subtraction done where it is exact (Sterbenz) next to a pole, so a bin close to
//     lambda omega^k = 1 keeps the small offset to full relative precision;
//   - L phi mod 2 = (L theta / pi mod 2) -/+ ((L k) mod 2n) / n, the first part reduced exactly
//     in two-float arithmetic, the second an exact integer ratio; where |L phi| < 1 it is the
//     product L phi itself, which keeps its relative precision as the angle shrinks;
//   - where |L l| < 2^-10 (a pole of the series, reached by channels on the unit circle) G is
//     L (1 + (L - 1) l / 2), whose omitted terms are below (L |l|)^2 / 6 relative;
//   - away from the pole (|phi| >= 1/16 half-turn, so |1 - z| > 0.19 when |lambda| ~ 1) the
//     same G = (z^L - 1) / (z - 1) comes from products instead: z = e^{-a^2} cis(theta) times
//     the bin's cis(-pi k / n), z^L = lambda^L times the bin's cis(-pi v_k); their absolute
//     errors of a few 2^-24 stay below 1e-6 relative to |z - 1| there.
// Cost: per state and bin two complex divisions (the bins at +-k), and near a pole two
// sincospif -- O(N L) per channel with more work per term than the O(N L) multiply-adds of
// dlr_kernel followed by an O(L log L) FFT, so the kernel route stays the default; this one
// needs no kernel buffer and no spectrum FFT.
#include <cuda_runtime.h>

#include "dlr_common.cuh"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 11;
int conv_log2_size(int64_t L);
cudaError_t launch_twiddles(int lg, void* ws, cudaStream_t s);  // dlr_conv.cu

namespace {

constexpr int kSpecThreads = 256;
constexpr int kMaxStates = 256;   // states per channel (shared-memory parameters)

struct SpecState {
  float a2, em1, e1, em1L, e1L;  // a^2, expm1(-a^2), e^-a^2, expm1(-L a^2), e^-L a^2
  float th_hi, th_lo;            // theta / pi in about [-1, 1], two-float
  float rL;                      // L theta / pi mod 2, in about [-1, 1]
  float w_re, w_im;
  float z_re, z_im;              // lambda = e^-a^2 cis(theta)
  float zl_re, zl_im;            // lambda^L = e^-L a^2 cis(pi rL)
};

// expm1(x + i pi f) from expm1(x), e^x and f (|f| <= 2)
__device__ __forceinline__ cf cexpm1_hf(float em1x, float ex, float f) {
  float s, c;
  sincospif(0.5f * f, &s, &c);
  const float sin_f = 2.f * s * c, cos_f = 1.f - 2.f * s * s;
  return {fmaf(em1x, cos_f, -2.f * s * s), ex * sin_f};
}

__device__ __forceinline__ float wrap2(float f) {  // to about (-1, 1]
  if (f > 1.f) f -= 2.f;
  if (f <= -1.f) f += 2.f;
  return f;
}

// G(lambda omega^{sign k}) for one state; kn = k / n (exact), vk = ((L k) mod 2n) / n (exact).
__device__ __forceinline__ cf geom(const SpecState& p, int L, float kn, float vk, int sign) {
  // phi = theta / pi - sign * k / n, the subtraction exact next to a pole: theta / pi is moved
  // by 2 (two-sum, the error kept) to the side where the pole can lie
  float t_hi = p.th_hi, t_e = 0.f;
  if (sign > 0 && t_hi < 0.f) {
    const ff t = two_sum(t_hi, 2.f);
    t_hi = t.hi;
    t_e = t.lo;
  } else if (sign < 0 && t_hi > 0.f) {
    const ff t = two_sum(t_hi, -2.f);
    t_hi = t.hi;
    t_e = t.lo;
  }
  const float d = sign > 0 ? t_hi - kn : t_hi + kn;
  const float phi = wrap2(d + (t_e + p.th_lo));
  const float Lf = (float)L;
  // L phi mod 2: near a pole (|L phi| < 1) the product of the accurate small phi, elsewhere the
  // exactly reduced difference (absolute error about 2^-24 half-turns on an O(1) angle)
  const float Phi = (fabsf(phi) * Lf < 1.f) ? Lf * phi
                                            : wrap2(wrap2(p.rL - (sign > 0 ? vk : -vk)));
  const float lr = -p.a2, li = 3.14159265358979f * phi;
  if (Lf * (fabsf(lr) + fabsf(li)) < 0x1p-10f) {
    // G = L (1 + (L - 1) l / 2) next to the pole
    const float h = 0.5f * (Lf - 1.f);
    return {Lf * fmaf(h, lr, 1.f), Lf * h * li};
  }
  const cf num = cexpm1_hf(p.em1L, p.e1L, Phi);
  const cf den = cexpm1_hf(p.em1, p.e1, phi);
  const float inv = 1.f / fmaf(den.re, den.re, den.im * den.im);
  return {(num.re * den.re + num.im * den.im) * inv, (num.im * den.re - num.re * den.im) * inv};
}

// G away from the pole: (z^L - 1) / (z - 1) with z = lambda cis(-sign pi k / n) and
// z^L = lambda^L cis(-sign pi v_k), (ck, sk) = cis(-pi k / n), (cv, sv) = cis(-pi v_k).
__device__ __forceinline__ cf geom_far(const SpecState& p, float ck, float sk, float cv, float sv,
                                       int sign) {
  const float sks = sign > 0 ? sk : -sk, svs = sign > 0 ? sv : -sv;
  const float zr = p.z_re * ck - p.z_im * sks, zi = fmaf(p.z_re, sks, p.z_im * ck);
  const float nr = fmaf(p.zl_re, cv, fmaf(-p.zl_im, svs, -1.f));
  const float ni = fmaf(p.zl_re, svs, p.zl_im * cv);
  const float dr = zr - 1.f, di = zi;
  const float inv = 1.f / fmaf(dr, dr, di * di);
  return {(nr * dr + ni * di) * inv, (ni * dr - nr * di) * inv};
}

// phi = theta / pi - sign k / n folded to about (-1, 1] (for the choice of path only)
__device__ __forceinline__ float phase_near(const SpecState& p, float kn, int sign) {
  float d = sign > 0 ? p.th_hi - kn : p.th_hi + kn;
  d -= 2.f * rintf(0.5f * d);
  return d;
}

// One CTA per (block of bins, channel); the channel's state parameters in shared memory.
__global__ void __launch_bounds__(kSpecThreads)
    spectrum_direct(const float* __restrict__ lr1, const float* __restrict__ li1,
                    const float2* __restrict__ W1, const float* __restrict__ lr2,
                    const float* __restrict__ li2, const float2* __restrict__ W2, int N, int L,
                    int lg, float2* __restrict__ spec) {
  __shared__ SpecState st[2][kMaxStates];
  const int h = blockIdx.y;
  const int n = 1 << lg;
  const int sets = lr2 ? 2 : 1;
  for (int i = threadIdx.x; i < sets * N; i += blockDim.x) {
    const int set = i / N, m = i - set * N;
    const float* lr = set ? lr2 : lr1;
    const float* li = set ? li2 : li1;
    const float2* W = set ? W2 : W1;
    const size_t o = (size_t)h * N + m;
    const lam_param lp = make_lam_param(lr[o], li[o]);
    SpecState p;
    p.a2 = lp.a2;
    p.em1 = expm1f(-lp.a2);
    p.e1 = expf(-lp.a2);
    p.em1L = expm1f(-(float)L * lp.a2);
    p.e1L = expf(-(float)L * lp.a2);
    p.th_hi = lp.th_hi;
    p.th_lo = lp.th_lo;
    p.rL = reduce_halfturns((float)L, lp.th_hi, lp.th_lo);
    float sn, cs;
    sincospif(lp.th_hi + lp.th_lo, &sn, &cs);
    p.z_re = p.e1 * cs;
    p.z_im = p.e1 * sn;
    sincospif(p.rL, &sn, &cs);
    p.zl_re = p.e1L * cs;
    p.zl_im = p.e1L * sn;
    const float2 w = W[o];
    p.w_re = w.x;
    p.w_im = w.y;
    st[set][m] = p;
  }
  __syncthreads();
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k > n) return;
  const float kn = ldexpf((float)k, -lg);
  const long long lk = ((long long)L * (long long)k) % (2LL * n);
  const float vk = ldexpf((float)lk, -lg);
  // the bin's twiddles for the far-from-pole path: cis(-pi k / n), cis(-pi v_k)
  float sk, ck, sv, cv;
  sincospif(kn, &sk, &ck);
  sk = -sk;
  sincospif(vk, &sv, &cv);
  sv = -sv;
  float cre = 0.f, cim = 0.f;
#pragma unroll 1
  for (int set = 0; set < sets; ++set) {
    // causal set: (A(k) + conj(A(-k))) / 2; anti-causal set: (A(-k) + conj(A(k))) / 2
    const int sp = set ? -1 : 1;
    float are = 0.f, aim = 0.f, bre = 0.f, bim = 0.f;
#pragma unroll 2
    for (int m = 0; m < N; ++m) {
      const SpecState& p = st[set][m];
      const cf gp = fabsf(phase_near(p, kn, sp)) < 0.0625f ? geom(p, L, kn, vk, sp)
                                                          : geom_far(p, ck, sk, cv, sv, sp);
      const cf gm = fabsf(phase_near(p, kn, -sp)) < 0.0625f ? geom(p, L, kn, vk, -sp)
                                                           : geom_far(p, ck, sk, cv, sv, -sp);
      are = fmaf(p.w_re, gp.re, fmaf(-p.w_im, gp.im, are));
      aim = fmaf(p.w_re, gp.im, fmaf(p.w_im, gp.re, aim));
      bre = fmaf(p.w_re, gm.re, fmaf(-p.w_im, gm.im, bre));
      bim = fmaf(p.w_re, gm.im, fmaf(p.w_im, gm.re, bim));
    }
    cre += 0.5f * (are + bre);
    cim += 0.5f * (aim - bim);
  }
  // the convolution's spectral step expects C_k / (4n) (1/M for the inverse transform and
  // 1/2 for its unpack); rows above 2^14 points use the cluster transform's order
  const float scale = 1.0f / (float)(4 * n);
  size_t idx = (size_t)k;
  if (lg > 14 && k < n) {
    const int nl = n >> 3;
    idx = (size_t)(k & 7) * nl + (k >> 3);
  }
  if (DLR_IN(idx, n + 1)) spec[(size_t)h * (n + 1) + idx] = make_float2(cre * scale, cim * scale);
}

}  // namespace

size_t conv_workspace_bytes(int64_t H, int64_t L);

// The spectra of H channels from their parameters (second set NULL when causal) into the
// convolution workspace `ws` (dlr_conv_workspace_size bytes): twiddle tables and spectra as
// dlr_conv_spectrum writes them.
cudaError_t launch_spectrum_direct(const float* lr1, const float* li1, const float* W1,
                                   const float* lr2, const float* li2, const float* W2, int H,
                                   int N, int L, void* ws, cudaStream_t s) {
  if (N < 1 || N > kMaxStates) return cudaErrorInvalidValue;
  const int lg = conv_log2_size(L);
  const int n = 1 << lg;
  cudaError_t e = launch_twiddles(lg, ws, s);
  if (e != cudaSuccess) return e;
  // the spectra follow the twiddle tables (the layout of the convolution workspace)
  const size_t twb = (sizeof(float2) * (size_t)n + 255) & ~size_t(255);
  const size_t tw2b = (sizeof(float2) * 2 * (size_t)n + 255) & ~size_t(255);
  float2* spec = reinterpret_cast<float2*>(static_cast<char*>(ws) + twb + tw2b);
  const dim3 grid((unsigned)((n + 1 + kSpecThreads - 1) / kSpecThreads), (unsigned)H);
  spectrum_direct<<<grid, kSpecThreads, 0, s>>>(lr1, li1, reinterpret_cast<const float2*>(W1),
                                                 lr2, li2, reinterpret_cast<const float2*>(W2),
                                                 N, L, lg, spec);
  return cudaGetLastError();
}

}  // namespace dlr
