/*
 * dlr.h -- C ABI of libdlr.so: diagonal linear recurrences (DLR, diagonal SSM, S5) on one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library never
 *    allocates, frees or keeps them; scratch memory is passed in as `workspace`, sized by the
 *    matching *_workspace_size() query (a size of 0 means no workspace is needed and the
 *    pointer may be NULL).
 *  - Sizes are int64_t element counts. Real tensors are float32, row-major, innermost index
 *    last. A complex value is two consecutive float32 (re, im).
 *  - Every compute call is asynchronous on `stream` (NULL = legacy default stream). Argument
 *    validation happens before anything is launched: an invalid call returns
 *    DLR_ERR_INVALID_ARG / DLR_ERR_UNSUPPORTED / DLR_ERR_WORKSPACE synchronously and launches
 *    nothing. A launch failure returns DLR_ERR_CUDA. Faults detected on the device (a bounded
 *    wait that ran out) are latched in a device status word read by dlr_get_device_status().
 *  - Tensor pointers must be 16-byte aligned (128-bit vector loads / bulk copies).
 *  - The arithmetic is float32 throughout except where an entry point says otherwise.
 *
 * Notation follows "Simplifying and Understanding State Space Models with Diagonal Linear
 * RNNs" (DLR) and "Simplified State Space Layers for Sequence Modeling" (S5).
 */
#ifndef DLR_H_
#define DLR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* dlr_stream_t;

typedef enum {
  DLR_OK = 0,
  DLR_ERR_INVALID_ARG = 1, /* NULL/misaligned pointer, non-positive or inconsistent size */
  DLR_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement           */
  DLR_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed                 */
  DLR_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (see dlr_get_device_status) */
  DLR_ERR_WORKSPACE = 5,   /* workspace missing or smaller than *_workspace_size()        */
  DLR_ERR_BOUNDS = 6       /* bounds-checked build only: an index outside its buffer was
                              found and the access skipped (see dlr_bounds_site)           */
} dlr_status;

/* Kernel cast. DLR paper section 2: y_k = sum_{j<=k} Re(K_j) u_{k-j} (the Re cast);
 * section 2.1: DLR-prod uses Re(K_j) * Im(K_j) instead. */
typedef enum { DLR_CAST_RE = 0, DLR_CAST_RE_IM = 1 } dlr_cast;

/* Direction. DLR paper section 2.1: the bidirectional DLR sums two independent DLRs, the
 * second one applied to the time-reversed sequence (lag 0 is counted by both). */
typedef enum { DLR_CAUSAL = 0, DLR_BIDIR = 1 } dlr_dir;

/* Precision tier of s5_layer's projections. */
typedef enum { DLR_FP32 = 0, DLR_BF16_TC = 1 } dlr_prec;

/* Discretisation of the continuous S5 system: the zero-order hold (S5 paper section 3) or the
 * bilinear transform ("The Annotated S4", part 1). */
typedef enum { DLR_DISC_ZOH = 0, DLR_DISC_BILINEAR = 1 } dlr_disc;

/* Decay-rate reparameterisations f(w) (the StableSSM discussion): e^w, log(1 + e^w),
 * 1 / (a w^2 + b). */
typedef enum { DLR_REPARAM_EXP = 0, DLR_REPARAM_SOFTPLUS = 1, DLR_REPARAM_BEST = 2 } dlr_reparam;

/* Kernels behind dlr_scan_ex. DLR_SCAN_FP32: every product in float32 FMA (N <= 128).
 * DLR_SCAN_TENSOR: the chunked scan's three dense contractions on tensor cores, each operand
 * split into two float16 halves with power-of-two scaling (three MMAs per product, float32
 * accumulation), the carries between chunks in float32 (N <= 64). DLR_SCAN_AUTO: TENSOR
 * when N <= 64, else FP32. */
typedef enum { DLR_SCAN_AUTO = 0, DLR_SCAN_FP32 = 1, DLR_SCAN_TENSOR = 2 } dlr_scan_algo;

/*
 * dlr_kernel -- the DLR convolution kernel (DLR paper section 2, Eq. 3/4 and section 2.2):
 *   lambda_{h,n} = exp(-log_re[h,n]^2 + i*log_im[h,n])
 *   K_{h,j}      = sum_n W_{h,n} lambda_{h,n}^j ,  j = 0..L-1
 *   out K[h,j]   = Re K_{h,j}                 (cast = DLR_CAST_RE)
 *                = Re K_{h,j} * Im K_{h,j}    (cast = DLR_CAST_RE_IM, "DLR-prod")
 * log_re, log_im: [H, N] float32. W: [H, N, 2] complex. K: [H, L] float32 (written).
 * lambda^j is formed from the parameters with an exactly reduced phase j*theta, not by
 * repeated multiplication of a rounded lambda. Limits: 1 <= N, 1 <= L < 2^24.
 */
dlr_status dlr_kernel(const float* log_re, const float* log_im, const float* W, int64_t H,
                      int64_t N, int64_t L, dlr_cast cast, float* K, dlr_stream_t stream);

/*
 * dlr_conv -- apply the (already cast) real kernels by FFT convolution (DLR paper section 2.1
 * and appendix A.1: the Toeplitz product as a circulant product of size >= 2L):
 *   causal : y[b,h,k] = sum_{j=0}^{k} K_fwd[h,j] u[b,h,k-j]
 *   bidir  : y[b,h,k] = sum_{j=0}^{k} K_fwd[h,j] u[b,h,k-j] + sum_{j=0}^{L-1-k} K_bwd[h,j] u[b,h,k+j]
 * u, y: [B, H, L] float32. K_fwd, K_bwd: [H, L] float32 (K_bwd NULL when dir = DLR_CAUSAL).
 * workspace: >= dlr_conv_workspace_size(H, L, dir) bytes of device memory holding the twiddle
 * table and the per-channel kernel spectra (no initialisation needed; overwritten).
 * u and y must not overlap. Limits: 1 <= L <= 65536 (rows longer than 16384 are transformed
 * by a cluster of 8 CTAs sharing the row through distributed shared memory).
 * dlr_conv is exactly dlr_conv_spectrum followed by dlr_conv_apply on the same stream.
 */
size_t dlr_conv_workspace_size(int64_t H, int64_t L, dlr_dir dir);
dlr_status dlr_conv(const float* u, const float* K_fwd, const float* K_bwd, dlr_dir dir,
                    int64_t B, int64_t H, int64_t L, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_conv_spectrum -- first half of dlr_conv: writes the twiddle table and the spectrum of
 * each channel's length-2n circulant column (n = next power of two >= L) into `workspace`.
 * The spectra depend only on the kernels, so one call can serve many dlr_conv_apply calls
 * (e.g. every batch) as long as the workspace is left untouched in between.
 */
dlr_status dlr_conv_spectrum(const float* K_fwd, const float* K_bwd, dlr_dir dir, int64_t H,
                             int64_t L, void* workspace, size_t workspace_bytes,
                             dlr_stream_t stream);

/*
 * dlr_conv_spectrum_direct -- the spectra that dlr_conv_spectrum would compute from the Re-cast
 * kernel, evaluated straight from the parameters instead ("The Annotated S4", part 2: the
 * truncated generating function of the kernel at the roots of unity; for the diagonal DLR of
 * "Simplifying and Understanding State Space Models with Diagonal Linear RNNs", section 2, a
 * sum of N geometric series per frequency: C_k = (A(k) + conj(A(-k))) / 2 with
 * A(k) = sum_n W_n (1 - (lambda_n w^k)^L) / (1 - lambda_n w^k), w = exp(-2 pi i / M)), so the
 * layer by FFT needs neither the kernel K nor its transform: dlr_conv_spectrum_direct followed
 * by dlr_conv_apply gives the same y as dlr_kernel + dlr_conv. With dir = DLR_BIDIR the second
 * parameter set forms the anti-causal column (section 2.1), lag 0 counted by both directions.
 *  - log_re, log_im [H, N], W [H, N, 2] (8-byte aligned): device pointers as in dlr_kernel;
 *    the second set NULL when dir = DLR_CAUSAL.
 *  - workspace: dlr_conv_workspace_size(H, L, dir) bytes, written (twiddle tables and spectra)
 *    in the layout dlr_conv_apply reads.
 *  - Re cast only (DLR-prod has no N-term generating function); N <= 256, L <= 65536, else
 *    DLR_ERR_UNSUPPORTED.
 *  - Cost O(N L) complex divisions per channel: for the workloads measured here it is slower
 *    than dlr_kernel + dlr_conv_spectrum; it needs no [H, L] kernel buffer.
 */
dlr_status dlr_conv_spectrum_direct(const float* log_re, const float* log_im, const float* W,
                                    const float* log_re2, const float* log_im2,
                                    const float* W2, dlr_dir dir, int64_t H, int64_t N,
                                    int64_t L, void* workspace, size_t workspace_bytes,
                                    dlr_stream_t stream);

/*
 * dlr_conv_apply -- second half of dlr_conv: y = FFT convolution of u with the spectra that
 * a preceding dlr_conv_spectrum (same H and L, earlier in stream order) left in `workspace`.
 * Reads the workspace only; one kernel launch, one CTA per (b, h) row.
 */
dlr_status dlr_conv_apply(const float* u, int64_t B, int64_t H, int64_t L, float* y,
                          const void* workspace, size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_conv_noalloc -- the same computation as dlr_conv (same kernels, same results), for
 * callers that cannot allocate device memory: programs whose host application owns every byte
 * of device memory through a plan fixed at start-up, or code on a latency-critical path where
 * the device-wide synchronisation a cudaMalloc may cause is not acceptable. The papers have no
 * counterpart of this entry point; it exists for such deployments only.
 *  - It allocates nothing (no cudaMalloc, no cudaFree, no allocating library call). Its scratch
 *    is a fixed 16 MiB array inside the library's device memory, held by every GPU that loads
 *    the library until the process exits.
 *  - Limit: the call needs 24*n (two twiddle tables) + 8*H*(n+1) bytes of scratch, n = the next
 *    power of two >= L; larger requests return DLR_ERR_WORKSPACE and launch nothing (e.g.
 *    up to H = 508 at L = 4096, up to H = 124 at L = 16384). This entry point takes
 *    L <= 16384 only (one CTA per row); longer rows, which dlr_conv runs on its cluster path,
 *    return DLR_ERR_UNSUPPORTED here.
 *  - The first call on a device looks up the scratch's device address (with that device
 *    current) and caches it; make that first call before any stream capture.
 *  - All calls in the process share the one scratch array, which keeps the last call's
 *    contents; nothing in it needs to start at zero. Calls whose executions overlap on the GPU
 *    (different streams, or several host threads) race on it: serialise them.
 * Arguments, layouts and other errors as for dlr_conv.
 */
dlr_status dlr_conv_noalloc(const float* u, const float* K_fwd, const float* K_bwd, dlr_dir dir,
                            int64_t B, int64_t H, int64_t L, float* y, dlr_stream_t stream);

/*
 * dlr_scan -- the DLR as a chunked scan of the recurrence (DLR paper section 2, Eq. 1; S5
 * paper section 2.2, parallel scan over a diagonal state matrix):
 *   x_{n,k} = lambda_n x_{n,k-1} + u_k  (x_{-1} = 0),   y_k = sum_n Re(W_n x_{n,k})
 * computed per (b,h) row without materialising the kernel. With dir = DLR_BIDIR the second
 * parameter set (log_re2, log_im2, W2) runs on the reversed sequence and its output is added.
 * Only the Re cast exists here (DLR-prod has no N-state recurrence; use dlr_conv).
 * u, y: [B, H, L]; parameter layouts as in dlr_kernel. u and y must not overlap.
 * Runs the tensor-core kernel of dlr_scan_ex when N <= 64 (it needs `workspace` of at least
 * dlr_scan_workspace_size(B, H, N, L) bytes, else DLR_ERR_WORKSPACE), the float32 one
 * otherwise (workspace unused, may be NULL). Limits: 1 <= N <= 128, 1 <= L < 2^24.
 */
size_t dlr_scan_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L);
dlr_status dlr_scan(const float* u, const float* log_re, const float* log_im, const float* W,
                    const float* log_re2, const float* log_im2, const float* W2, dlr_dir dir,
                    int64_t B, int64_t H, int64_t N, int64_t L, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_scan_ex -- dlr_scan with the kernel chosen by `algo` (dlr_scan is DLR_SCAN_AUTO).
 * DLR_SCAN_TENSOR computes, per channel and chunk of 64 steps, the chunk-end states, the
 * in-chunk Toeplitz product with the first 64 kernel taps and the carried-state output as
 * tensor-core contractions, and runs the carry recurrence across chunks in float32 (S5 paper
 * section 2.2; the chunked form of the DLR recurrence). A first kernel writes each channel's
 * tables (powers of lambda, the taps, the operand images) into `workspace`
 * (dlr_scan_workspace_size bytes: about 83 KB per channel). Same arguments, layouts and limits
 * as dlr_scan, except N <= 64 for DLR_SCAN_TENSOR (DLR_ERR_UNSUPPORTED above). Faults of its
 * bounded waits are reported through dlr_get_device_status(). DLR_SCAN_FP32 needs no
 * workspace.
 */
dlr_status dlr_scan_ex(const float* u, const float* log_re, const float* log_im, const float* W,
                       const float* log_re2, const float* log_im2, const float* W2, dlr_dir dir,
                       int64_t B, int64_t H, int64_t N, int64_t L, float* y,
                       dlr_scan_algo algo, void* workspace, size_t workspace_bytes,
                       dlr_stream_t stream);

/*
 * dlr_scan_prepare / dlr_scan_apply -- the two halves of the tensor-core dlr_scan for one
 * parameter set (same method and precision as DLR_SCAN_TENSOR), for callers that run many
 * batches through the same parameters: the tables depend only on (log_re, log_im, W).
 * dlr_scan_prepare writes the channel tables into `workspace` (dlr_scan_workspace_size bytes,
 * 16-byte aligned; N <= 64, else DLR_ERR_UNSUPPORTED). dlr_scan_apply runs the layer on u with
 * the tables that a preceding dlr_scan_prepare (same H and N, earlier in stream order) left in
 * `workspace`, which it only reads: reverse = 0 writes y = DLR(u); reverse = 1 adds
 * rev(DLR(rev(u))) to y (the second direction of the bidirectional layer, DLR paper section
 * 2.1). u, y: [B, H, L], not overlapping each other or the workspace. dlr_scan_ex with
 * DLR_SCAN_TENSOR is prepare + apply (twice for DLR_BIDIR). One kernel launch each; faults of
 * apply's bounded waits are reported through dlr_get_device_status().
 */
dlr_status dlr_scan_prepare(const float* log_re, const float* log_im, const float* W, int64_t H,
                            int64_t N, void* workspace, size_t workspace_bytes,
                            dlr_stream_t stream);
dlr_status dlr_scan_apply(const float* u, int64_t B, int64_t H, int64_t N, int64_t L,
                          int reverse, float* y, const void* workspace, size_t workspace_bytes,
                          dlr_stream_t stream);

/*
 * dlr_scan_host -- the causal DLR layer (Re cast) of dlr_scan with DLR_SCAN_TENSOR on HOST
 * buffers: u, y [B, H, L] and log_re, log_im [H, N], W [H, N, 2] are host pointers (page-locked
 * for the copies to overlap anything), the device working copies live in `workspace` (device
 * memory, dlr_scan_host_workspace_size bytes, 16-byte aligned; the library still allocates
 * nothing). The batch is split into pieces of about a quarter of the batch rows, the first
 * and last groups halved (for B < 4, into channel groups; one piece when L % 4 != 0): the
 * copies in, the layer and the copies out run on three internal streams joined by events, so
 * the copy of one piece in, the compute of another and the copy of a third out overlap. Asynchronous with respect to the host; ordered
 * after the work already on `stream` and before the work enqueued on it later, so y may be
 * read after a synchronisation of `stream`. Same limits as dlr_scan_apply (N <= 64).
 * If an enqueue fails part-way, the call waits for the pieces already queued before it returns
 * the error, so the host buffers and the workspace are no longer in use when it returns.
 */
size_t dlr_scan_host_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L);
dlr_status dlr_scan_host(const float* u, const float* log_re, const float* log_im,
                         const float* W, int64_t B, int64_t H, int64_t N, int64_t L, float* y,
                         void* workspace, size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_scan_backward_params -- the parameter gradients of the causal DLR layer (Re cast): for a
 * loss whose gradient with respect to y is g [B, H, L] (u the layer's input), with
 * c_j = sum_b sum_k g_{b,k} u_{b,k-j}, S0 = sum_j c_j lambda^j, S1 = sum_j j c_j lambda^j
 * (DLR paper section 2, gradient analysis: d K_j / d W_n = lambda_n^j, d K_j / d lambda_n =
 * W_n j lambda_n^{j-1}; section 2.2: lambda = exp(-a^2 + i theta)):
 *   dW [H, N, 2] = (Re S0, -Im S0),  d_log_re [H, N] = -2 a Re(W S1),
 *   d_log_im [H, N] = -Im(W S1).
 * Two routes, chosen from N and L alone:
 *  - N >= 16 and L <= 65536: c itself by transforms, c = IFFT(sum_b FFT(g_b) conj FFT(u_b)):
 *    for L <= 8192 with both rows of a batch entry in one complex transform of
 *    M = 2^ceil(log2(2L - 1)) points, one CTA per channel; for longer rows through the
 *    spectrum and apply kernels of dlr_conv (the rows' spectra, their products summed over
 *    the batch, the inverse by applying that spectrum to an impulse); then S0 and S1 per state
 *    as sums over the lags with lambda^j = lambda^{32m} lambda^t, both factors evaluated
 *    directly from the parameters;
 *  - otherwise: sums over the steps of g against the states of two recurrences driven by u,
 *    x_k = lambda x_{k-1} + u_k and D_k = lambda (D_{k-1} + x_{k-1}) (lambda times
 *    dx/d lambda): S0 = sum g x, S1 = sum g D, per (b, h, state) with lambda as a float pair,
 *    then summed over the batch.
 * u, g [B, H, L] (4-byte aligned); parameters as in dlr_kernel; the three outputs (dW 8-byte
 * aligned) must not overlap the parameters or each other. workspace: device memory,
 * dlr_scan_backward_params_workspace_size(B, H, N, L) bytes, 16-byte aligned (the first
 * route: the M-point twiddle table and c [H, L] floats, for L > 8192 instead two dlr_conv
 * workspaces for B * H rows, one for H rows and an impulse buffer [H, L]; the second: 16 * B *
 * H * N; each part rounded up to 256 bytes). Two kernel launches (three on the first route); L < 2^24,
 * N <= 65536. The workspace size is 0 for arguments out of range. dlr_layer_backward gives
 * the same for the bidirectional layer and the DLR-prod cast, with the input gradient.
 */
size_t dlr_scan_backward_params_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L);
dlr_status dlr_scan_backward_params(const float* u, const float* g, const float* log_re,
                                    const float* log_im, const float* W, int64_t B, int64_t H,
                                    int64_t N, int64_t L, float* d_log_re, float* d_log_im,
                                    float* dW, void* workspace, size_t workspace_bytes,
                                    dlr_stream_t stream);

/*
 * dlr_layer_backward -- the gradients of the DLR layer as dlr_kernel + dlr_conv apply it:
 * causal or bidirectional (DLR paper section 2.1: y = DLR1(u) + rev(DLR2(rev(u))), the
 * second direction with the second parameter set), Re cast or DLR-prod cast (section 2.1:
 * kappa_j = Re K_j Im K_j), for a loss whose gradient with respect to y is g [B, H, L]:
 *  - du [B, H, L] (optional: NULL skips it): du_k = sum_j kappa1_j g_{k+j} + sum_j kappa2_j
 *    g_{k-j}, the layer's adjoint (the two directions swapped), by the FFT convolution of g
 *    with kappa2 as its causal and kappa1 as its anti-causal kernel (kappa2 = 0 for a causal
 *    layer);
 *  - the parameter gradients of each direction, from the lag correlation
 *    c_j = sum_b sum_k g_{b,k} u_{b,k-j} (the second direction uses c_{-j}, i.e. the causal
 *    layer on the reversed rows), with S0 = sum_j w_j lambda^j and S1 = sum_j j w_j lambda^j:
 *      Re cast (w = c):              dW = (Re S0, -Im S0), d_log_re = -2a Re(W S1),
 *                                    d_log_im = -Im(W S1);
 *      DLR-prod cast (w = c K, K the complex kernel, since d kappa_j = Im(K_j dK_j)):
 *                                    dW = (Im S0, Re S0),  d_log_re = -2a Im(W S1),
 *                                    d_log_im = Re(W S1).
 *    As dlr_scan_backward_params: c by transforms when N >= 16 (and always for the DLR-prod
 *    cast, which needs c itself), else the blocked recurrences (on the reversed rows for the
 *    second direction).
 * u, g, du 16-byte aligned; parameters as in dlr_kernel, the second set (and its three
 * outputs) given exactly when dir == DLR_BIDIR; outputs as dlr_scan_backward_params (none may
 * overlap a parameter, another output, u, g or the workspace). workspace: device memory,
 * dlr_layer_backward_workspace_size(B, H, N, L, dir, cast) bytes (0 for arguments out of
 * range), 16-byte aligned. Limits: L <= 65536, N <= 65536. Faults of the tensor-core kernel
 * generator's bounded
 * waits (N >= 256, or N >= 64 at L >= 16384) are reported through dlr_get_device_status().
 */
size_t dlr_layer_backward_workspace_size(int64_t B, int64_t H, int64_t N, int64_t L,
                                         dlr_dir dir, dlr_cast cast);
dlr_status dlr_layer_backward(const float* u, const float* g, const float* log_re,
                              const float* log_im, const float* W, const float* log_re2,
                              const float* log_im2, const float* W2, dlr_dir dir, dlr_cast cast,
                              int64_t B, int64_t H, int64_t N, int64_t L, float* du,
                              float* d_log_re, float* d_log_im, float* dW, float* d_log_re2,
                              float* d_log_im2, float* dW2, void* workspace,
                              size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_scan_backward_input -- the input gradient of the causal DLR layer (Re cast): for a loss
 * whose gradient with respect to y is g [B, H, L],
 *   du_k = sum_{j <= L-1-k} Re K_j g_{k+j},   K_j = sum_n W_n lambda_n^j,
 * i.e. the same layer run backwards in time on g (the layer is the causal convolution of u
 * with Re K, DLR paper section 2; its adjoint is the correlation with the same kernel).
 * Computed by the tensor-core scan's reversed pass with the layer's own parameters: du is
 * zeroed, the channel tables go to `workspace` (dlr_scan_workspace_size bytes, as dlr_scan)
 * and the reversed pass adds into du. g and du [B, H, L] must not overlap each other or the
 * workspace. Limits as the tensor-core path of dlr_scan (N <= 64). A memset and two kernel
 * launches; faults of the bounded waits are reported through dlr_get_device_status().
 */
dlr_status dlr_scan_backward_input(const float* g, const float* log_re, const float* log_im,
                                   const float* W, int64_t B, int64_t H, int64_t N, int64_t L,
                                   float* du, void* workspace, size_t workspace_bytes,
                                   dlr_stream_t stream);

/*
 * dlr_step_prepare + dlr_step -- the causal DLR layer (Re cast) advanced from a carried state,
 * the recurrent mode used to feed a sequence a few samples at a time ("The Annotated S4",
 * part 1 "An SSM Neural Network": the layer's RNN mode with its state cache; part 3 "Sampling
 * and Caching"):
 *   x_{n,t} = lambda_n x_{n,t-1} + u_t,   y_t = sum_n Re(W_n x_{n,t}),   t = 0 .. T-1,
 * with x_{n,-1} the state found in x on entry; on return x holds x_{n,T-1}. A zero x starts a
 * fresh sequence, and feeding a sequence in consecutive pieces gives the outputs of one
 * dlr_scan over the whole of it (DLR paper section 2, Eq. 1).
 * dlr_step_prepare evaluates lambda_n = exp(-(log_re)^2 + i log_im) of one parameter set
 * (log_re, log_im [H, N], W [H, N, 2]) in double precision and keeps it as a float pair, with
 * W, in `workspace` (device, >= dlr_step_workspace_size(H, N) bytes, 16-byte aligned).
 * dlr_step reads those tables (same H and N, earlier in stream order) and u [B, H, T],
 * updates x [B, H, N, 2] (float pairs, read and written) and writes y [B, H, T]. u, y, x and
 * the workspace must not overlap. T = 0 returns at once. Limits: N <= 256, T < 2^24. One
 * kernel launch each.
 */
size_t dlr_step_workspace_size(int64_t H, int64_t N);
dlr_status dlr_step_prepare(const float* log_re, const float* log_im, const float* W, int64_t H,
                            int64_t N, void* workspace, size_t workspace_bytes,
                            dlr_stream_t stream);
dlr_status dlr_step(const float* u, int64_t B, int64_t H, int64_t N, int64_t T, float* x,
                    float* y, const void* workspace, size_t workspace_bytes,
                    dlr_stream_t stream);

/*
 * s5_layer -- S5 SSM outputs (S5 paper section 3: diagonalised MIMO system; zero-order hold
 * with one timescale per state; diagonal feedthrough):
 *   Delta_p   = exp(log_delta[p])
 *   Lbar_p    = exp(Lambda_p Delta_p),   Bbar[p,:] = (Lbar_p - 1) / Lambda_p * Bt[p,:]
 *   x_k       = Lbar (.) x_{k-1} + Bbar u_k   (x_{-1} = 0)
 *   y_k       = Re(Ct x_k) + D (.) u_k
 * u, y: [B, L, H] float32. lambda: [P, 2]. log_delta: [P]. Bt: [P, H, 2]. Ct: [H, P, 2].
 * D: [H]. prec = DLR_FP32: float32 results throughout -- the two projections on tensor cores
 * as three tf32 products per float32 product (each operand split into its tf32 part and the
 * float32 remainder: hi*hi + hi*lo + lo*hi, float32 accumulation; error near float32
 * rounding), the scan in float32 arithmetic. prec = DLR_BF16_TC: the two
 * projections on tensor cores with bfloat16 operands and float32 accumulation (u is read as
 * float32 and rounded to bfloat16 inside the kernel); the projected input and the states
 * between the projections are kept in bfloat16, the scan arithmetic is float32.
 * workspace: >= s5_workspace_size(B, L, H, P, prec) bytes. u and y must not overlap.
 * Limits: H % 32 == 0, P % 32 == 0, 32 <= H, P <= 1024. Faults of the tensor-core pipelines'
 * bounded waits are reported through dlr_get_device_status().
 */
size_t s5_workspace_size(int64_t B, int64_t L, int64_t H, int64_t P, dlr_prec prec);
dlr_status s5_layer(const float* u, const float* lambda, const float* log_delta,
                    const float* Bt, const float* Ct, const float* D, int64_t B, int64_t L,
                    int64_t H, int64_t P, dlr_prec prec, float* y, void* workspace,
                    size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_get_device_status -- synchronise `stream`, then read and clear the device status word
 * shared by all kernels of this library on the current device. Returns DLR_OK when no kernel
 * reported a fault since the last call, DLR_ERR_TIMEOUT when a bounded wait gave up, or
 * DLR_ERR_CUDA when the synchronisation itself failed.
 */
dlr_status dlr_get_device_status(dlr_stream_t stream);

/*
 * dlr_selftest_timeout -- exercises the device-side failure reporting without faulting the
 * GPU: one thread waits on a shared-memory barrier that nothing will ever complete, with a
 * wait limit of `limit_ms` milliseconds (1..2000), the same kind of bounded wait the
 * tensor-core pipelines use. When the limit runs out the kernel records DLR_ERR_TIMEOUT in the
 * device status word and returns normally, so the context stays usable; the next
 * dlr_get_device_status() reports DLR_ERR_TIMEOUT and clears it. Returns DLR_OK once launched.
 */
dlr_status dlr_selftest_timeout(int limit_ms, dlr_stream_t stream);

/*
 * The bounds-checked build. A library compiled with DLR_BOUNDS_CHECK checks the shared- and
 * global-memory indices of its kernels' accesses: an index outside its buffer skips the access,
 * records DLR_ERR_BOUNDS in the device status word (read by dlr_get_device_status) and the
 * first failing site. It computes the same results as the normal build, more slowly; it
 * stands in for a memory checker.
 *   dlr_bounds_checked()     1 in the checked build, 0 otherwise.
 *   dlr_bounds_site()        synchronise the device, return and clear the first failing site
 *                            (file number * 100000 + source line; 0: none, -1: CUDA error).
 *   dlr_selftest_bounds()    checked build: one kernel reads an element one past the end of a
 *                            32-element buffer through the check, which skips it; the next
 *                            dlr_get_device_status reports DLR_ERR_BOUNDS and dlr_bounds_site a
 *                            nonzero site. Normal build: DLR_ERR_UNSUPPORTED, nothing launched.
 */
int dlr_bounds_checked(void);
int dlr_bounds_site(void);
dlr_status dlr_selftest_bounds(dlr_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* dlr_status_string(dlr_status status);

/* The CUDA runtime's message for the last error that a call made on this host thread
 * reported as DLR_ERR_CUDA ("no error" if none). The string is static; do not free it. */
const char* dlr_last_cuda_error(void);

/*
 * s5_layer_ex -- s5_layer with a choice of discretisation. disc = DLR_DISC_ZOH is s5_layer;
 * disc = DLR_DISC_BILINEAR discretises each state by the bilinear transform ("The Annotated
 * S4", part 1: A_bar = (I - Delta/2 A)^-1 (I + Delta/2 A), B_bar = (I - Delta/2 A)^-1 Delta B;
 * for the diagonal system Lambda_bar = (1 + z/2) / (1 - z/2), B_bar = Delta / (1 - z/2) B~,
 * z = Lambda Delta, evaluated per state in double precision). Everything else, including both
 * precision tiers, limits and the workspace, as s5_layer.
 */
dlr_status s5_layer_ex(const float* u, const float* lambda, const float* log_delta,
                       const float* Bt, const float* Ct, const float* D, int64_t B, int64_t L,
                       int64_t H, int64_t P, dlr_prec prec, dlr_disc disc, float* y,
                       void* workspace, size_t workspace_bytes, dlr_stream_t stream);

/*
 * s5_layer_tv -- the S5 layer with a step that changes from step to step ("Simplified State
 * Space Layers for Sequence Modeling", section 2.2: a different A_bar at each step, for
 * irregularly sampled sequences; section 6.3). dt [B, L]: the gap before each observation
 * (dt > 0, in units of the base step); state p steps by Delta_p dt_{b,k} with a zero-order
 * hold: Lambda_bar = exp(Lambda_p Delta_p dt), B_bar = (Lambda_bar - 1) / Lambda_p B~_p,
 * x_k = Lambda_bar_k x_{k-1} + B_bar_k u_k, y_k = Re(C~ x_k) + D u_k. Float32 tier only; other
 * arguments, layouts and limits as s5_layer with DLR_FP32; workspace:
 * s5_layer_tv_workspace_size bytes (the float32 tier's). dt must not overlap y.
 */
size_t s5_layer_tv_workspace_size(int64_t B, int64_t L, int64_t H, int64_t P);
dlr_status s5_layer_tv(const float* u, const float* dt, const float* lambda,
                       const float* log_delta, const float* Bt, const float* Ct, const float* D,
                       int64_t B, int64_t L, int64_t H, int64_t P, float* y, void* workspace,
                       size_t workspace_bytes, dlr_stream_t stream);

/*
 * dlr_params_from_dss_exp -- DSS_exp as a DLR (DLR paper section 2: the continuous diagonal
 * state space x' = Lambda x + u, y = Re <W, x>, discretised by a zero-order hold over steps
 * Delta, is the DLR with lambda = exp(Delta Lambda) and the input scaling folded into W):
 *   log_re = sqrt(-Delta Re Lambda), log_im = Delta Im Lambda, W_out = W (exp(Delta Lambda) - 1) / Lambda.
 * Lambda [H, N, 2], W [H, N, 2] (8-byte aligned), log_delta [H] (one step per channel);
 * outputs log_re, log_im [H, N], W_out [H, N, 2] (8-byte aligned), not overlapping the inputs
 * or each other; all device pointers. Evaluated in double precision per (h, n). A state with
 * Re Lambda > 0 cannot be held by |lambda| <= 1: it is mapped to |lambda| = 1 and
 * DLR_ERR_INVALID_ARG is recorded in the device status (dlr_get_device_status).
 */
dlr_status dlr_params_from_dss_exp(const float* Lambda, const float* log_delta, const float* W,
                                   int64_t H, int64_t N, float* log_re, float* log_im,
                                   float* W_out, dlr_stream_t stream);

/*
 * dlr_log_re_from_reparam -- (log Lambda)_re for decay rates given by a reparameterisation
 * f(w) of the recurrent weights (the StableSSM discussion of lambda = f(w)): |lambda| =
 * exp(-f(w)), so log_re = sqrt(f(w)), with f = e^w (DLR_REPARAM_EXP), log(1 + e^w)
 * (DLR_REPARAM_SOFTPLUS) or 1 / (a w^2 + b) (DLR_REPARAM_BEST; a >= 0, b > 0, else
 * DLR_ERR_INVALID_ARG). w and log_re: `count` floats on the device (4-byte aligned).
 */
dlr_status dlr_log_re_from_reparam(const float* w, int64_t count, dlr_reparam kind, float a,
                                   float b, float* log_re, dlr_stream_t stream);

/* Library ABI version (incremented on any signature change or added entry point). */
int dlr_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DLR_H_ */
