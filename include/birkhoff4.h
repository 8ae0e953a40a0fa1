/*
 * birkhoff4.h -- C ABI of libbirkhoff4.so: the per-token 4x4 Birkhoff
 * projection on one NVIDIA GB300 (sm_103a).
 *
 * Source: "Accelerating the Birkhoff Projection for Manifold-Constrained
 * Hyper-Connections" (technical summary of arXiv 2606.07574; Spanish and
 * French renderings), cited below as [mHC sN]:
 *   s1    mHC projects each token's residual mixing matrix onto the Birkhoff
 *         polytope; current practice is Sinkhorn-Knopp with a small fixed
 *         iteration count (e.g. 20);
 *   s2    the projection is entropic optimal transport;
 *   s2.1  forward: Newton's method on the dual reduced to m-1 = 3 free
 *         variables, closed-form gradient and Hessian, rows shifted by their
 *         maximum before the softmax;
 *   s2.2  backward: implicit differentiation, the last Newton Hessian being
 *         the matrix of the linear system;
 *   s2.3  one kernel processes many 4x4 matrices in a batch.
 *
 * The operation.  A token is a logit matrix X in R^{4x4}.  Its projection is
 *   P = diag(e^a) exp(X) diag(e^b),   P 1 = 1,  P^T 1 = 1,
 * the unique doubly stochastic matrix of that form (entropic OT with
 * epsilon = 1 and unit marginals).  b is the column dual in natural-log
 * units, gauge b[3] = 0.  The backward pass maps an upstream gradient
 * G = dL/dP to dX = (dP/dX)^T G.
 *
 * Layout.  X, P, dP (= G) and dX are contiguous row-major [T,4,4] arrays in
 * device memory: element (t,i,j) at offset 16*t + 4*i + j (i = row,
 * j = column).  b is [T,4] float32, b[t][3] = 0.  fp32 arrays hold float;
 * bf16 arrays hold bfloat16 bit patterns (uint16_t).  All arithmetic is fp32;
 * bf16 inputs are widened exactly and bf16 outputs are rounded to nearest
 * even.
 *
 * Ownership and execution.  Every pointer is caller-owned device memory; the
 * library allocates nothing.  Work is enqueued on `stream` and runs
 * asynchronously; the caller synchronises.  Calls on different streams or
 * host threads are independent.  In-place use is allowed where noted: each
 * token is read completely before any of it is written.
 *
 * Errors.  Every entry point returns 0 (B4_OK) or a positive code:
 *   B4_EINVAL   a NULL pointer with T > 0, T < 0, a bad option, iters < 0;
 *   B4_ECUDA    a CUDA error while preparing or launching (no kernel ran, or
 *               the launch failed); birkhoff4_last_cuda_error() returns the
 *               cudaError_t value (the library links its own CUDA runtime,
 *               so the caller's cudaGetLastError does not see it);
 *   B4_ENOTIMPL not available in this build.
 * T = 0 returns B4_OK and launches nothing.  Arguments are checked on the
 * host before any CUDA call.  A base address that is not 16-byte aligned is
 * not an error: it selects a slower kernel with plain loads.  Kernels never
 * trap.  A token whose X holds a NaN or an infinity gets an all-NaN P (and
 * NaN b); other tokens are unaffected.  Not reaching the tolerance within the
 * iteration cap is not an error: P is the last iterate, and the _ex variant
 * can count such tokens.
 */
#ifndef BIRKHOFF4_H
#define BIRKHOFF4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BIRKHOFF4_VERSION 2

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *birkhoff4_stream_t;

enum birkhoff4_status {
    B4_OK = 0,
    B4_EINVAL = 1,
    B4_ECUDA = 2,
    B4_ENOTIMPL = 3,
    B4_ESCRATCH = 4 /* request larger than the static scratch (see below) */
};

enum birkhoff4_dtype {
    B4_F32 = 0,
    B4_BF16 = 1
};

/* How the Newton passes assign tokens to threads [mHC s2.3: a batched     */
/* per-token kernel; the mapping is the implementation's choice].  Every   */
/* schedule computes the same iteration; they differ in speed, and in the  */
/* last bits of slow tokens (see B4_SCHED_QUEUE) and, for LANES4, in the  */
/* rounding of sums taken in another order.                                */
enum birkhoff4_schedule {
    B4_SCHED_DEFAULT = 0, /* the measured fastest: B4_SCHED_QUEUE          */
    /* One thread per token; a warp solves its 32 tokens for at most 7     */
    /* evaluations (8 in the passes with a backward), parks the unsolved   */
    /* ones (dual, residual, index, count)                                 */
    /* in shared memory and solves them later in full warps of parked      */
    /* tokens, 2 evaluations per round, re-evaluating P in the log domain  */
    /* from X and the dual on each resume (which replaces the periodic     */
    /* log-domain refresh).  Needs 16-byte aligned arrays (else as LANE).  */
    B4_SCHED_QUEUE = 1,
    /* One thread per token from start to finish: a warp runs as long as   */
    /* its slowest token.                                                  */
    B4_SCHED_LANE = 2,
    /* Four lanes per token, one row each [mHC s2.3: a matrix spread over  */
    /* lanes, column sums by __shfl_xor_sync]: contiguous 16-byte loads    */
    /* and stores, column sums and Hessian weights as butterfly sums over  */
    /* the four lanes, the 3x3 solve repeated in each.  A warp waits for   */
    /* its slowest of 8 tokens.  fp32 forward only (B4_ENOTIMPL for bf16   */
    /* and for the fused pass); unaligned arrays run as LANE.              */
    B4_SCHED_LANES4 = 3
};

/* Options of birkhoff4_forward_ex and birkhoff4_forward_backward_ex.      */
/* Zero-initialise, then set fields.                                       */
typedef struct birkhoff4_opts {
    int32_t in_dtype;   /* B4_F32 or B4_BF16 (X) */
    int32_t out_dtype;  /* B4_F32 or B4_BF16 (P) */
    int32_t max_evals;  /* cap on evaluations of P per token, 1..1024; 0 = 48 */
    float tol;          /* stop at max_j |colsum_j(P) - 1| <= tol; 0 = 1e-6 */
    int32_t *evals_out; /* NULL or device [T]: evaluations used per token (the
                           log-domain re-evaluation on a resume is not one) */
    unsigned long long *nonconv_count; /* NULL or device counter: += tokens
                                          that stopped above tol */
    int32_t schedule;   /* a birkhoff4_schedule; 0 = B4_SCHED_DEFAULT */
} birkhoff4_opts;

/* ---------------------------------------------------------------------- */
/* Forward [mHC s2.1]: X -> P (and optionally b).                          */
/*                                                                        */
/* Per token: b starts from the column-mean estimate                       */
/* b_j = -(mean_i X_ij - mean_i X_i3); each evaluation forms the row       */
/* softmax of X + b (first in the log domain with every row shifted by its */
/* maximum, then by multiplicative updates of the previous P, evaluated    */
/* again in the log domain when a parked token resumes (B4_SCHED_QUEUE) or */
/* every 8 evaluations (B4_SCHED_LANE)); the gradient is colsum(P) - 1 and */
/* the Hessian sum_i diag(p_i) - p_i p_i^T restricted to columns 0..2; the */
/* 3x3 Newton system is solved by Laplacian elimination; the step is       */
/* clamped to 3 (natural-log units) in the max norm and, from the fifth    */
/* step on, damped by 1/(1+lambda) when the Newton decrement lambda        */
/* exceeds 1.  The loop stops when the residual                            */
/* max_j |colsum_j - 1| <= tol (1e-6), when it stagnates below 64*tol, or  */
/* after max_evals (48) evaluations.  P is the last evaluation (unit row   */
/* sums up to rounding).                                                   */
/*                                                                        */
/* X: [T,4,4] (read).  P: [T,4,4] (written; may equal X).  b: NULL or      */
/* [T,4] float32 (written).                                               */
/* ---------------------------------------------------------------------- */
int birkhoff4_forward(const float *X, float *P, float *b, int64_t T, birkhoff4_stream_t stream);
int birkhoff4_forward_bf16(const uint16_t *X, uint16_t *P, float *b, int64_t T,
                           birkhoff4_stream_t stream);
/* Any dtype pair (e.g. bf16 X -> fp32 P), tolerance, cap and statistics. */
int birkhoff4_forward_ex(const void *X, void *P, float *b, int64_t T, const birkhoff4_opts *opts,
                         birkhoff4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Backward [mHC s2.2]: (P, G) -> dX = (dP/dX)^T G, nothing unrolled.      */
/*                                                                        */
/* With D_kl = G_kl - sum_j p_kj G_kj, v_l = sum_k p_kl D_kl and lambda    */
/* the solution of H lambda = v (H = the dual Hessian at P, the matrix of  */
/* the last Newton step, lambda_3 = 0):                                    */
/*   dX_kq = p_kq (D_kq - sum_l p_kl (lambda_q - lambda_l)).               */
/* P is first rescaled to unit row sums (a bf16 P is off by up to 2^-8).   */
/* H is regularised by adding 1e-7 * max_e w_e to its edge weights w_e     */
/* (a relative change of 1e-7 on well-conditioned tokens; it bounds the    */
/* amplification of rounding on nearly one-hot P).                         */
/*                                                                        */
/* X: [T,4,4] or NULL; read only when P is NULL, in which case P is        */
/* recomputed from X by the forward iteration (nothing stored between the  */
/* passes).  P: [T,4,4] from birkhoff4_forward, or NULL.  dP: [T,4,4].     */
/* dX: [T,4,4] (written; may equal dP or P).                               */
/* ---------------------------------------------------------------------- */
int birkhoff4_backward(const float *X, const float *P, const float *dP, float *dX, int64_t T,
                       birkhoff4_stream_t stream);
int birkhoff4_backward_bf16(const uint16_t *X, const uint16_t *P, const uint16_t *dP,
                            uint16_t *dX, int64_t T, birkhoff4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Fused forward + backward [mHC s2.1, s2.2]: one pass reads X and dP and  */
/* writes P (if non-NULL) and dX, with the backward using the fp32 P held  */
/* in registers (the Hessian of the last Newton step reused directly).     */
/* ---------------------------------------------------------------------- */
int birkhoff4_forward_backward(const float *X, const float *dP, float *P, float *dX, int64_t T,
                               birkhoff4_stream_t stream);
int birkhoff4_forward_backward_bf16(const uint16_t *X, const uint16_t *dP, uint16_t *P,
                                    uint16_t *dX, int64_t T, birkhoff4_stream_t stream);
/* The fused pass with options: opts->in_dtype == opts->out_dtype gives    */
/* the dtype of X, dP, P and dX; tol, max_evals, the statistics and the    */
/* schedule as in birkhoff4_forward_ex.  P == NULL: dX only (P recomputed  */
/* in registers, nothing else written).                                    */
int birkhoff4_forward_backward_ex(const void *X, const void *dP, void *P, void *dX, int64_t T,
                                  const birkhoff4_opts *opts, birkhoff4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* General n x n tokens, 2 <= n <= 8 [mHC s2.1: the dual reduces to m-1    */
/* free variables for m columns; s2.2].  The same forward iteration (b     */
/* gauge b[n-1] = 0, tolerance 1e-6, cap 48) and backward as above, for    */
/* [T, n, n] row-major fp32 arrays (element (t,i,j) at n*n*t + n*i + j);  */
/* b: NULL or [T, n].  Tokens are staged through shared memory with plain  */
/* loads (n^2 * 4-byte rows are not all TMA-aligned); no alignment         */
/* requirement beyond 4 bytes.  In place (P == X, dX == dP) is allowed.    */
/* n outside 2..8 returns B4_EINVAL.                                       */
/* ---------------------------------------------------------------------- */
int birkhoff4_forward_nxn(const float *X, float *P, float *b, int32_t n, int64_t T,
                          birkhoff4_stream_t stream);
int birkhoff4_backward_nxn(const float *P, const float *dP, float *dX, int32_t n, int64_t T,
                           birkhoff4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Host-resident tokens [mHC s2.1, s2.2; batched as in s2.3]: forward and  */
/* backward of tokens that live in host memory, streamed through the GPU.  */
/*                                                                        */
/* X_h, dP_h: host [T,4,4] inputs; P_h (or NULL) and dX_h: host [T,4,4]    */
/* outputs; all of dtype `dtype` (B4_F32 or B4_BF16).  Pin them            */
/* (cudaHostAlloc / cudaHostRegister) for the copies to overlap.           */
/* workspace: caller-owned device memory of workspace_bytes, split into    */
/* nstreams slots of four token arrays of `chunk` tokens each, chunk =     */
/* workspace_bytes / (nstreams * 4 * row bytes) (64 B fp32, 32 B bf16);    */
/* it must hold at least one token per slot.  streams: nstreams (1..16)    */
/* caller-owned streams; chunk c runs on streams[c % nstreams]: copy in,   */
/* the fused forward+backward pass (P recomputed and not copied out when   */
/* P_h is NULL), copy out.  Copies of one stream overlap the kernels of    */
/* another.  Returns once everything is enqueued: synchronise every stream */
/* before reading the outputs or reusing the workspace.                    */
/* ---------------------------------------------------------------------- */
int birkhoff4_forward_backward_host(const void *X_h, const void *dP_h, void *P_h, void *dX_h,
                                    int64_t T, int32_t dtype, void *workspace,
                                    size_t workspace_bytes, const birkhoff4_stream_t *streams,
                                    int32_t nstreams);

/* ---------------------------------------------------------------------- */
/* The same host-streaming pass without any device allocation.  The pages  */
/* have no counterpart: this is a deployment variant for callers that      */
/* cannot allocate device memory -- code that must not call cudaMalloc     */
/* because it synchronises the device, code whose device memory is owned   */
/* by another framework's allocator, plugins or sandboxes where device     */
/* allocations are not allowed.                                            */
/*                                                                        */
/* Arguments and results as birkhoff4_forward_backward_host, except that   */
/* the staging area is a static device array of B4_STATIC_SCRATCH_BYTES    */
/* (32 MiB) inside the library.  chunk_tokens: tokens per chunk; 0 takes  */
/* the largest chunk that fits (32 MiB / (nstreams * 4 * row bytes), e.g.  */
/* 65536 fp32 tokens with 2 streams).  A chunk that does not fit returns   */
/* B4_ESCRATCH; T itself is not limited (the call loops over chunks).      */
/* Every stream must belong to the current device (else B4_EINVAL, before  */
/* anything is enqueued).                                                  */
/* First call on a device: it looks up the array's device address          */
/* (cudaGetSymbolAddress, with that device current).  With CUDA's lazy     */
/* module loading (the default) that lookup loads the library's module on  */
/* the device, which reserves the 32 MiB there and may synchronise the     */
/* device; the array then stays reserved until the process exits.  Make   */
/* one warm-up call before latency-critical work.  The address is cached   */
/* per device and CUDA context and looked                                  */
/* up again after a context change (cudaDeviceReset included).  Apart from */
/* that lookup the call only enqueues copies and kernels; it never calls   */
/* cudaMalloc, cudaFree or any other allocating routine.  Every call uses  */
/* the same array: calls whose work overlaps on the GPU (concurrent        */
/* streams, or a second call before the first call's streams have         */
/* finished) race on it, so order them (for example by reusing the same    */
/* streams).  Nothing in the array needs to start at zero: every staging   */
/* slot is filled by a copy before it is read.                             */
/* ---------------------------------------------------------------------- */
#define B4_STATIC_SCRATCH_BYTES (32ull << 20)
int birkhoff4_forward_backward_host_static(const void *X_h, const void *dP_h, void *P_h,
                                           void *dX_h, int64_t T, int32_t dtype,
                                           int64_t chunk_tokens,
                                           const birkhoff4_stream_t *streams, int32_t nstreams);

/* ---------------------------------------------------------------------- */
/* Host-resident tokens, zero copy [mHC s2.1, s2.2; batched as in s2.3]:   */
/* the fused forward + backward on tokens that stay in page-locked host    */
/* memory.  The kernel reads X and dP and writes P and dX over the host    */
/* link itself: no device buffer and no cudaMemcpy.  On a GPU whose host   */
/* memory is coherently attached (GB300: NVLink-C2C) the SMs' own loads    */
/* and stores can outrun the copy engines.  Same layouts and dtypes as     */
/* birkhoff4_forward_backward_host.  Every buffer must be host memory the */
/* device can address: page-locked and mapped (cudaHostAlloc /             */
/* cudaMallocHost, or cudaHostRegister with cudaHostRegisterMapped), or,   */
/* on systems where the GPU addresses all host memory (Grace-based GB300), */
/* any host memory.  If cudaHostGetDevicePointer refuses a buffer,         */
/* B4_EINVAL is returned (birkhoff4_last_cuda_error has the code) and      */
/* nothing runs.  P_h may be                                               */
/* NULL (P not written); in-place use (P_h == X_h, dX_h == dP_h) is        */
/* allowed.  Asynchronous on `stream`: the host must not touch the buffers */
/* until the stream has been synchronised.                                 */
/* ---------------------------------------------------------------------- */
int birkhoff4_forward_backward_mapped(const void *X_h, const void *dP_h, void *P_h, void *dX_h,
                                      int64_t T, int32_t dtype, birkhoff4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Reference: fixed-iteration Sinkhorn-Knopp [mHC s1], the scheme current  */
/* mHC uses (e.g. iters = 20), kept for the accuracy comparison.           */
/* Log domain, b = 0 start; one iteration is a row normalisation           */
/* a_i = -LSE_j(X_ij + b_j) followed by a column normalisation             */
/* b_j = -LSE_i(X_ij + a_i); P = exp(X + a 1^T + 1 b^T) after the last     */
/* iteration (iters = 0 gives exp(X)).                                     */
/* X: [T,4,4] (read).  P: [T,4,4] (written; may equal X).  iters >= 0.     */
/* ---------------------------------------------------------------------- */
int birkhoff4_sinkhorn(const float *X, float *P, int iters, int64_t T, birkhoff4_stream_t stream);
int birkhoff4_sinkhorn_bf16(const uint16_t *X, uint16_t *P, int iters, int64_t T,
                            birkhoff4_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Diagnostics.                                                           */
/* ---------------------------------------------------------------------- */
/* Message for a status code (static string, never NULL). */
const char *birkhoff4_strerror(int code);
/* BIRKHOFF4_VERSION of the loaded library. */
int birkhoff4_version(void);
/* cudaError_t value behind the last B4_ECUDA returned on this host thread
 * (0 if none). */
int birkhoff4_last_cuda_error(void);
/* Device-side fault latch of the current device.  Kernels wait on their   */
/* own TMA transfers with a time limit (2 s); a wait that runs out sets    */
/* bit 0, the kernel drains what it issued and returns early (its tile     */
/* outputs are then incomplete).  Synchronises the device; writes the      */
/* latch to *out and clears it if `clear` is non-zero.                     */
int birkhoff4_device_status(unsigned int *out, int clear);
/* Self-test of that time limit: one CTA waits on a barrier nothing        */
/* completes, for limit_ns nanoseconds (1..10^9), then records bit 1 in    */
/* the latch and returns.  Synchronous.  Faults nothing.                   */
int birkhoff4_selftest_wait_timeout(int64_t limit_ns);
/* Microbenchmark of the ex2 (MUFU) rate: n_blocks CTAs of 256 threads run */
/* `iters` dependent-chain-free ex2.approx per thread; out[0] receives the */
/* elapsed device time in ms (measured with events on `stream`), out[1]    */
/* the number of ex2 executed.  Synchronous.                               */
int birkhoff4_mufu_probe(float *out_host, int n_blocks, int iters, birkhoff4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BIRKHOFF4_H */
