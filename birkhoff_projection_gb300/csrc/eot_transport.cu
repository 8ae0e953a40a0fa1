// eot_transport.cu -- the transport application of streaming entropic OT
// and the Hessian-vector product built on it ("FlashSinkhorn: IO-Aware
// Entropic OT on GPU", Methodik s3).  With the plan of given potentials,
// pi_ij = a_i b_j exp((f_i + g_j - ||x_i - y_j||^2)/eps), the kernel
// computes O = pi V for values V [m, dv] (V = Y gives pi Y) and the row
// masses r_i = sum_j pi_ij without storing pi, as two chained tensor-core
// products per key tile (attention form): S = Q K^T (TF32) into TMEM,
// P = 2^(S c1 + bias_j + rowterm_i) written by the epilogue warps back over
// S in TMEM, then O += P V^T into TMEM with P read from TMEM (f16, scaled)
// and V^T from shared memory.  Because the potential f fixes each row's
// normaliser, no running maximum is needed and O is never rescaled.  From
// O and r follow the gradient of the entropic OT cost with respect to X,
// 2 (r_i x_i - O_i), and the barycentric map O_i / r_i.
//
// Layout of this file: the kernel shapes and parameters; small packing,
// row-term, fix-up and CG kernels; transport_kernel (producer, MMA and
// epilogue roles, four modes); the host side (workspace layout, launches,
// plan_prepare / plan_apply, the HVP's conjugate gradients).  The extern
// "C" entries are declared and documented in eot_stream.h.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <vector>

#include "b4_device.cuh"
#include "b4_launch.cuh"
#include "eot_common.cuh"
#include "eot_device.cuh"
#include "eot_stream.h"

namespace b4 {
int record_cuda_error(cudaError_t e);              // birkhoff4_api.cu
unsigned int* device_fault_latch(cudaError_t* e);  // birkhoff4_api.cu
}  // namespace b4

namespace eot {
namespace tr {

constexpr int DV = 256;                    // value coordinates per launch, at most (O columns)
constexpr int NEPI = 8;                    // epilogue warps: NEPI / 4 per TMEM lane quarter
constexpr int NTHREADS = 64 + 32 * NEPI;   // + producer warp + MMA warp
constexpr int NBIAS = 4;                   // key-tile bias slots
constexpr int A_BYTES = BM * KC * 4;       // 16 KB: 128 query rows x 32 coordinates
constexpr int RING_BYTES = 200 * 1024;     // operand ring: Q/K chunks and value chunks
constexpr int NSLOT_MAX = 8;
constexpr int TMEM_COLS = 512;             // S / P buffers, then O
constexpr int NBUF_MAX = 2;
constexpr int GROUPS = NEPI / 4;           // key groups per tile (one per epilogue warp of a quarter)
constexpr int KEY_PAD = 768;               // key counts padded to a multiple of every tile width
constexpr int MAX_CTAS = 256;              // partial-result slots are sized for this many CTAs
static_assert(NEPI % 4 == 0, "whole lane quarters");

// What a launch computes:
//   VALUES  O = P V on the tensor cores (P from TMEM, V^T from shared memory);
//   MOMENT  the same with P weighted by S' = W Y^T (see transport_kernel);
//   VECTOR  one value column: o_i = sum_j p_ij v_j on the CUDA cores of the
//           epilogue, which leaves the tensor pipe to S alone;
//   HALF    VALUES with P and V as f16 operands (kind::f16, 16 keys per MMA
//           instead of 8): P scaled per row by 2^15 / a_i, V by one power of
//           two; a P entry past the f16 range sets a flag on which a VALUES
//           launch of the same slice redoes the work.
enum Mode : int { VALUES = 0, MOMENT = 1, VECTOR = 2, HALF = 3 };

// Shapes of one kernel instance: BN keys per tile; two S / P buffers for
// 192-key value tiles (slices of at most 128 columns: 2 x 192 + 128 TMEM
// columns) and for 256-key vector tiles (no O in TMEM), one for 256-key
// value tiles and for the moment form (which keeps S' beside S).  Each ring
// slot holds one K chunk of S (query and key coordinates) or a group of
// value chunks.
template <int BN_, int MODE>
struct Shape {
  static constexpr int BN = BN_;
  static constexpr int NBUF =
      ((BN_ == 192 && (MODE == VALUES || MODE == HALF)) || MODE == VECTOR) ? 2 : 1;
  static constexpr int NA = MODE == MOMENT ? 2 : 1;  // query operands per K chunk
  static constexpr int SLOT = NA * A_BYTES + BN * KC * 4;
  static constexpr int NSLOT = RING_BYTES / SLOT;
  static constexpr int CPT = BN / KC;          // 32-key chunks per tile
  static constexpr int CPG = CPT / GROUPS;     // chunks per epilogue warp
  static constexpr int VK = MODE == HALF ? 64 : KC;  // keys per value chunk (one 128-byte row)
  static constexpr int VPT = BN / VK;          // value chunks per tile
  static constexpr int O_COL = MODE == MOMENT ? 2 * BN : NBUF * BN;
  static constexpr int MAX_DV = MODE == VECTOR ? 1 : TMEM_COLS - O_COL;
  static constexpr int SMEM = NSLOT * SLOT + 1024;
  static_assert(NSLOT >= 3 && NSLOT <= NSLOT_MAX, "ring depth");
  static_assert(CPT % GROUPS == 0, "whole chunks per epilogue warp");
  static_assert(O_COL <= TMEM_COLS && (MODE == VECTOR || MAX_DV >= 128), "O columns");
  static_assert(SLOT % 1024 == 0, "slots keep the 1024-byte swizzle alignment");
  static_assert(SMEM + 2 * NBIAS * BN * 4 + 4096 <= 227 * 1024, "shared memory");
};

struct Params {
  CUtensorMap qmap;      // query points [nq_pad, d_pad], box {32, 128}
  CUtensorMap kmap;      // key points [nk_pad, d_pad], box {32, BN}
  CUtensorMap vmap;      // key points transposed [d_pad, nk_pad], box {32 keys, dv}
  CUtensorMap wmap;      // moment form: the query directions [nq_pad, d_pad], box {32, 128}
  const float* kbias;    // [nk_pad] (g_j - ||y_j||^2) log2(e)/eps + log2 b_j; -inf past nk
  const float* rowterm;  // [nq_pad] (f_i - ||x_i||^2) log2(e)/eps + log2 a_i; -inf past nq
  const float* kval;     // VECTOR: the value column [nk_pad], zero past nk
  const float* rowterm16;  // HALF: (f_i - ||x_i||^2) log2(e)/eps + 15: exponent of p_ij 2^15 / a_i
  const float* rowscale;   // HALF: a_i 2^-15, which takes a scaled p back to p
  const float* vscale;   // HALF: {s_V, 1 / s_V}, the power of two V was scaled by
  unsigned int* guard;   // HALF sets it when a scaled p leaves the f16 range
  int32_t guard_mode;    // 1: run only if *guard is set (the VALUES redo); 2: only if clear

  float* out;            // [nq, d]: columns v0 .. v0 + dv - 1 (those below d) written
  float* mass;           // [nq] row masses, or NULL
  float* part_o;         // [ctas][2][128][dv]: O of row blocks this CTA covers in part
  float* part_mass;      // [ctas][2][128]: their row masses
  int64_t nq;
  int32_t d, v0, dv;
  int32_t vg;            // value chunks per ring slot
  int32_t n_kt, n_kc;
  // Work of CTA b: first n_full whole row blocks b, b + ctas, ... (every
  // CTA sweeps the same key tiles at about the same time, so they share
  // them in L2); then the row blocks from full_rb on, whose tiles
  // T = (row block - full_rb) * n_kt + key tile are cut into one contiguous
  // run per CTA: t_base tiles, one more if b < t_rem.
  int64_t n_full, full_rb;
  int64_t t_base, t_rem;
  float c1;              // 2 log2(e) / eps
  unsigned int* fault;
};

// Whether a launch with this guard is to do nothing (uniform over the grid).
__device__ __forceinline__ bool guard_skips(const Params& p) {
  if (p.guard_mode == 0) return false;
  const unsigned int g = *reinterpret_cast<volatile unsigned int*>(p.guard);
  return p.guard_mode == 1 ? g == 0u : g != 0u;
}

// First tile and tile count of CTA b's run of the last row blocks.
__host__ __device__ __forceinline__ int64_t run_start(const Params& p, int64_t b) {
  return b * p.t_base + (b < p.t_rem ? b : p.t_rem);
}
__host__ __device__ __forceinline__ int64_t run_count(const Params& p, int64_t b) {
  return p.t_base + (b < p.t_rem ? 1 : 0);
}
// The CTA whose run holds tile T of the last row blocks.
__host__ __device__ __forceinline__ int64_t run_owner(const Params& p, int64_t T) {
  const int64_t cut = p.t_rem * (p.t_base + 1);
  return T < cut ? T / (p.t_base + 1) : p.t_rem + (T - cut) / p.t_base;
}
// The partial slot of CTA b that holds row block full_rb + tr (tr-th of
// the run's row blocks): 2b for the first row block of its run, 2b + 1 for
// its last.
__host__ __device__ __forceinline__ int64_t fixup_slot(const Params& p, int64_t b, int64_t tr) {
  return b * 2 + (run_start(p, b) / p.n_kt == tr ? 0 : 1);
}

// The tiles of CTA b in the order it processes them: its whole row blocks
// b, b + ctas, ... (n_full of them), then its run of the last row blocks.
// Each role of the kernel walks them with one of these; there is a
// division only where the run begins, not per tile.
struct TileWalk {
  int64_t u, rb, kt;  // local tile index, row block, key tile
  int64_t n_kt, u_run, t0, full_rb, ctas;
  __host__ __device__ TileWalk(const Params& p, int64_t b, int64_t ctas_)
      : u(0), rb(b), kt(0), n_kt(p.n_kt), u_run(p.n_full * p.n_kt), t0(run_start(p, b)),
        full_rb(p.full_rb), ctas(ctas_) {
    if (u_run == 0) run_begin();
  }
  __host__ __device__ void run_begin() {
    rb = full_rb + t0 / n_kt;
    kt = t0 % n_kt;
  }
  __host__ __device__ void advance() {
    ++u;
    if (u == u_run) {
      run_begin();
    } else if (++kt == n_kt) {
      kt = 0;
      rb += u < u_run ? ctas : 1;
    }
  }
};

// MMA instruction descriptor (kind::tf32, fp32 accumulation, both operands
// K-major) for M = 128 and a run-time N.
__device__ __forceinline__ uint32_t idesc_tf32_n(int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}
// The same for kind::f16 with A and B both f16 (format 0), fp32 accumulation.
__device__ __forceinline__ uint32_t idesc_f16_n(int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

// Transposed packing of the key points for the value operand:
// dst[k][j] = tf32(src[j][k]) for j < rows, k < d, zero elsewhere in
// [d_pad, rows_pad].  32 x 32 tiles through shared memory, both sides
// coalesced.
__global__ void pack_transposed_kernel(const float* __restrict__ src, int64_t rows, int32_t d,
                                       int64_t rows_pad, int32_t d_pad, float* __restrict__ dst) {
  __shared__ float t[32][33];
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int k0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t j = j0 + r;
    const int k = k0 + threadIdx.x;
    t[r][threadIdx.x] = (j < rows && k < d) ? tf32_rna(src[j * d + k]) : 0.0f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int k = k0 + r;
    const int64_t j = j0 + threadIdx.x;
    if (k < d_pad && j < rows_pad) dst[static_cast<int64_t>(k) * rows_pad + j] = t[threadIdx.x][r];
  }
}

// rowterm_i = (f_i - ||x_i||^2) log2(e)/eps + log2(a_i) for i < nq, -inf
// for the padding rows.
__global__ void rowterm_kernel(const float* __restrict__ f, const float* __restrict__ log_a,
                               const float* __restrict__ qnorm, int64_t nq, int64_t nq_pad,
                               float scale, float* __restrict__ rt) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nq_pad) return;
  rt[i] = i < nq ? fmaf(f[i] - qnorm[i], scale, log_a[i] * b4::LOG2E) : -INFINITY;
}

// HALF mode: rt16_i = (f_i - ||x_i||^2) log2(e)/eps + 15 and rsc_i =
// a_i 2^-15, so that 2^(S c1 + bias_j + rt16_i) = p_ij 2^15 / a_i; -inf and 0
// for the padding rows.
__global__ void rowterm16_kernel(const float* __restrict__ f, const float* __restrict__ log_a,
                                 const float* __restrict__ qnorm, int64_t nq, int64_t nq_pad,
                                 float scale, float* __restrict__ rt16, float* __restrict__ rsc) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nq_pad) return;
  rt16[i] = i < nq ? fmaf(f[i] - qnorm[i], scale, 15.0f) : -INFINITY;
  rsc[i] = i < nq ? exp2f(fmaf(log_a[i], b4::LOG2E, -15.0f)) : 0.0f;
}

// max |V| over the whole array, as the bits of a non-negative float
// (ordered like the values), into *vmax (zeroed by the caller).
__global__ void vmax_kernel(const float* __restrict__ V, int64_t total, unsigned int* __restrict__ vmax) {
  __shared__ unsigned int sh;
  if (threadIdx.x == 0) sh = 0u;
  __syncthreads();
  unsigned int m = 0u;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float a = fabsf(V[e]);
    const unsigned int b = a != a ? 0x7f800000u : __float_as_uint(a);  // NaN counts as inf
    m = b > m ? b : m;
  }
  atomicMax(&sh, m);
  __syncthreads();
  if (threadIdx.x == 0) atomicMax(vmax, sh);
}

// The power of two s_V that puts max |V| in [2^14, 2^15) (1 for V = 0):
// vscale = {s_V, 1 / s_V}, both exact.  A non-finite V sets the guard, so
// the f16 pass is redone in TF32 (where it gives what TF32 gives).
__global__ void vscale_kernel(const unsigned int* __restrict__ vmax, float* __restrict__ vscale,
                              unsigned int* __restrict__ guard) {
  const float m = __uint_as_float(*vmax);
  int e = 0;
  if (!(m <= 3.0e38f)) {
    *guard = 1u;
  } else if (m > 0.0f) {
    frexpf(m, &e);  // m in [2^(e-1), 2^e)
    e = e < -100 ? -100 : e;
  } else {
    e = 15;
  }
  vscale[0] = ldexpf(1.0f, 15 - e);
  vscale[1] = ldexpf(1.0f, e - 15);
}

// f16 transposed packing of s_V V (the HALF value operand):
// dst[k][j] = f16(s_V src[j][k]), zero padded to [d_pad, rows_pad].
__global__ void pack_transposed_f16_kernel(const float* __restrict__ src, int64_t rows, int32_t d,
                                           int64_t rows_pad, int32_t d_pad,
                                           const float* __restrict__ vscale, __half* __restrict__ dst) {
  __shared__ float t[32][33];
  const float sv = vscale[0];
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int k0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t j = j0 + r;
    const int k = k0 + threadIdx.x;
    t[r][threadIdx.x] = (j < rows && k < d) ? src[j * d + k] * sv : 0.0f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int k = k0 + r;
    const int64_t j = j0 + threadIdx.x;
    if (k < d_pad && j < rows_pad) dst[static_cast<int64_t>(k) * rows_pad + j] = __float2half_rn(t[threadIdx.x][r]);
  }
}

// grad_ik = 2 (r_i x_ik - (pi Y)_ik).
__global__ void grad_kernel(const float* __restrict__ X, const float* __restrict__ PY,
                            const float* __restrict__ mass, int64_t n, int32_t d,
                            float* __restrict__ grad) {
  const int64_t total = n * d;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    grad[e] = 2.0f * fmaf(mass[e / d], X[e], -PY[e]);
}

// Row blocks whose key tiles were split between CTAs: the sum of the
// partial O (and row masses) those CTAs left in their slots, in CTA order
// (deterministic).  Grid: x = row block of the runs, y = 1024-element part
// of its 128 x dv partial O (y = 0 also sums the masses); blocks that one
// CTA covered whole were written by the transport kernel and are skipped.
constexpr int kFixupElems = 1024;
__global__ void fixup_kernel(const __grid_constant__ Params p) {
  if (guard_skips(p)) return;
  __shared__ int64_t base[MAX_CTAS];          // first partial row of each contributing CTA
  const int64_t rb = p.full_rb + blockIdx.x;  // a row block of the runs
  const int64_t tr = blockIdx.x;                // its index among them
  const int64_t b_lo = run_owner(p, tr * p.n_kt), b_hi = run_owner(p, tr * p.n_kt + p.n_kt - 1);
  if (b_lo == b_hi) return;
  const int nb = static_cast<int>(b_hi - b_lo + 1);  // at most the CTA count
  // slot 0 holds the first row block of a CTA's run, slot 1 its last
  for (int k = threadIdx.x; k < nb; k += blockDim.x) {
    const int64_t b = b_lo + k;
    base[k] = fixup_slot(p, b, tr) * BM;
  }
  __syncthreads();
  const int dv = p.dv;
  const int e1 = min(BM * dv, static_cast<int>(blockIdx.y + 1) * kFixupElems);
  for (int e = blockIdx.y * kFixupElems + threadIdx.x; e < e1; e += blockDim.x) {
    const int row = e / dv, c = e - row * dv;
    float acc = 0.0f;
    for (int k = 0; k < nb; ++k) acc += p.part_o[(base[k] + row) * dv + c];
    const int64_t r = rb * BM + row;
    if (r < p.nq && p.v0 + c < p.d) p.out[r * p.d + p.v0 + c] = acc;
  }
  if (p.mass != nullptr && blockIdx.y == 0) {
    for (int row = threadIdx.x; row < BM; row += blockDim.x) {
      float acc = 0.0f;
      for (int k = 0; k < nb; ++k) acc += p.part_mass[base[k] + row];
      const int64_t r = rb * BM + row;
      if (r < p.nq) p.mass[r] = acc;
    }
  }
}

// ---------------------------------------------------------------------------
// Hessian-vector product helpers (one thread per row / element)
// ---------------------------------------------------------------------------
// xv_i = x_i . v_i;  r_i = 2 (a_i xv_i - (pi Y)_i . v_i);  W_i = [xv_i, v_i]
__global__ void hvp_prep_kernel(const float* __restrict__ X, const float* __restrict__ V,
                                const float* __restrict__ PY, const float* __restrict__ log_a,
                                int64_t n, int32_t d, float* __restrict__ xv, float* __restrict__ r,
                                float* __restrict__ W) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float sx = 0.0f, sp = 0.0f;
  for (int k = 0; k < d; ++k) {
    const float v = V[i * d + k];
    sx = fmaf(X[i * d + k], v, sx);
    sp = fmaf(PY[i * d + k], v, sp);
    W[i * (d + 1) + 1 + k] = v;
  }
  xv[i] = sx;
  W[i * (d + 1)] = sx;
  r[i] = 2.0f * fmaf(__expf(log_a[i]), sx, -sp);
}

// c_j = 2 ((pi^T xv)_j - y_j . (pi^T V)_j) from Mr = pi^T [xv, V]
__global__ void hvp_col_kernel(const float* __restrict__ Y, const float* __restrict__ Mr,
                               int64_t m, int32_t d, float* __restrict__ c) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= m) return;
  float s = 0.0f;
  for (int k = 0; k < d; ++k) s = fmaf(Y[j * d + k], Mr[j * (d + 1) + 1 + k], s);
  c[j] = 2.0f * (Mr[j * (d + 1)] - s);
}

// U_j = [dg_j, dg_j y_j]
__global__ void hvp_values_kernel(const float* __restrict__ Y, const float* __restrict__ dg, int64_t m,
                                  int32_t d, float* __restrict__ U) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= m) return;
  U[j * (d + 1)] = dg[j];
  for (int k = 0; k < d; ++k) U[j * (d + 1) + 1 + k] = dg[j] * Y[j * d + k];
}

// (H v)_ik = 2 a_i v_ik - (2/eps) (df_i PY_ik + G2_i,1+k - 2 xv_i PY_ik + 2 MV_ik)
__global__ void hvp_final_kernel(const float* __restrict__ V, const float* __restrict__ PY,
                                 const float* __restrict__ xv, const float* __restrict__ df,
                                 const float* __restrict__ G2, const float* __restrict__ MV,
                                 const float* __restrict__ log_a, int64_t n, int32_t d,
                                 float two_over_eps, float* __restrict__ out) {
  const int64_t total = n * d;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / d;
    const int64_t k = e - i * d;
    const float t = fmaf(df[i] - 2.0f * xv[i], PY[e], G2[i * (d + 1) + 1 + k] + 2.0f * MV[e]);
    out[e] = fmaf(2.0f * __expf(log_a[i]), V[e], -two_over_eps * t);
  }
}

// Conjugate gradients on [[diag(a), pi], [pi^T, diag(b)]] z = rhs, with the
// diagonal as preconditioner; vectors are [n | m] concatenated.  Dot products
// reduce in two fixed passes (deterministic), scalars stay on the device.
constexpr int kDotBlocks = 256;
__global__ void dot_partial_kernel(const float* __restrict__ x, const float* __restrict__ y,
                                   int64_t N, double* __restrict__ part) {
  __shared__ double sh[256];
  double acc = 0.0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < N;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    acc += static_cast<double>(x[i]) * static_cast<double>(y[i]);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = sh[0];
}
__global__ void dot_final_kernel(const double* __restrict__ part, double* __restrict__ out) {
  __shared__ double sh[kDotBlocks];
  sh[threadIdx.x] = part[threadIdx.x];
  __syncthreads();
  for (int o = kDotBlocks / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = sh[0];
}
// Ap = diag * p + [pi p2 ; pi^T p1] (the two products already in Pp)
__global__ void cg_matvec_kernel(const float* __restrict__ diag, const float* __restrict__ p,
                                 const float* __restrict__ Pp, int64_t N, float* __restrict__ Ap) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < N) Ap[i] = fmaf(diag[i], p[i], Pp[i]);
}
// The two plan products of a step are computed separately and each carries
// the rounding of its scores, so the operator CG sees is symmetric only to
// about 1e-3: the residual r^T D^-1 r levels off near 1e-8 of its first
// value and, iterated further, grows again.  So the iteration stops (alpha =
// beta = 0 from then on) once r^T D^-1 r is 1e-8 of its first value or has
// risen 1e4-fold above the smallest value seen, and the iterate with the
// smallest value is the one returned.
constexpr double kCgRelTol2 = 1e-8;
constexpr double kCgRise = 1e4;
__device__ __forceinline__ bool cg_live(const double* rs, const double* rs0, const double* best) {
  return *rs > 1e-300 && *rs > kCgRelTol2 * *rs0 && *rs <= kCgRise * *best;
}
// z += alpha p, res -= alpha Ap, s = res / diag; alpha = rs / pAp (0 once
// the iteration has stopped)
__global__ void cg_step_kernel(const double* __restrict__ rs, const double* __restrict__ pAp,
                               const double* __restrict__ rs0, const double* __restrict__ best,
                               const float* __restrict__ p,
                               const float* __restrict__ Ap, const float* __restrict__ diag,
                               int64_t N, float* __restrict__ z, float* __restrict__ res,
                               float* __restrict__ sv) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const double den = *pAp;
  const float alpha =
      (den > 1e-300 && cg_live(rs, rs0, best)) ? static_cast<float>(*rs / den) : 0.0f;
  z[i] = fmaf(alpha, p[i], z[i]);
  res[i] = fmaf(-alpha, Ap[i], res[i]);
  sv[i] = res[i] / diag[i];
}
// p = s + beta p, beta = rs_new / rs
__global__ void cg_dir_kernel(const double* __restrict__ rs, const double* __restrict__ rs_new,
                              const double* __restrict__ rs0, const double* __restrict__ best,
                              const float* __restrict__ sv, int64_t N, float* __restrict__ p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const float beta = (cg_live(rs, rs0, best) && cg_live(rs_new, rs0, best))
                         ? static_cast<float>(*rs_new / *rs)
                         : 0.0f;
  p[i] = fmaf(beta, p[i], sv[i]);
}
// One thread: keep = (rs < best), and best = min(best, rs).
__global__ void cg_best_kernel(const double* __restrict__ rs, double* __restrict__ best,
                               double* __restrict__ keep) {
  const bool b = *rs < *best;
  *keep = b ? 1.0 : 0.0;
  if (b) *best = *rs;
}
// stop = 1 once the iteration has stopped (the next step's alpha is 0), so
// that the next step's plan products need not be computed.
__global__ void cg_stop_kernel(const double* __restrict__ rs, const double* __restrict__ rs0,
                               const double* __restrict__ best, unsigned int* __restrict__ stop) {
  *stop = cg_live(rs, rs0, best) ? 0u : 1u;
}
// zb = z where the iterate just made is the best so far.
__global__ void cg_keep_kernel(const double* __restrict__ keep, const float* __restrict__ z,
                               int64_t N, float* __restrict__ zb) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < N && *keep != 0.0) zb[i] = z[i];
}
__global__ void copy_scalar_kernel(const double* __restrict__ src, double* __restrict__ dst) {
  *dst = *src;
}
// Partial sums of z . n0 with n0 = (1 on the first n entries, -1 on the
// rest): the direction along which (df, dg) leave pi's perturbation, and so
// H v, unchanged (df_i + dg_j is what enters).
__global__ void null_partial_kernel(const float* __restrict__ z, int64_t n, int64_t N,
                                    double* __restrict__ part) {
  __shared__ double sh[256];
  double acc = 0.0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < N;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    acc += i < n ? static_cast<double>(z[i]) : -static_cast<double>(z[i]);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = sh[0];
}
// z -= (z . n0 / N) n0: the drift CG accumulates along n0 is removed, so
// the final combination does not cancel large equal and opposite offsets.
__global__ void null_remove_kernel(const double* __restrict__ zn, int64_t n, int64_t N,
                                   float* __restrict__ z) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const float c = static_cast<float>(*zn / static_cast<double>(N));
  z[i] -= i < n ? c : -c;
}
// z = zb = 0, res = rhs, s = res / diag, p = s; diag = [a ; b]
__global__ void cg_init_kernel(const float* __restrict__ rhs, const float* __restrict__ log_a,
                               const float* __restrict__ log_b, int64_t n, int64_t N,
                               float* __restrict__ diag, float* __restrict__ z,
                               float* __restrict__ zb, float* __restrict__ res,
                               float* __restrict__ sv, float* __restrict__ p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const float dg = __expf(i < n ? log_a[i] : log_b[i - n]);
  diag[i] = dg;
  z[i] = 0.0f;
  zb[i] = 0.0f;
  res[i] = rhs[i];
  sv[i] = rhs[i] / dg;
  p[i] = sv[i];
}

// p = 2^(acc c1 + bias_j + rt) for one 32-key chunk of a row, in place over
// the accumulator bits; returns the chunk's sum.
__device__ __forceinline__ float p_chunk(uint32_t (&v)[32], const float4* kb, float c1, float rt) {
  const float2 cc = make_float2(c1, c1);
  const float2 rr = make_float2(rt, rt);
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 b = kb[i];
    float2 s0 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])),
                           cc, __fadd2_rn(make_float2(b.x, b.y), rr));
    float2 s1 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                           cc, __fadd2_rn(make_float2(b.z, b.w), rr));
    s0.x = b4::ex2(s0.x);
    s0.y = b4::ex2(s0.y);
    s1.x = b4::ex2(s1.x);
    s1.y = b4::ex2(s1.y);
    acc[(2 * i) & 3] = __fadd2_rn(acc[(2 * i) & 3], s0);
    acc[(2 * i + 1) & 3] = __fadd2_rn(acc[(2 * i + 1) & 3], s1);
    v[4 * i] = __float_as_uint(s0.x);
    v[4 * i + 1] = __float_as_uint(s0.y);
    v[4 * i + 2] = __float_as_uint(s1.x);
    v[4 * i + 3] = __float_as_uint(s1.y);
  }
  const float2 t = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return t.x + t.y;
}

// One CTA per SM.  CTA b first takes whole row blocks b, b + G, ... (all
// CTAs sweep the same key tiles together and share them in L2), then an
// equal contiguous run of the remaining tiles T = row block * n_kt + key
// tile, so that the last wave is full (TileWalk).  A CTA's tiles of one row
// block form a segment; a segment that is not the whole row block leaves
// its O and row masses in the CTA's partial slots for fixup_kernel.  Warp
// roles:
//   0      producer (lane 0): per tile the key biases (bulk copy, a ring of
//          their own), and the operand ring in the order the MMA thread
//          reads it: the K chunks of S(T) (query and key coordinates) and
//          the value chunks of P V(T), vg chunks per slot;
//   1      TMEM owner and MMA issuer (lane 0): S(T) into S / P buffer
//          T % NBUF; O += P(T) V(T)^T with P(T) read from that buffer, which
//          is released when those MMAs complete.  With two buffers S(T) is
//          issued before P V(T - 1), so the epilogue of one tile overlaps the
//          products of its neighbours; with one, P V(T - 1) goes first;
//   2..9   epilogue: thread t of warp w owns query row 32 (w % 4) + t and key
//          group (w - 2) / 4 (BN / 2 keys of each tile): p = 2^(S c1 + bias +
//          rowterm) stored over its S columns in TMEM (as f16 pairs over
//          their first half in the HALF mode), the row mass, and at the end
//          of a segment its chunks of O.
// HALF: VALUES with the f16 second product (scales and overflow flag: see
// Mode).
// MOMENT: the second-moment form used by the Hessian-vector product: with a
// direction w_i per query, the weights become pi_ij (w_i . y_j), so O_i =
// sum_j pi_ij (w_i . y_j) y_j.  A second MMA per K chunk (the packed
// directions as A, the same key tile as B) writes S' = W Y^T beside S, and
// the epilogue multiplies.
// VECTOR: a single value column.  The producer copies each tile's values
// beside its biases, the MMA thread issues S alone, and the epilogue forms
// o_i = sum_j p_ij v_j in registers and releases the S buffer itself.
template <int BN_, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1) transport_kernel(const __grid_constant__ Params p) {
  using C = Shape<BN_, MODE>;
  constexpr bool MOMENT = MODE == tr::MOMENT;
  constexpr bool VEC = MODE == VECTOR;
  constexpr bool H16 = MODE == HALF;
  constexpr int VK = C::VK;
  constexpr int VPT = C::VPT;
  // the VALUES redo of a HALF launch runs only if that launch overflowed;
  // guard_mode 2 skips a launch whose flag is set (a finished CG)
  if (guard_skips(p)) return;
  constexpr int BN = C::BN;
  constexpr int NBUF = C::NBUF;
  constexpr int SLOT = C::SLOT;
  constexpr int NSLOT = C::NSLOT;
  constexpr int CPG = C::CPG;
  constexpr uint32_t O_COL = C::O_COL;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t slot_full[NSLOT_MAX], slot_empty[NSLOT_MAX];
  // p_full is per S / P buffer: one barrier shared by all tiles could see
  // the epilogue complete tile T + 1's phase before the MMA thread had
  // observed tile T's, and the parity wait would then miss it.  Per buffer,
  // the next arrival needs S(T + NBUF), which the MMA thread issues only
  // after it has consumed tile T's phase.
  __shared__ uint64_t acc_full[NBUF_MAX], acc_empty[NBUF_MAX], p_full[NBUF_MAX];
  __shared__ uint64_t o_full, o_empty, mma_done;
  __shared__ uint64_t bias_full[NBIAS], bias_empty[NBIAS];
  __shared__ __align__(16) float bias_sm[NBIAS][BN];
  __shared__ __align__(16) float val_sm[VEC ? NBIAS : 1][VEC ? BN : 4];
  __shared__ float mass_sh[GROUPS > 1 ? GROUPS - 1 : 1][BM];
  __shared__ float vec_sh[VEC && GROUPS > 1 ? GROUPS - 1 : 1][VEC ? BM : 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_kt = p.n_kt;
  const int64_t u_run = p.n_full * n_kt;  // local index of this CTA's first run tile
  const int64_t cnt = u_run + run_count(p, blockIdx.x);
  const TileWalk walk0(p, blockIdx.x, gridDim.x);  // this CTA's first tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      b4::mbar_init(&slot_full[s], 1);
      b4::mbar_init(&slot_empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      b4::mbar_init(&acc_full[b], 1);
      b4::mbar_init(&acc_empty[b], VEC ? NEPI : 1);  // VECTOR: released by the epilogue warps
      b4::mbar_init(&p_full[b], NEPI);
    }
    for (int b = 0; b < NBIAS; ++b) {
      b4::mbar_init(&bias_full[b], 1);
      b4::mbar_init(&bias_empty[b], NEPI);
    }
    b4::mbar_init(&o_full, 1);
    b4::mbar_init(&o_empty, NEPI);
    b4::mbar_init(&mma_done, 1);
    abort_sh = 0;
    b4::mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    b4::prefetch_tmap(&p.qmap);
    b4::prefetch_tmap(&p.kmap);
    b4::prefetch_tmap(&p.vmap);
    if (MOMENT) b4::prefetch_tmap(&p.wmap);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t vbytes = static_cast<uint32_t>(p.dv) * KC * 4;
  const int vg = p.vg;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      uint32_t it = 0, nb = 0;  // ring slots and bias slots filled
      TileWalk cs = walk0, cv = walk0;  // the tiles of S loads and of value loads
      // the K chunks of S(u), after the biases of tile u
      auto load_s = [&](int64_t u) -> bool {
        const int64_t rb = cs.rb, kt = cs.kt;
        cs.advance();
        const int bs = static_cast<int>(u % NBIAS);
        if (!wait_bar(&bias_empty[bs], (static_cast<uint32_t>(u / NBIAS) & 1u) ^ 1u, abort_flag,
                      p.fault))
          return false;
        b4::mbar_arrive_expect_tx(&bias_full[bs], (VEC ? 2 : 1) * BN * 4);
        bulk_load_1d(bias_sm[bs], p.kbias + static_cast<int64_t>(kt) * BN, BN * 4, &bias_full[bs]);
        if (VEC)
          bulk_load_1d(val_sm[bs], p.kval + static_cast<int64_t>(kt) * BN, BN * 4, &bias_full[bs]);
        ++nb;
        for (int kc = 0; kc < p.n_kc; ++kc, ++it) {
          const int s = static_cast<int>(it % NSLOT);
          if (!wait_bar(&slot_empty[s], ((it / NSLOT) & 1u) ^ 1u, abort_flag, p.fault)) return false;
          unsigned char* st = ring + s * SLOT;
          b4::mbar_arrive_expect_tx(&slot_full[s], SLOT);
          const int qy = static_cast<int>(rb * BM), ky = static_cast<int>(kt * BN);
          b4::tma_load_2d(st, &p.qmap, &slot_full[s], kc * KC, qy);
          if (MOMENT) b4::tma_load_2d(st + A_BYTES, &p.wmap, &slot_full[s], kc * KC, qy);
          b4::tma_load_2d(st + C::NA * A_BYTES, &p.kmap, &slot_full[s], kc * KC, ky);
        }
        return true;
      };
      // the value chunks of P V(u), vg per slot (u in order)
      auto load_v = [&](int64_t) -> bool {
        const int64_t kt = cv.kt;
        cv.advance();
        for (int c = 0; c < VPT; c += vg, ++it) {
          const int s = static_cast<int>(it % NSLOT);
          if (!wait_bar(&slot_empty[s], ((it / NSLOT) & 1u) ^ 1u, abort_flag, p.fault)) return false;
          unsigned char* st = ring + s * SLOT;
          b4::mbar_arrive_expect_tx(&slot_full[s], static_cast<uint32_t>(vg) * vbytes);
          for (int g = 0; g < vg; ++g)
            b4::tma_load_2d(st + g * vbytes, &p.vmap, &slot_full[s],
                            static_cast<int>(kt * BN) + (c + g) * VK, p.v0);
        }
        return true;
      };
      bool ok = true;
      for (int64_t k = 0; k <= cnt && ok; ++k) {
        if (VEC) {
          if (k < cnt) ok = load_s(k);
        } else if (NBUF == 1) {
          if (k > 0) ok = load_v(k - 1);
          if (ok && k < cnt) ok = load_s(k);
        } else {
          if (k < cnt) ok = load_s(k);
          if (ok && k > 0) ok = load_v(k - 1);
        }
      }
      // every issued copy lands before the CTA may exit
      for (uint32_t j = it > static_cast<uint32_t>(NSLOT) ? it - NSLOT : 0u; j < it; ++j)
        b4::mbar_wait(&slot_full[j % NSLOT], (j / NSLOT) & 1u, kWaitLimitNs);
      for (uint32_t j = nb > static_cast<uint32_t>(NBIAS) ? nb - NBIAS : 0u; j < nb; ++j)
        b4::mbar_wait(&bias_full[j % NBIAS], (j / NBIAS) & 1u, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_tf32_n(BN);
      const uint32_t id_o = H16 ? idesc_f16_n(p.dv) : idesc_tf32_n(p.dv);
      uint32_t it = 0;   // ring slots consumed
      uint32_t seg = 0;  // segments (runs of one row block) begun
      // S(T) = Q K^T into buffer u % NBUF, once that buffer's P has been used
      auto issue_s = [&](int64_t u) -> bool {
        const int buf = static_cast<int>(u % NBUF);
        const uint32_t use = static_cast<uint32_t>(u / NBUF);
        if (!wait_bar(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.fault)) return false;
        tc_fence_after();
        const uint32_t d_s = tmem + static_cast<uint32_t>(buf * BN);
        for (int kc = 0; kc < p.n_kc; ++kc, ++it) {
          const int s = static_cast<int>(it % NSLOT);
          if (!wait_bar(&slot_full[s], (it / NSLOT) & 1u, abort_flag, p.fault)) return false;
          tc_fence_after();
          const uint32_t a = b4::smem_addr(ring + s * SLOT);
          const uint64_t da = desc_sw128_kmajor(a), db = desc_sw128_kmajor(a + C::NA * A_BYTES);
#pragma unroll
          for (int kk = 0; kk < KC / KSTEP; ++kk) {
            const uint64_t adv = static_cast<uint64_t>(kk * KSTEP * 4 / 16);
            mma_tf32(d_s, da + adv, db + adv, id_s, (kc | kk) != 0);
            if (MOMENT)  // S' = W Y^T into the columns after S
              mma_tf32(d_s + BN, desc_sw128_kmajor(a + A_BYTES) + adv, db + adv, id_s,
                       (kc | kk) != 0);
          }
          mma_commit(&slot_empty[s]);
        }
        mma_commit(&acc_full[buf]);
        return true;
      };
      // O += P(u) V(u)^T with P(u) read from its TMEM buffer (u in order)
      TileWalk cp = walk0;
      auto issue_pv = [&](int64_t u) -> bool {
        const int64_t kt = cp.kt;
        cp.advance();
        const bool first = kt == 0 || u == 0 || u == u_run, last = kt == n_kt - 1 || u == cnt - 1;
        if (first && !wait_bar(&o_empty, (seg & 1u) ^ 1u, abort_flag, p.fault)) return false;
        const int buf = static_cast<int>(u % NBUF);
        if (!wait_bar(&p_full[buf], static_cast<uint32_t>(u / NBUF) & 1u, abort_flag, p.fault))
          return false;
        tc_fence_after();
        for (int c = 0; c < VPT; c += vg, ++it) {
          const int s = static_cast<int>(it % NSLOT);
          if (!wait_bar(&slot_full[s], (it / NSLOT) & 1u, abort_flag, p.fault)) return false;
          tc_fence_after();
          for (int g = 0; g < vg; ++g) {
            const uint64_t dvd = desc_sw128_kmajor(b4::smem_addr(ring + s * SLOT + g * vbytes));
            if (H16) {
              // 16 keys per MMA; P of key k sits in its epilogue group's
              // columns, two keys per column
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const int k0 = (c + g) * 64 + kk * 16;
                const int gk = (k0 / (CPG * KC)) * CPG * KC;  // first key of its group
                const uint32_t pa = tmem + static_cast<uint32_t>(buf * BN + gk + (k0 - gk) / 2);
                mma_f16_ts(tmem + O_COL, pa, dvd + static_cast<uint64_t>(kk * 2), id_o,
                           !(first && c + g == 0 && kk == 0));
              }
            } else {
              const uint32_t pa = tmem + static_cast<uint32_t>(buf * BN + (c + g) * KC);
#pragma unroll
              for (int kk = 0; kk < KC / KSTEP; ++kk) {
                const uint64_t adv = static_cast<uint64_t>(kk * KSTEP * 4 / 16);
                mma_tf32_ts(tmem + O_COL, pa + static_cast<uint32_t>(kk * KSTEP), dvd + adv, id_o,
                            !(first && c + g == 0 && kk == 0));
              }
            }
          }
          mma_commit(&slot_empty[s]);
        }
        mma_commit(&acc_empty[buf]);  // the S / P buffer is free once these MMAs are done
        if (last) {
          mma_commit(&o_full);
          ++seg;
        }
        return true;
      };
      bool ok = true;
      for (int64_t k = 0; k <= cnt && ok; ++k) {
        if (VEC) {
          if (k < cnt) ok = issue_s(k);
        } else if (NBUF == 1) {
          if (k > 0) ok = issue_pv(k - 1);
          if (ok && k < cnt) ok = issue_s(k);
        } else {
          if (k < cnt) ok = issue_s(k);
          if (ok && k > 0) ok = issue_pv(k - 1);
        }
      }
      // all MMAs issued by this thread complete before TMEM is released
      mma_commit(&mma_done);
      b4::mbar_wait(&mma_done, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t sg = 0;  // segments finished
    int64_t r = 0, kt0 = 0;
    float rt = 0.0f, mass = 0.0f, ov = 0.0f;  // ov: VECTOR's sum_j p_ij v_j
    float rsc = 1.0f;                         // HALF: a_i 2^-15 (scaled p -> p)
    bool ok = true;
    TileWalk ce = walk0;
    for (int64_t u = 0; u < cnt; ++u, ce.advance()) {
      const int64_t rb = ce.rb, kt = ce.kt;
      if (u == 0 || kt == 0 || u == u_run) {  // a segment begins
        r = rb * BM + row;
        rt = H16 ? p.rowterm16[r] : p.rowterm[r];
        if (H16) rsc = p.rowscale[r];
        mass = 0.0f;
        ov = 0.0f;
        kt0 = kt;
      }
      const int buf = static_cast<int>(u % NBUF);
      const int bs = static_cast<int>(u % NBIAS);
      ok = wait_bar(&acc_full[buf], static_cast<uint32_t>(u / NBUF) & 1u, abort_flag, p.fault) &&
           wait_bar(&bias_full[bs], static_cast<uint32_t>(u / NBIAS) & 1u, abort_flag, p.fault);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        // this warp's CPG chunks: the next chunk's TMEM load overlaps the
        // current one's arithmetic; P is stored over S in place
        const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(buf * BN + grp * CPG * KC);
        const float4* kb = reinterpret_cast<const float4*>(&bias_sm[bs][grp * CPG * KC]);
        uint32_t v[32], w[32];
        bool big = false;  // HALF: a chunk of scaled p reached the f16 range
        tmem_ld32(taddr, v);
        tmem_wait32(v);
#pragma unroll
        for (int ch = 0; ch < CPG; ++ch) {
          if (ch + 1 < CPG) tmem_ld32(taddr + static_cast<uint32_t>((ch + 1) * KC), w);
          const float csum = p_chunk(v, kb + ch * 8, p.c1, rt);
          mass += csum;
          if (H16) {  // P as f16 pairs over the first half of this group's S columns
            big = big || !(csum < 65504.0f);
            uint32_t h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const __half2 x = __floats2half2_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
              h[i] = *reinterpret_cast<const uint32_t*>(&x);
            }
            tmem_st16(tmem + lane_base + static_cast<uint32_t>(buf * BN + grp * CPG * KC + ch * 16), h);
          }
          if (VEC) {  // the value column on the CUDA cores; S is not written back
            const float4* vv = reinterpret_cast<const float4*>(&val_sm[bs][(grp * CPG + ch) * KC]);
            float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = vv[i];
              a0 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])),
                              make_float2(x.x, x.y), a0);
              a1 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                              make_float2(x.z, x.w), a1);
            }
            const float2 a = __fadd2_rn(a0, a1);
            ov += a.x + a.y;
          }
          if (MOMENT) {  // weight pi_ij (w_i . y_j): S' sits BN columns after S
            uint32_t sp[32];
            tmem_ld32(taddr + static_cast<uint32_t>(BN + ch * KC), sp);
            tmem_wait32(sp);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = __float_as_uint(__uint_as_float(v[i]) * __uint_as_float(sp[i]));
          }
          if (!VEC && !H16) tmem_st32(taddr + static_cast<uint32_t>(ch * KC), v);
          if (ch + 1 < CPG) {
            tmem_wait32(w);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = w[i];
          }
        }
        if (H16 && __any_sync(0xffffffffu, big) && lane == 0) atomicOr(p.guard, 1u);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(VEC ? &acc_empty[buf] : &p_full[buf]);
          mbar_arrive(&bias_empty[bs]);
        }
      }
      // end of a segment (or a failed wait): O and the row masses.  Every
      // epilogue warp reaches the two named barriers below once per segment,
      // or once more when it gives up, so none waits for a warp that left.
      if (!ok || kt == n_kt - 1 || u == cnt - 1) {
        const bool whole = kt0 == 0 && kt == n_kt - 1;  // the segment is the whole row block
        // partial segments lie in the run: its first uses slot 0, its last slot 1
        const int64_t pslot =
            static_cast<int64_t>(blockIdx.x) * 2 + (sg == static_cast<uint32_t>(p.n_full) ? 0 : 1);
        if (ok && !VEC) {
          ok = wait_bar(&o_full, sg & 1u, abort_flag, p.fault);
          ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && !VEC) {
          tc_fence_after();
          for (int c = grp; c * KC < p.dv; c += GROUPS) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + O_COL + static_cast<uint32_t>(c * KC), o);
            tmem_wait32(o);
            if (H16) {  // undo the scales of p (a_i 2^-15) and of V (1 / s_V)
              const float sc = rsc * p.vscale[1];
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * sc);
            }
            if (whole) {
              if (r < p.nq) {
                float* orow = p.out + r * p.d;
                const int c0 = p.v0 + c * KC;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (c0 + i < p.d) orow[c0 + i] = __uint_as_float(o[i]);
              }
            } else {
              float4* prow = reinterpret_cast<float4*>(p.part_o + (pslot * BM + row) * p.dv + c * KC);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                prow[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                      __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_empty);
        }
        // row masses (and VECTOR's o_i): the key groups of a row
        if (H16) mass *= rsc;
        if (grp > 0) {
          mass_sh[grp - 1][row] = mass;
          if (VEC) vec_sh[grp - 1][row] = ov;
        }
        named_bar_sync(1, 32 * NEPI);
        if (grp == 0 && ok && !*abort_flag) {
          if (p.mass != nullptr) {
            float m = mass;
#pragma unroll
            for (int g = 0; g < GROUPS - 1; ++g) m += mass_sh[g][row];
            if (!whole)
              p.part_mass[pslot * BM + row] = m;
            else if (r < p.nq)
              p.mass[r] = m;
          }
          if (VEC) {
            float o = ov;
#pragma unroll
            for (int g = 0; g < GROUPS - 1; ++g) o += vec_sh[g][row];
            if (!whole)
              p.part_o[pslot * BM + row] = o;
            else if (r < p.nq)
              p.out[r * p.d + p.v0] = o;
          }
        }
        named_bar_sync(1, 32 * NEPI);
        ++sg;
        if (*abort_flag || !ok) break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace tr

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct TrLayout {
  int64_t n_pad, m_pad, n_rb, ctas;
  int32_t d_pad, v_pad;
  // byte offsets (yt: the values, transposed; po, pm: partial O and masses;
  // yh, rt16, rsc, misc: the f16 values, scaled row terms, row scales and
  // {max |V|, guard, s_V, 1 / s_V} of the HALF mode)
  size_t x, y, yt, xn, yn, kb, rt, wq, wn, po, pm, yh, rt16, rsc, misc, total;
};

// moment: also room for the packed query directions (wq) and their norms
TrLayout tr_layout(int64_t n, int64_t m, int32_t d, int32_t dv, bool moment = false) {
  TrLayout L;
  L.n_pad = round_up(std::max<int64_t>(n, 1), ROW_PAD);
  L.m_pad = round_up(std::max<int64_t>(m, 1), tr::KEY_PAD);
  L.n_rb = L.n_pad / BM;
  L.d_pad = static_cast<int32_t>(round_up(d, KC));
  L.v_pad = static_cast<int32_t>(round_up(dv, KC));
  // partial slots for at most one CTA per 128-key tile (the narrowest tiles)
  L.ctas = std::min<int64_t>(tr::MAX_CTAS, L.n_rb * (L.m_pad / 128));
  const int64_t dvs = std::min<int64_t>(tr::DV, L.v_pad);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_bytes(bytes);
    return at;
  };
  L.x = take(static_cast<size_t>(L.n_pad) * L.d_pad * 4);
  L.y = take(static_cast<size_t>(L.m_pad) * L.d_pad * 4);
  L.yt = take(static_cast<size_t>(L.m_pad) * L.v_pad * 4);
  L.xn = take(static_cast<size_t>(L.n_pad) * 4);
  L.yn = take(static_cast<size_t>(L.m_pad) * 4);
  L.kb = take(static_cast<size_t>(L.m_pad) * 4);
  L.rt = take(static_cast<size_t>(L.n_pad) * 4);
  L.wq = L.wn = 0;
  if (moment) {
    L.wq = take(static_cast<size_t>(L.n_pad) * L.d_pad * 4);
    L.wn = take(static_cast<size_t>(L.n_pad) * 4);
  }
  L.po = take(static_cast<size_t>(L.ctas) * 2 * BM * dvs * 4);
  L.pm = take(static_cast<size_t>(L.ctas) * 2 * BM * 4);
  L.yh = take(static_cast<size_t>(L.m_pad) * L.v_pad * 2);
  L.rt16 = take(static_cast<size_t>(L.n_pad) * 4);
  L.rsc = take(static_cast<size_t>(L.n_pad) * 4);
  L.misc = take(64);
  L.total = o;
  return L;
}

bool tr_sizes_ok(int64_t n, int64_t m, int32_t d, int32_t dv) {
  return n >= 0 && m >= 0 && n <= kMaxPoints && m <= kMaxPoints && d >= 1 && d <= 16384 &&
         dv >= 1 && dv <= 16384;
}

// The work split of n_rb row blocks of n_kt key tiles over `ctas` CTAs:
// whole waves of row blocks first (one per CTA), the rest in equal runs.
void make_schedule(tr::Params& p, int64_t n_rb, int64_t n_kt, int64_t ctas) {
  p.n_kt = static_cast<int32_t>(n_kt);
  p.n_full = n_rb / ctas;
  p.full_rb = p.n_full * ctas;
  const int64_t run_tiles = (n_rb - p.full_rb) * n_kt;
  p.t_base = run_tiles / ctas;
  p.t_rem = run_tiles % ctas;
}

// One launch of transport_kernel<BN, MODE> for the value slice in p
// (v0, dv), then the fix-up of the row blocks that were split between CTAs.
template <int BN, int MODE>
cudaError_t launch_shape(tr::Params& p, const TrLayout& L, const float* yp, int dev, int nsm,
                         cudaStream_t stream) {
  using C = tr::Shape<BN, MODE>;
  static std::atomic<int> attr_done[64];
  if (dev >= 64 || attr_done[dev].load(std::memory_order_acquire) == 0) {
    const cudaError_t err = cudaFuncSetAttribute(tr::transport_kernel<BN, MODE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    if (dev < 64) attr_done[dev].store(1, std::memory_order_release);
  }
  if (p.dv > C::MAX_DV || !encode_rows128(&p.kmap, yp, L.m_pad, L.d_pad, BN))
    return cudaErrorInvalidValue;
  // value chunks per ring slot: the largest divisor of the chunks per tile
  // that fits (a chunk is one 128-byte row per value coordinate)
  const int vbytes = p.dv * 128;
  p.vg = 1;
  for (int g = C::VPT; g >= 1; --g)
    if (C::VPT % g == 0 && g * vbytes <= C::SLOT) {
      p.vg = g;
      break;
    }
  const int64_t n_kt = L.m_pad / BN;
  const int64_t ctas = std::min<int64_t>(std::min<int64_t>(nsm, L.n_rb * n_kt), L.ctas);
  make_schedule(p, L.n_rb, n_kt, ctas);
  tr::transport_kernel<BN, MODE><<<static_cast<unsigned>(ctas), tr::NTHREADS, C::SMEM, stream>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || L.n_rb == p.full_rb) return err;
  const dim3 fgrid(static_cast<unsigned>(L.n_rb - p.full_rb),
                   static_cast<unsigned>((BM * p.dv + tr::kFixupElems - 1) / tr::kFixupElems));
  tr::fixup_kernel<<<fgrid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// Key-tile shape of a slice: 192-key tiles with two S / P buffers when the
// slice has at most 128 value columns (the epilogue of one tile overlaps the
// products of the next), else 256-key tiles with one; the moment form keeps
// S' beside S in 128-key tiles.  A single value column goes to the CUDA
// cores (VECTOR, 256-key tiles, two S buffers): as a tensor product it
// would cost as many MMA instructions per tile as 64 columns.
// Tensor map of the value operand: rows v0 .. v0 + dv - 1 of the transposed
// values [v_pad, m_pad] (fp32, or f16 for the HALF mode), boxes of one
// 128-byte row of keys per value coordinate.
bool encode_values(CUtensorMap* map, const void* base, const TrLayout& L, int32_t v_pad,
                   int32_t dv, bool half) {
  b4::EncodeTiledFn fn = b4::encode_fn();
  if (fn == nullptr) return false;
  const int esize = half ? 2 : 4;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.m_pad), static_cast<cuuint64_t>(v_pad)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.m_pad) * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(dv)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_transport(const tr::Params& base, const TrLayout& L, int32_t v_pad,
                             const float* yp, const float* yt, const void* yh, int32_t v0,
                             int32_t dv, float* mass, bool moment, cudaStream_t stream,
                             unsigned int* skip = nullptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int nsm = b4::sm_count(dev);
  if (nsm <= 0) return cudaErrorInvalidDevice;
  tr::Params p = base;
  if (!encode_values(&p.vmap, yt, L, v_pad, dv, false)) return cudaErrorInvalidValue;
  p.v0 = v0;
  p.dv = dv;
  p.mass = mass;
  p.guard_mode = 0;
  if (moment) return launch_shape<128, tr::MOMENT>(p, L, yp, dev, nsm, stream);
  if (base.d == 1) {
    p.dv = 1;
    p.kval = yt;  // row 0 of the transposed values: v_j, zero past m
    if (skip != nullptr) {  // nothing to do once *skip is set
      p.guard = skip;
      p.guard_mode = 2;
    }
    return launch_shape<256, tr::VECTOR>(p, L, yp, dev, nsm, stream);
  }
  // f16 operands for P V, then the TF32 redo that runs only if they overflowed
  tr::Params h = p;
  if (!encode_values(&h.vmap, yh, L, v_pad, dv, true)) return cudaErrorInvalidValue;
  p.guard_mode = 1;
  if (dv <= 128) {
    err = launch_shape<192, tr::HALF>(h, L, yp, dev, nsm, stream);
    return err != cudaSuccess ? err : launch_shape<192, tr::VALUES>(p, L, yp, dev, nsm, stream);
  }
  err = launch_shape<256, tr::HALF>(h, L, yp, dev, nsm, stream);
  return err != cudaSuccess ? err : launch_shape<256, tr::VALUES>(p, L, yp, dev, nsm, stream);
}

// The plan of given potentials between queries Q and keys K, prepared once
// (packed points, key biases, row terms, the query tensor map) and then
// applied to any values V [nk, dv <= dv_max] by plan_apply.
struct Plan {
  TrLayout L;
  tr::Params p;        // all but the value slice and the output
  const float* yp;     // the packed keys
  unsigned char* w;    // the plan's workspace region (tr_layout(...).total bytes)
  int64_t nk;
  bool moment;
};

// Arguments are checked by the callers.  Wd != NULL: the moment form, with
// directions Wd [nq, d].
cudaError_t plan_prepare(const float* Xq, const float* Xk, const float* fq, const float* gk,
                         const float* log_q, const float* log_k, int64_t nq, int64_t nk, int32_t d,
                         int32_t dv_max, float eps, const float* Wd, unsigned char* w,
                         unsigned int* fault, cudaStream_t s, Plan* P) {
  const bool moment = Wd != nullptr;
  const TrLayout L = tr_layout(nq, nk, d, dv_max, moment);
  P->L = L;
  P->w = w;
  P->nk = nk;
  P->moment = moment;
  float* xp = reinterpret_cast<float*>(w + L.x);
  float* yp = reinterpret_cast<float*>(w + L.y);
  float* xn = reinterpret_cast<float*>(w + L.xn);
  float* yn = reinterpret_cast<float*>(w + L.yn);
  float* kb = reinterpret_cast<float*>(w + L.kb);
  float* rt = reinterpret_cast<float*>(w + L.rt);
  P->yp = yp;
  const float scale = static_cast<float>(1.4426950408889634 / eps);
  const unsigned rgrid = static_cast<unsigned>((L.n_pad + 255) / 256);
  cudaError_t e = pack(Xq, nq, d, L.n_pad, L.d_pad, xp, nullptr, xn, s);
  if (e == cudaSuccess) e = pack(Xk, nk, d, L.m_pad, L.d_pad, yp, nullptr, yn, s);
  float* wq = moment ? reinterpret_cast<float*>(w + L.wq) : nullptr;
  if (e == cudaSuccess && moment)
    e = pack(Wd, nq, d, L.n_pad, L.d_pad, wq, nullptr, reinterpret_cast<float*>(w + L.wn), s);
  if (e == cudaSuccess) e = bias(gk, log_k, yn, nk, L.m_pad, eps, kb, s);
  if (e == cudaSuccess) {
    tr::rowterm_kernel<<<rgrid, 256, 0, s>>>(fq, log_q, xn, nq, L.n_pad, scale, rt);
    if (!moment && dv_max > 1)
      tr::rowterm16_kernel<<<rgrid, 256, 0, s>>>(fq, log_q, xn, nq, L.n_pad, scale,
                                                 reinterpret_cast<float*>(w + L.rt16),
                                                 reinterpret_cast<float*>(w + L.rsc));
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  tr::Params& p = P->p;
  if (!encode_rows128(&p.qmap, xp, L.n_pad, L.d_pad, BM) ||
      (moment && !encode_rows128(&p.wmap, wq, L.n_pad, L.d_pad, BM)))
    return cudaErrorInvalidValue;
  if (!moment) p.wmap = p.qmap;
  unsigned int* misc = reinterpret_cast<unsigned int*>(w + L.misc);  // vmax, guard, s_V, 1/s_V
  p.kbias = kb;
  p.rowterm = rt;
  p.kval = nullptr;
  p.rowterm16 = reinterpret_cast<float*>(w + L.rt16);
  p.rowscale = reinterpret_cast<float*>(w + L.rsc);
  p.vscale = reinterpret_cast<float*>(misc + 2);
  p.guard = misc + 1;
  p.guard_mode = 0;
  p.out = nullptr;
  p.mass = nullptr;
  p.part_o = reinterpret_cast<float*>(w + L.po);
  p.part_mass = reinterpret_cast<float*>(w + L.pm);
  p.nq = nq;
  p.d = 0;
  p.n_kc = L.d_pad / KC;
  p.c1 = static_cast<float>(2.0 * 1.4426950408889634 / eps);
  p.fault = fault;
  return cudaSuccess;
}

// out [nq, dv] = pi V (weights pi_ij (w_i . y_j) for the moment form) and,
// if mass != NULL, mass = pi 1; V [nk, dv], 1 <= dv <= the plan's dv_max.
// skip (one value column only): a device flag; once it is set, the
// products are not computed and out keeps what it held.
cudaError_t plan_apply(const Plan& P, const float* V, int32_t dv, float* out, float* mass,
                       cudaStream_t s, unsigned int* skip = nullptr) {
  const TrLayout& L = P.L;
  unsigned char* w = P.w;
  const int32_t v_pad = static_cast<int32_t>(round_up(dv, KC));
  float* vt = reinterpret_cast<float*>(w + L.yt);
  const dim3 grid(static_cast<unsigned>(L.m_pad / 32), static_cast<unsigned>(v_pad / 32));
  tr::pack_transposed_kernel<<<grid, dim3(32, 8), 0, s>>>(V, P.nk, dv, L.m_pad, v_pad, vt);
  cudaError_t e = cudaGetLastError();
  // HALF operands (several value columns, not the moment form): the V scale
  // and the f16 values; the guard starts clear
  if (e == cudaSuccess && !P.moment && dv > 1) {
    unsigned int* misc = reinterpret_cast<unsigned int*>(w + L.misc);
    e = cudaMemsetAsync(misc, 0, 2 * sizeof(unsigned int), s);
    if (e == cudaSuccess) {
      const int64_t total = P.nk * static_cast<int64_t>(dv);
      const unsigned vb = static_cast<unsigned>(std::min<int64_t>((total + 255) / 256, 1024));
      tr::vmax_kernel<<<vb, 256, 0, s>>>(V, total, misc);
      tr::vscale_kernel<<<1, 1, 0, s>>>(misc, reinterpret_cast<float*>(misc + 2), misc + 1);
      tr::pack_transposed_f16_kernel<<<grid, dim3(32, 8), 0, s>>>(
          V, P.nk, dv, L.m_pad, v_pad, P.p.vscale, reinterpret_cast<__half*>(w + L.yh));
      e = cudaGetLastError();
    }
  }
  tr::Params p = P.p;
  p.out = out;
  p.d = dv;
  // one launch per slice of up to 256 value coordinates; the first also
  // writes the row masses
  for (int32_t v0 = 0; v0 < v_pad && e == cudaSuccess; v0 += tr::DV) {
    const int32_t w_slice = std::min<int32_t>(tr::DV, v_pad - v0);
    e = launch_transport(p, L, v_pad, P.yp, vt, w + L.yh, v0, w_slice, v0 == 0 ? mass : nullptr,
                         P.moment, s, dv == 1 ? skip : nullptr);
  }
  return e;
}

// The plan of (f, g) applied to the values V [m, dv]: out = pi V, mass =
// pi 1.  With directions Wd [n, d] (moment form) the weights are
// pi_ij (w_i . y_j) instead: out_i = sum_j pi_ij (w_i . y_j) v_j.
int apply_impl(const float* X, const float* Y, const float* f, const float* g, const float* log_a,
               const float* log_b, const float* V, int32_t dv, float* out, float* mass, int64_t n,
               int64_t m, int32_t d, float eps, void* workspace, size_t workspace_bytes,
               cudaStream_t s, const float* Wd = nullptr) {
  const bool moment = Wd != nullptr;
  if (!tr_sizes_ok(n, m, d, dv) || !(eps > 0.0f) || !std::isfinite(eps)) return B4_EINVAL;
  if (n == 0) return B4_OK;
  if (m == 0) return B4_EINVAL;
  if (X == nullptr || Y == nullptr || f == nullptr || g == nullptr || log_a == nullptr ||
      log_b == nullptr || V == nullptr || out == nullptr || mass == nullptr)
    return B4_EINVAL;
  const TrLayout L = tr_layout(n, m, d, dv, moment);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < L.total)
    return B4_EINVAL;
  cudaError_t e = cudaSuccess;
  unsigned int* fault = b4::device_fault_latch(&e);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  Plan P;
  e = plan_prepare(X, Y, f, g, log_a, log_b, n, m, d, dv, eps, Wd,
                   static_cast<unsigned char*>(workspace), fault, s, &P);
  if (e == cudaSuccess) e = plan_apply(P, V, dv, out, mass, s);
  return b4::record_cuda_error(e);
}

// Workspace of the Hessian-vector product: the plan of (f, g) with X as
// queries (fwd) and with Y as queries (rev; after CG, the moment form's
// plan), then the vectors.
struct HvpLayout {
  size_t fwd, rev, py, xv, rhs, w, mr, z, zb, res, sv, pv, ap, pp, diag, mass, u, g2, mv, part, scal,
      total;
};

HvpLayout hvp_layout(int64_t n, int64_t m, int32_t d) {
  HvpLayout H;
  const size_t fwd = tr_layout(n, m, d, d + 1).total;
  const size_t rev = std::max(tr_layout(m, n, d, d + 1).total, tr_layout(n, m, d, d, true).total);
  const size_t N = static_cast<size_t>(n + m);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_bytes(bytes);
    return at;
  };
  H.fwd = take(fwd);
  H.rev = take(rev);
  H.py = take(static_cast<size_t>(n) * d * 4);
  H.xv = take(static_cast<size_t>(n) * 4);
  H.rhs = take(N * 4);
  H.w = take(static_cast<size_t>(n) * (d + 1) * 4);
  H.mr = take(static_cast<size_t>(m) * (d + 1) * 4);
  H.z = take(N * 4);
  H.zb = take(N * 4);
  H.res = take(N * 4);
  H.sv = take(N * 4);
  H.pv = take(N * 4);
  H.ap = take(N * 4);
  H.pp = take(N * 4);
  H.diag = take(N * 4);
  H.mass = take(static_cast<size_t>(std::max(n, m)) * 4);
  H.u = take(static_cast<size_t>(m) * (d + 1) * 4);
  H.g2 = take(static_cast<size_t>(n) * (d + 1) * 4);
  H.mv = take(static_cast<size_t>(n) * d * 4);
  H.part = take(tr::kDotBlocks * sizeof(double));
  H.scal = take(8 * sizeof(double));
  H.total = o;
  return H;
}

// (H v) for the entropic OT cost at potentials (f, g): see eot_hvp.
int hvp_impl(const float* X, const float* Y, const float* f, const float* g, const float* log_a,
             const float* log_b, const float* V, float* out, int64_t n, int64_t m, int32_t d,
             float eps, int32_t cg_iters, void* workspace, size_t workspace_bytes, cudaStream_t s) {
  if (!tr_sizes_ok(n, m, d, d + 1) || !(eps > 0.0f) || !std::isfinite(eps) || cg_iters < 0 ||
      cg_iters > 100000)
    return B4_EINVAL;
  if (n == 0) return B4_OK;
  if (m == 0) return B4_EINVAL;
  if (X == nullptr || Y == nullptr || f == nullptr || g == nullptr || log_a == nullptr ||
      log_b == nullptr || V == nullptr || out == nullptr)
    return B4_EINVAL;
  const HvpLayout H = hvp_layout(n, m, d);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < H.total)
    return B4_EINVAL;
  unsigned char* w = static_cast<unsigned char*>(workspace);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(w + off); };
  const int64_t N = n + m;
  cudaError_t e = cudaSuccess;
  unsigned int* fault = b4::device_fault_latch(&e);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  float *PY = F(H.py), *xv = F(H.xv), *rhs = F(H.rhs), *W = F(H.w), *Mr = F(H.mr), *z = F(H.z);
  float *zb = F(H.zb), *res = F(H.res), *sv = F(H.sv), *pv = F(H.pv), *Ap = F(H.ap), *Pp = F(H.pp);
  float *diag = F(H.diag), *mass = F(H.mass), *U = F(H.u), *G2 = F(H.g2), *MV = F(H.mv);
  double* part = reinterpret_cast<double*>(w + H.part);
  // rs[2], pAp, rs0, z . n0, best, keep, and (as an unsigned int) the stop flag
  double* scal = reinterpret_cast<double*>(w + H.scal);
  unsigned int* stop = reinterpret_cast<unsigned int*>(scal + 7);
  const unsigned bn = static_cast<unsigned>((N + 255) / 256);
  const unsigned bq = static_cast<unsigned>((n + 255) / 256);
  const unsigned bk = static_cast<unsigned>((m + 255) / 256);
  auto dot = [&](const float* x, const float* y, double* outp) {
    tr::dot_partial_kernel<<<tr::kDotBlocks, 256, 0, s>>>(x, y, N, part);
    tr::dot_final_kernel<<<1, tr::kDotBlocks, 0, s>>>(part, outp);
    return cudaGetLastError();
  };
  // the plan in both directions, prepared once for every application below
  Plan fwd, rev;
  e = plan_prepare(X, Y, f, g, log_a, log_b, n, m, d, d + 1, eps, nullptr, w + H.fwd, fault, s, &fwd);
  if (e == cudaSuccess)
    e = plan_prepare(Y, X, g, f, log_b, log_a, m, n, d, d + 1, eps, nullptr, w + H.rev, fault, s, &rev);
  // pi Y, then r and the values [x.v, V]
  if (e == cudaSuccess) e = plan_apply(fwd, Y, d, PY, mass, s);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  tr::hvp_prep_kernel<<<bq, 256, 0, s>>>(X, V, PY, log_a, n, d, xv, rhs, W);
  // pi^T [x.v, V], then c
  if ((e = plan_apply(rev, W, d + 1, Mr, mass, s)) != cudaSuccess) return b4::record_cuda_error(e);
  tr::hvp_col_kernel<<<bk, 256, 0, s>>>(Y, Mr, m, d, rhs + n);
  // conjugate gradients for (df, dg)
  tr::cg_init_kernel<<<bn, 256, 0, s>>>(rhs, log_a, log_b, n, N, diag, z, zb, res, sv, pv);
  e = dot(res, sv, scal + 0);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  tr::copy_scalar_kernel<<<1, 1, 0, s>>>(scal + 0, scal + 3);
  tr::copy_scalar_kernel<<<1, 1, 0, s>>>(scal + 0, scal + 5);
  if ((e = cudaMemsetAsync(stop, 0, sizeof(double), s)) != cudaSuccess)
    return b4::record_cuda_error(e);
  for (int32_t k = 0; k < cg_iters; ++k) {
    double* rs = scal + (k & 1);
    double* rs_next = scal + ((k + 1) & 1);
    // once the iteration has stopped, the products are skipped on the device
    if ((e = plan_apply(fwd, pv + n, 1, Pp, nullptr, s, stop)) != cudaSuccess ||
        (e = plan_apply(rev, pv, 1, Pp + n, nullptr, s, stop)) != cudaSuccess)
      return b4::record_cuda_error(e);
    tr::cg_matvec_kernel<<<bn, 256, 0, s>>>(diag, pv, Pp, N, Ap);
    if ((e = dot(pv, Ap, scal + 2)) != cudaSuccess) return b4::record_cuda_error(e);
    tr::cg_step_kernel<<<bn, 256, 0, s>>>(rs, scal + 2, scal + 3, scal + 5, pv, Ap, diag, N, z,
                                          res, sv);
    if ((e = dot(res, sv, rs_next)) != cudaSuccess) return b4::record_cuda_error(e);
    tr::cg_best_kernel<<<1, 1, 0, s>>>(rs_next, scal + 5, scal + 6);
    tr::cg_stop_kernel<<<1, 1, 0, s>>>(rs_next, scal + 3, scal + 5, stop);
    tr::cg_keep_kernel<<<bn, 256, 0, s>>>(scal + 6, z, N, zb);
    tr::cg_dir_kernel<<<bn, 256, 0, s>>>(rs, rs_next, scal + 3, scal + 5, sv, N, pv);
  }
  // the best iterate, without its component along n0
  tr::null_partial_kernel<<<tr::kDotBlocks, 256, 0, s>>>(zb, n, N, part);
  tr::dot_final_kernel<<<1, tr::kDotBlocks, 0, s>>>(part, scal + 4);
  tr::null_remove_kernel<<<bn, 256, 0, s>>>(scal + 4, n, N, zb);
  // pi [dg, dg y], the second moment, and the combination
  tr::hvp_values_kernel<<<bk, 256, 0, s>>>(Y, zb + n, m, d, U);
  if ((e = plan_apply(fwd, U, d + 1, G2, nullptr, s)) != cudaSuccess) return b4::record_cuda_error(e);
  // the second moment: the moment form's plan in the region of rev (done)
  Plan mom;
  e = plan_prepare(X, Y, f, g, log_a, log_b, n, m, d, d, eps, V, w + H.rev, fault, s, &mom);
  if (e == cudaSuccess) e = plan_apply(mom, Y, d, MV, nullptr, s);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  const int64_t tot = n * static_cast<int64_t>(d);
  const int64_t blocks = std::min<int64_t>((tot + 255) / 256, 1 << 20);
  tr::hvp_final_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      V, PY, xv, zb, G2, MV, log_a, n, d, 2.0f / eps, out);
  return b4::record_cuda_error(cudaGetLastError());
}

}  // namespace
}  // namespace eot

extern "C" int eot_transport_schedule(int64_t n_rb, int32_t n_kt, int32_t ctas, int64_t* owner) {
  if (n_rb < 1 || n_kt < 1 || ctas < 1 || ctas > eot::tr::MAX_CTAS || n_rb > (int64_t(1) << 24) ||
      n_rb * n_kt < ctas || n_rb * n_kt > (int64_t(1) << 28))
    return B4_EINVAL;
  using eot::tr::Params;
  Params p{};
  eot::make_schedule(p, n_rb, n_kt, ctas);
  const int64_t W = n_rb * n_kt;
  std::vector<int64_t> own(static_cast<size_t>(W), -1), slot(static_cast<size_t>(W), -1);
  std::vector<int64_t> holder(static_cast<size_t>(2 * ctas), -1);  // row block in each slot
  int bad = 0;
  for (int64_t b = 0; b < ctas; ++b) {
    // the walk, segments and partial slots of transport_kernel's epilogue
    eot::tr::TileWalk w(p, b, ctas);
    const int64_t cnt = w.u_run + eot::tr::run_count(p, b);
    std::vector<int64_t> seg;
    int64_t kt0 = 0, sg = 0;
    for (int64_t u = 0; u < cnt; ++u, w.advance()) {
      if (u == 0 || w.kt == 0 || u == w.u_run) {
        seg.clear();
        kt0 = w.kt;
      }
      const int64_t T = w.rb * n_kt + w.kt;
      if (w.rb < 0 || w.rb >= n_rb || own[static_cast<size_t>(T)] != -1) {
        ++bad;  // outside the grid, or visited twice
        continue;
      }
      own[static_cast<size_t>(T)] = b;
      seg.push_back(T);
      if (w.kt == n_kt - 1 || u == cnt - 1) {
        const bool whole = kt0 == 0 && w.kt == n_kt - 1;
        const int64_t s = whole ? -1 : b * 2 + (sg == p.n_full ? 0 : 1);
        if (s >= 0) {
          if (holder[static_cast<size_t>(s)] != -1) ++bad;  // a slot holding two row blocks
          holder[static_cast<size_t>(s)] = w.rb;
        }
        for (const int64_t t : seg) slot[static_cast<size_t>(t)] = s;
        ++sg;
      }
    }
  }
  for (int64_t T = 0; T < W; ++T)
    if (own[static_cast<size_t>(T)] == -1) ++bad;  // never visited
  // what fixup_kernel reads for every row block of the runs
  for (int64_t rb = 0; rb < n_rb; ++rb) {
    const int64_t lo = own[static_cast<size_t>(rb * n_kt)], hi = own[static_cast<size_t>(rb * n_kt + n_kt - 1)];
    if (rb < p.full_rb) {
      if (slot[static_cast<size_t>(rb * n_kt)] != -1) ++bad;  // whole-wave blocks are written whole
      continue;
    }
    const int64_t tr = rb - p.full_rb;
    const int64_t b_lo = eot::tr::run_owner(p, tr * n_kt), b_hi = eot::tr::run_owner(p, tr * n_kt + n_kt - 1);
    if (b_lo != lo || b_hi != hi) ++bad;
    for (int64_t kt = 0; kt < n_kt; ++kt) {
      const size_t T = static_cast<size_t>(rb * n_kt + kt);
      const int64_t want = b_lo == b_hi ? -1 : eot::tr::fixup_slot(p, own[T], tr);
      if (slot[T] != want) ++bad;
    }
  }
  if (owner != nullptr)
    for (int64_t T = 0; T < W; ++T) owner[T] = own[static_cast<size_t>(T)];
  return bad == 0 ? B4_OK : -bad;
}

extern "C" size_t eot_transport_workspace_bytes(int64_t n, int64_t m, int32_t d) {
  if (!eot::tr_sizes_ok(n, m, d, d)) return 0;
  return eot::tr_layout(n, m, d, d).total;
}

extern "C" size_t eot_apply_plan_workspace_bytes(int64_t n, int64_t m, int32_t d, int32_t dv) {
  if (!eot::tr_sizes_ok(n, m, d, dv)) return 0;
  return eot::tr_layout(n, m, d, dv).total;
}

extern "C" int eot_apply_plan(const float* X, const float* Y, const float* f, const float* g,
                              const float* log_a, const float* log_b, const float* V, int32_t dv,
                              float* out, float* mass, int64_t n, int64_t m, int32_t d, float eps,
                              void* workspace, size_t workspace_bytes, birkhoff4_stream_t stream) {
  return eot::apply_impl(X, Y, f, g, log_a, log_b, V, dv, out, mass, n, m, d, eps, workspace,
                         workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int eot_transport(const float* X, const float* Y, const float* f, const float* g,
                             const float* log_a, const float* log_b, float* PY, float* mass,
                             float* grad, int64_t n, int64_t m, int32_t d, float eps,
                             void* workspace, size_t workspace_bytes, birkhoff4_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int st = eot::apply_impl(X, Y, f, g, log_a, log_b, Y, d, PY, mass, n, m, d, eps, workspace,
                                 workspace_bytes, s);
  if (st != B4_OK || n == 0 || grad == nullptr) return st;
  const int64_t total = n * static_cast<int64_t>(d);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 1 << 20);
  eot::tr::grad_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(X, PY, mass, n, d, grad);
  return b4::record_cuda_error(cudaGetLastError());
}

extern "C" size_t eot_hvp_workspace_bytes(int64_t n, int64_t m, int32_t d) {
  if (!eot::tr_sizes_ok(n, m, d, d + 1)) return 0;
  return eot::hvp_layout(n, m, d).total;
}

extern "C" int eot_hvp(const float* X, const float* Y, const float* f, const float* g,
                       const float* log_a, const float* log_b, const float* V, float* out,
                       int64_t n, int64_t m, int32_t d, float eps, int32_t cg_iters,
                       void* workspace, size_t workspace_bytes, birkhoff4_stream_t stream) {
  return eot::hvp_impl(X, Y, f, g, log_a, log_b, V, out, n, m, d, eps, cg_iters, workspace,
                       workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}
