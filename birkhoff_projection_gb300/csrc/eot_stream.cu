// eot_stream.cu -- streaming entropic OT between point clouds ("FlashSinkhorn:
// IO-Aware Entropic OT on GPU", Methodik s1-s2): the log-domain Sinkhorn
// potential update as a row-wise online log-sum-exp over a biased
// dot-product score matrix whose products run on the tcgen05 tensor cores.
// The extern "C" entries are declared and documented in eot_stream.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

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

#ifndef EOT_NEPI
#define EOT_NEPI 16
#endif
constexpr int NEPI = EOT_NEPI;  // epilogue warps: NEPI / 4 column groups per TMEM lane quarter
constexpr int GROUPS = NEPI / 4;
static_assert(NEPI % 4 == 0 && NEPI >= 4, "whole lane quarters");
constexpr int NTHREADS = 64 + 32 * NEPI;
constexpr int NBIAS = 4;       // key-tile bias buffers in shared memory

#ifndef EOT_BN1
#define EOT_BN1 256
#endif
#ifndef EOT_BN3
#define EOT_BN3 128
#endif

template <int BN, int PASSES>
struct Cfg {
  static constexpr int NOPS = PASSES == 1 ? 1 : 2;  // hi, or hi and lo
  static constexpr int A_BYTES = BM * KC * 4;
  static constexpr int B_BYTES = BN * KC * 4;
  static constexpr int STAGE_BYTES = NOPS * (A_BYTES + B_BYTES);
  static constexpr int NSTAGE = (200 * 1024) / STAGE_BYTES;
  static constexpr int SMEM = NSTAGE * STAGE_BYTES + 1024;  // + 1024-byte alignment slack
  static constexpr int TMEM_COLS = 2 * BN;                   // two accumulator buffers
  static_assert(NSTAGE >= 2, "at least two pipeline stages");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns");
};

struct LseParams {
  CUtensorMap qmap[2];  // query points hi, lo: [nq_pad rows, d_pad], box {32, 128}
  CUtensorMap kmap[2];  // key points hi, lo: [nk_pad rows, d_pad], box {32, BN}
  const float* qnorm;   // [nq_pad] squared norms of the query points
  const float* kbias;   // [nk_pad] (h_j - ||y_j||^2) log2(e)/eps + log2(w_j); -inf past nk
  float* out;           // [nq]
  float2* part;         // [n_seg][nq_pad] partial (max, sum) per row when n_seg > 1
  int64_t nq, nq_pad;
  int32_t n_rb;         // query row blocks (nq_pad / 128)
  int32_t n_seg;        // key segments per row block (work items = n_rb * n_seg)
  int32_t n_kt;         // key tiles (nk_pad / BN)
  int32_t n_kc;         // K chunks (d_pad / 32)
  float c1;             // 2 log2(e) / eps
  float out_scale;      // eps ln 2
  unsigned int* fault;
};

// First key tile of segment `seg` of `n_seg`.
__device__ __forceinline__ int seg_begin(int seg, int n_seg, int n_kt) {
  return static_cast<int>(static_cast<int64_t>(seg) * n_kt / n_seg);
}

// One 32-column chunk of a row: scores s_j = acc_j c1 + bias_j (log2
// units; the biases come from shared memory, the same for every lane), then
// the running sum of 2^(s - m) against the row's reference m.  The
// reference lags behind the true maximum: a chunk is first summed against
// the current m, and only when that sum leaves [0, 2^64] (which includes
// the first chunk of a row, m = -inf) is the exact maximum taken, the
// running sum rescaled and the chunk summed again.  Every term is then at
// most 2^64 and a row's sum at most 2^95, so nothing overflows and fp32
// keeps its relative accuracy, while most chunks skip the maximum entirely.
// Packed pair arithmetic and four partial sums keep the dependency chains
// short.
__device__ __forceinline__ float chunk_sum(const float2 (&sc)[16], float ms) {
  const float2 neg = make_float2(-ms, -ms);
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float2 e = __fadd2_rn(sc[i], neg);
    e.x = b4::ex2(e.x);
    e.y = b4::ex2(e.y);
    acc[i & 3] = __fadd2_rn(acc[i & 3], e);
  }
  const float2 t = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return t.x + t.y;
}

__device__ __forceinline__ void lse_chunk(const uint32_t (&r)[32], const float4* kb, float c1,
                                          float& m_run, float& s_run) {
  float2 sc[16];
  const float2 cc = make_float2(c1, c1);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 b = kb[i];
    sc[2 * i] = __ffma2_rn(make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])),
                           cc, make_float2(b.x, b.y));
    sc[2 * i + 1] =
        __ffma2_rn(make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), cc,
                   make_float2(b.z, b.w));
  }
  const float t = chunk_sum(sc, m_run);
  if (t <= 0x1p64f) {
    s_run += t;
    return;
  }
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    mx[i] = b4::max3(sc[2 * i].x, sc[2 * i].y, fmaxf(sc[2 * i + 1].x, sc[2 * i + 1].y));
  const float cm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  const float mn = fmaxf(m_run, cm);
  const float ms = mn == -INFINITY ? 0.0f : mn;
  s_run = fmaf(s_run, b4::ex2(m_run - ms), chunk_sum(sc, ms));
  m_run = mn;
}

// Online log-sum-exp over the score matrix S = (2 Q K^T) log2(e)/eps + bias,
// row-stationary: each CTA takes 128 query rows at a time and streams every
// key tile.  Warp roles: 0 = TMA producer, 1 = TMEM owner and MMA issuer,
// 2.. = epilogue (TMEM -> registers -> running max / sum per row).  Thread
// t of epilogue warp w owns row 32 (w % 4) + t (the TMEM lane quarter that
// warp may read) for one column group (a contiguous 1 / GROUPS of each
// tile's columns); the groups of a row are merged through shared memory
// when the row block is done.  Two TMEM accumulators let the MMAs of key
// tile t + 1 run while the epilogue reduces tile t.
template <int BN, int PASSES>
__global__ void __launch_bounds__(NTHREADS, 1) lse_kernel(const __grid_constant__ LseParams p) {
  using C = Cfg<BN, PASSES>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[C::NSTAGE], empty[C::NSTAGE], acc_full[2], acc_empty[2], mma_done;
  __shared__ uint64_t bias_full[NBIAS], bias_empty[NBIAS];
  __shared__ __align__(16) float bias_sm[NBIAS][BN];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float2 merge_sh[GROUPS > 1 ? GROUPS - 1 : 1][BM];
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      b4::mbar_init(&full[s], 1);
      b4::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      b4::mbar_init(&acc_full[b], 1);
      b4::mbar_init(&acc_empty[b], NEPI);
    }
    for (int b = 0; b < NBIAS; ++b) {
      b4::mbar_init(&bias_full[b], 1);
      b4::mbar_init(&bias_empty[b], NEPI);
    }
    b4::mbar_init(&mma_done, 1);
    abort_sh = 0;
    b4::mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    b4::prefetch_tmap(&p.qmap[0]);
    b4::prefetch_tmap(&p.kmap[0]);
    if (PASSES == 3) {
      b4::prefetch_tmap(&p.qmap[1]);
      b4::prefetch_tmap(&p.kmap[1]);
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0, tt = 0;
      const int n_items = p.n_rb * p.n_seg;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x) {
        const int rb = item % p.n_rb, seg = item / p.n_rb;
        const int kt1 = seg_begin(seg + 1, p.n_seg, p.n_kt);
        for (int kt = seg_begin(seg, p.n_seg, p.n_kt); kt < kt1 && !*abort_flag; ++kt) {
          // the key tile's biases into the shared ring
          const int slot = static_cast<int>(tt % NBIAS);
          if (!wait_bar(&bias_empty[slot], ((tt / NBIAS) & 1u) ^ 1u, abort_flag, p.fault)) break;
          b4::mbar_arrive_expect_tx(&bias_full[slot], BN * 4);
          bulk_load_1d(bias_sm[slot], p.kbias + static_cast<int64_t>(kt) * BN, BN * 4,
                       &bias_full[slot]);
          ++tt;
          for (int kc = 0; kc < p.n_kc; ++kc) {
            const int s = static_cast<int>(it % C::NSTAGE);
            const uint32_t ph = (it / C::NSTAGE) & 1u;
            if (!wait_bar(&empty[s], ph ^ 1u, abort_flag, p.fault)) break;
            unsigned char* st = smem + s * C::STAGE_BYTES;
            b4::mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
            b4::tma_load_2d(st, &p.qmap[0], &full[s], kc * KC, rb * BM);
            b4::tma_load_2d(st + C::A_BYTES, &p.kmap[0], &full[s], kc * KC, kt * BN);
            if (PASSES == 3) {
              b4::tma_load_2d(st + C::A_BYTES + C::B_BYTES, &p.qmap[1], &full[s], kc * KC, rb * BM);
              b4::tma_load_2d(st + 2 * C::A_BYTES + C::B_BYTES, &p.kmap[1], &full[s], kc * KC,
                              kt * BN);
            }
            ++it;
          }
        }
      }
      // Every issued copy must land before the CTA may exit: wait for the
      // last use of each stage and bias slot (already consumed on the normal
      // path).
      const uint32_t first = it > static_cast<uint32_t>(C::NSTAGE) ? it - C::NSTAGE : 0u;
      for (uint32_t j = first; j < it; ++j)
        b4::mbar_wait(&full[j % C::NSTAGE], (j / C::NSTAGE) & 1u, kWaitLimitNs);
      const uint32_t tfirst = tt > static_cast<uint32_t>(NBIAS) ? tt - NBIAS : 0u;
      for (uint32_t j = tfirst; j < tt; ++j)
        b4::mbar_wait(&bias_full[j % NBIAS], (j / NBIAS) & 1u, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32<BM, BN>();
      uint32_t it = 0, tc = 0;
      bool ok = true;
      const int n_items = p.n_rb * p.n_seg;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int seg = item / p.n_rb;
        const int kt1 = seg_begin(seg + 1, p.n_seg, p.n_kt);
        for (int kt = seg_begin(seg, p.n_seg, p.n_kt); kt < kt1 && ok; ++kt, ++tc) {
          const int buf = static_cast<int>(tc & 1u);
          const uint32_t use = tc >> 1;
          if (!(ok = wait_bar(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag, p.fault))) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
          for (int kc = 0; kc < p.n_kc; ++kc, ++it) {
            const int s = static_cast<int>(it % C::NSTAGE);
            if (!(ok = wait_bar(&full[s], (it / C::NSTAGE) & 1u, abort_flag, p.fault))) break;
            tc_fence_after();
            const uint32_t a_hi = b4::smem_addr(smem + s * C::STAGE_BYTES);
            const uint32_t b_hi = a_hi + C::A_BYTES;
            const uint64_t da = desc_sw128_kmajor(a_hi), db = desc_sw128_kmajor(b_hi);
#pragma unroll
            for (int kk = 0; kk < KC / KSTEP; ++kk) {
              const uint64_t adv = static_cast<uint64_t>(kk * KSTEP * 4 / 16);
              if (PASSES == 3) {
                const uint32_t a_lo = b_hi + C::B_BYTES;
                const uint32_t b_lo = a_lo + C::A_BYTES;
                mma_tf32(d_tmem, desc_sw128_kmajor(a_lo) + adv, db + adv, idesc, (kc | kk) != 0);
                mma_tf32(d_tmem, da + adv, desc_sw128_kmajor(b_lo) + adv, idesc, 1u);
                mma_tf32(d_tmem, da + adv, db + adv, idesc, 1u);
              } else {
                mma_tf32(d_tmem, da + adv, db + adv, idesc, (kc | kk) != 0);
              }
            }
            mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
          }
          if (!ok) break;
          mma_commit(&acc_full[buf]);
        }
      }
      // all MMAs issued by this thread complete before TMEM is released
      mma_commit(&mma_done);
      b4::mbar_wait(&mma_done, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: online LSE per row ----------------
    constexpr int COLS = BN / GROUPS;
    constexpr int NCH = COLS / 32;
    static_assert(COLS % 32 == 0 && NCH >= 1, "whole 32-column chunks per group");
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tc = 0;
    const int n_items = p.n_rb * p.n_seg;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int rb = item % p.n_rb, seg = item / p.n_rb;
      const int kt1 = seg_begin(seg + 1, p.n_seg, p.n_kt);
      float m_run = -INFINITY, s_run = 0.0f;
      bool ok = true;
      for (int kt = seg_begin(seg, p.n_seg, p.n_kt); kt < kt1; ++kt, ++tc) {
        const int buf = static_cast<int>(tc & 1u);
        const uint32_t use = tc >> 1;
        const int slot = static_cast<int>(tc % NBIAS);
        ok = wait_bar(&acc_full[buf], use & 1u, abort_flag, p.fault) &&
             wait_bar(&bias_full[slot], (tc / NBIAS) & 1u, abort_flag, p.fault);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int col0 = buf * BN + grp * COLS;
        const float4* kb = reinterpret_cast<const float4*>(&bias_sm[slot][grp * COLS]);
        uint32_t ra[32], rn[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(col0), ra);
        tmem_wait32(ra);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if (c + 1 < NCH) tmem_ld32(tmem + lane_base + static_cast<uint32_t>(col0 + 32 * (c + 1)), rn);
          lse_chunk(ra, kb + 8 * c, p.c1, m_run, s_run);
          if (c + 1 < NCH) {
            tmem_wait32(rn);
#pragma unroll
            for (int i = 0; i < 32; ++i) ra[i] = rn[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acc_empty[buf]);
          mbar_arrive(&bias_empty[slot]);
        }
      }
      // merge the column groups of each row (all epilogue warps reach both
      // barriers; an abort is seen by all of them after the first)
      if (grp > 0) merge_sh[grp - 1][row] = make_float2(m_run, s_run);
      named_bar_sync(1, 32 * NEPI);
      if (grp == 0 && ok && !*abort_flag) {
        float mn = m_run;
#pragma unroll
        for (int g = 0; g < GROUPS - 1; ++g) mn = fmaxf(mn, merge_sh[g][row].x);
        const float ms = mn == -INFINITY ? 0.0f : mn;
        float st = s_run * b4::ex2(m_run - ms);
#pragma unroll
        for (int g = 0; g < GROUPS - 1; ++g) {
          const float2 o = merge_sh[g][row];
          st = fmaf(o.y, b4::ex2(o.x - ms), st);
        }
        const int64_t r = static_cast<int64_t>(rb) * BM + row;
        if (p.n_seg > 1)
          p.part[static_cast<int64_t>(seg) * p.nq_pad + r] = make_float2(mn, st);
        else if (r < p.nq)
          p.out[r] = p.qnorm[r] - p.out_scale * (mn + b4::lg2(st));
      }
      named_bar_sync(1, 32 * NEPI);
      if (*abort_flag) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Pack one cloud: rows padded to rows_pad and coordinates to d_pad with zeros,
// rounded to TF32 (hi) and, for the split form, the TF32 remainder (lo); the
// squared norm of each point from its fp32 coordinates.  One warp per row.
__global__ void pack_kernel(const float* __restrict__ src, int64_t rows, int32_t d, int64_t rows_pad,
                            int32_t d_pad, float* __restrict__ hi, float* __restrict__ lo,
                            float* __restrict__ norm) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows_pad) return;
  float acc = 0.0f;
  for (int k = lane; k < d_pad; k += 32) {
    const float v = (r < rows && k < d) ? src[r * d + k] : 0.0f;
    acc = fmaf(v, v, acc);
    const float h = tf32_rna(v);
    hi[r * d_pad + k] = h;
    if (lo != nullptr) lo[r * d_pad + k] = tf32_rna(v - h);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) norm[r] = acc;
}

// Key-side bias in log2 units: (h_j - ||k_j||^2) log2(e)/eps + log2(w_j),
// -inf for the padding keys so that they add nothing to any sum.
__global__ void bias_kernel(const float* __restrict__ h, const float* __restrict__ log_w,
                            const float* __restrict__ knorm, int64_t nk, int64_t nk_pad,
                            float scale, float* __restrict__ kb) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= nk_pad) return;
  kb[j] = j < nk ? fmaf(h[j] - knorm[j], scale, log_w[j] * b4::LOG2E) : -INFINITY;
}

// Combine the key segments' partial (max, sum) of each row into the
// potential: out_r = qnorm_r - eps ln2 (M + log2 sum_k s_k 2^(m_k - M)).
__global__ void merge_kernel(const float2* __restrict__ part, int n_seg, int64_t nq, int64_t nq_pad,
                             const float* __restrict__ qnorm, float out_scale,
                             float* __restrict__ out) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= nq) return;
  float mx = -INFINITY;
  for (int k = 0; k < n_seg; ++k) mx = fmaxf(mx, part[k * nq_pad + r].x);
  const float ms = mx == -INFINITY ? 0.0f : mx;
  float st = 0.0f;
  for (int k = 0; k < n_seg; ++k) {
    const float2 v = part[k * nq_pad + r];
    st = fmaf(v.y, b4::ex2(v.x - ms), st);
  }
  out[r] = qnorm[r] - out_scale * (mx + b4::lg2(st));
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
cudaError_t pack(const float* src, int64_t rows, int32_t d, int64_t rows_pad, int32_t d_pad,
                 float* hi, float* lo, float* norm, cudaStream_t s) {
  const int64_t blocks = (rows_pad + 7) / 8;
  pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(src, rows, d, rows_pad, d_pad, hi, lo,
                                                            norm);
  return cudaGetLastError();
}

cudaError_t bias(const float* h, const float* log_w, const float* knorm, int64_t nk, int64_t nk_pad,
                 float eps, float* kb, cudaStream_t s) {
  const int64_t blocks = (nk_pad + 255) / 256;
  bias_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      h, log_w, knorm, nk, nk_pad, static_cast<float>(1.4426950408889634 / eps), kb);
  return cudaGetLastError();
}

namespace {

constexpr int kMaxSegments = 32;

// Key segments per row block: the count (1..32, at least 4 key tiles each)
// whose work items fill the last wave of `slots` resident CTAs best;
// another split is taken only when it fills at least 2% more.
int choose_segments(int64_t n_rb, int n_kt, int slots) {
  auto fill = [&](int S) {
    const int64_t items = n_rb * S;
    const int64_t waves = (items + slots - 1) / slots;
    return static_cast<double>(items) / static_cast<double>(waves * slots);
  };
  int best = 1;
  double best_fill = fill(1);
  for (int S = 2; S <= kMaxSegments && n_kt / S >= 4; ++S) {
    const double f = fill(S);
    if (f > best_fill + 0.02) {
      best = S;
      best_fill = f;
    }
  }
  return best;
}


struct Layout {
  int64_t n_pad, m_pad;
  int32_t d_pad;
  size_t x_hi, x_lo, y_hi, y_lo, x_norm, y_norm, bias, part, total;  // byte offsets
};

Layout layout(int64_t n, int64_t m, int32_t d, int32_t passes) {
  Layout L;
  L.n_pad = round_up(std::max<int64_t>(n, 1), ROW_PAD);
  L.m_pad = round_up(std::max<int64_t>(m, 1), ROW_PAD);
  L.d_pad = static_cast<int32_t>(round_up(d, KC));
  const size_t xs = align_bytes(static_cast<size_t>(L.n_pad) * L.d_pad * 4);
  const size_t ys = align_bytes(static_cast<size_t>(L.m_pad) * L.d_pad * 4);
  size_t o = 0;
  L.x_hi = o;
  o += xs;
  L.y_hi = o;
  o += ys;
  L.x_lo = L.y_lo = 0;
  if (passes == 3) {
    L.x_lo = o;
    o += xs;
    L.y_lo = o;
    o += ys;
  }
  L.x_norm = o;
  o += align_bytes(static_cast<size_t>(L.n_pad) * 4);
  L.y_norm = o;
  o += align_bytes(static_cast<size_t>(L.m_pad) * 4);
  L.bias = o;
  o += align_bytes(static_cast<size_t>(std::max(L.n_pad, L.m_pad)) * 4);
  L.part = o;
  o += align_bytes(static_cast<size_t>(std::max(L.n_pad, L.m_pad)) * 8 * kMaxSegments);
  L.total = o;
  return L;
}

bool sizes_ok(int64_t n, int64_t m, int32_t d, int32_t passes) {
  return n >= 0 && m >= 0 && n <= kMaxPoints && m <= kMaxPoints && d >= 1 && d <= 16384 &&
         (passes == 1 || passes == 3);
}

// One side of the problem as packed in the workspace.
struct Side {
  const float* hi;
  const float* lo;
  const float* norm;
  int64_t n, n_pad;
};

template <int BN, int PASSES>
cudaError_t launch_lse(const Side& qs, const Side& ks, int32_t d_pad, const float* kbias,
                       float2* part, float* out, float eps, unsigned int* fault,
                       cudaStream_t stream) {
  using C = Cfg<BN, PASSES>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int nsm = b4::sm_count(dev);
  if (nsm <= 0) return cudaErrorInvalidDevice;
  static std::atomic<int> attr_done[64];
  if (dev < 64 && attr_done[dev].load(std::memory_order_acquire) == 0) {
    err = cudaFuncSetAttribute(lse_kernel<BN, PASSES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM);
    if (err != cudaSuccess) return err;
    attr_done[dev].store(1, std::memory_order_release);
  }
  LseParams p;
  if (!encode_rows128(&p.qmap[0], qs.hi, qs.n_pad, d_pad, BM) ||
      !encode_rows128(&p.kmap[0], ks.hi, ks.n_pad, d_pad, BN))
    return cudaErrorInvalidValue;
  if (PASSES == 3) {
    if (!encode_rows128(&p.qmap[1], qs.lo, qs.n_pad, d_pad, BM) ||
        !encode_rows128(&p.kmap[1], ks.lo, ks.n_pad, d_pad, BN))
      return cudaErrorInvalidValue;
  } else {
    p.qmap[1] = p.qmap[0];
    p.kmap[1] = p.kmap[0];
  }
  p.qnorm = qs.norm;
  p.kbias = kbias;
  p.out = out;
  p.part = part;
  p.nq = qs.n;
  p.nq_pad = qs.n_pad;
  p.n_rb = static_cast<int32_t>(qs.n_pad / BM);
  p.n_kt = static_cast<int32_t>(ks.n_pad / BN);
  p.n_seg = choose_segments(p.n_rb, p.n_kt, nsm);
  p.n_kc = d_pad / KC;
  p.c1 = static_cast<float>(2.0 * 1.4426950408889634 / eps);
  p.out_scale = static_cast<float>(eps * 0.6931471805599453);
  p.fault = fault;
  const int grid = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(p.n_rb) * p.n_seg, nsm));
  lse_kernel<BN, PASSES><<<grid, NTHREADS, C::SMEM, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess || p.n_seg == 1) return err;
  const int64_t blocks = (qs.n + 255) / 256;
  merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(part, p.n_seg, qs.n, qs.n_pad,
                                                                  qs.norm, p.out_scale, out);
  return cudaGetLastError();
}

// f-type update of the query side qs against the key side ks.
cudaError_t update(const Side& qs, const Side& ks, int32_t d_pad, const float* h, const float* log_w,
                   float* kb, float2* part, float* out, float eps, int32_t passes,
                   unsigned int* fault, cudaStream_t s) {
  cudaError_t e = bias(h, log_w, ks.norm, ks.n, ks.n_pad, eps, kb, s);
  if (e != cudaSuccess) return e;
  if (passes == 3) return launch_lse<EOT_BN3, 3>(qs, ks, d_pad, kb, part, out, eps, fault, s);
  return launch_lse<EOT_BN1, 1>(qs, ks, d_pad, kb, part, out, eps, fault, s);
}

struct Packed {
  Side x, y;
  int32_t d_pad;
  float* kb;
  float2* part;
};

bool workspace_ok(const void* ws, size_t bytes, const Layout& L) {
  return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && bytes >= L.total;
}

cudaError_t pack_both(const float* X, const float* Y, int64_t n, int64_t m, int32_t d,
                      int32_t passes, void* ws, const Layout& L, Packed* P, cudaStream_t s) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  float* xhi = reinterpret_cast<float*>(w + L.x_hi);
  float* yhi = reinterpret_cast<float*>(w + L.y_hi);
  float* xlo = passes == 3 ? reinterpret_cast<float*>(w + L.x_lo) : nullptr;
  float* ylo = passes == 3 ? reinterpret_cast<float*>(w + L.y_lo) : nullptr;
  float* xn = reinterpret_cast<float*>(w + L.x_norm);
  float* yn = reinterpret_cast<float*>(w + L.y_norm);
  P->x = Side{xhi, xlo, xn, n, L.n_pad};
  P->y = Side{yhi, ylo, yn, m, L.m_pad};
  P->d_pad = L.d_pad;
  P->kb = reinterpret_cast<float*>(w + L.bias);
  P->part = reinterpret_cast<float2*>(w + L.part);
  cudaError_t e = pack(X, n, d, L.n_pad, L.d_pad, xhi, xlo, xn, s);
  if (e != cudaSuccess) return e;
  return pack(Y, m, d, L.m_pad, L.d_pad, yhi, ylo, yn, s);
}

}  // namespace
}  // namespace eot

extern "C" size_t eot_workspace_bytes(int64_t n, int64_t m, int32_t d, int32_t passes) {
  if (!eot::sizes_ok(n, m, d, passes)) return 0;
  return eot::layout(n, m, d, passes).total;
}

extern "C" int eot_update(const float* Xq, const float* Xk, const float* h, const float* log_w,
                          float* out, int64_t nq, int64_t nk, int32_t d, float eps, int32_t passes,
                          void* workspace, size_t workspace_bytes, birkhoff4_stream_t stream) {
  if (!eot::sizes_ok(nq, nk, d, passes) || !(eps > 0.0f) || !std::isfinite(eps)) return B4_EINVAL;
  if (nq == 0) return B4_OK;
  if (nk == 0) return B4_EINVAL;
  if (Xq == nullptr || Xk == nullptr || h == nullptr || log_w == nullptr || out == nullptr)
    return B4_EINVAL;
  const eot::Layout L = eot::layout(nq, nk, d, passes);
  if (!eot::workspace_ok(workspace, workspace_bytes, L)) return B4_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  unsigned int* fault = b4::device_fault_latch(&e);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  eot::Packed P;
  e = eot::pack_both(Xq, Xk, nq, nk, d, passes, workspace, L, &P, s);
  if (e == cudaSuccess) e = eot::update(P.x, P.y, P.d_pad, h, log_w, P.kb, P.part, out, eps, passes, fault, s);
  return b4::record_cuda_error(e);
}

extern "C" int eot_sinkhorn(const float* X, const float* Y, const float* log_a, const float* log_b,
                            float* f, float* g, int64_t n, int64_t m, int32_t d, float eps,
                            int32_t iters, int32_t passes, void* workspace, size_t workspace_bytes,
                            birkhoff4_stream_t stream) {
  if (!eot::sizes_ok(n, m, d, passes) || !(eps > 0.0f) || !std::isfinite(eps) || iters < 0)
    return B4_EINVAL;
  if (n == 0 && m == 0) return B4_OK;
  if (n == 0 || m == 0) return B4_EINVAL;
  if (iters == 0) return B4_OK;
  if (X == nullptr || Y == nullptr || log_a == nullptr || log_b == nullptr || f == nullptr ||
      g == nullptr)
    return B4_EINVAL;
  const eot::Layout L = eot::layout(n, m, d, passes);
  if (!eot::workspace_ok(workspace, workspace_bytes, L)) return B4_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  unsigned int* fault = b4::device_fault_latch(&e);
  if (e != cudaSuccess) return b4::record_cuda_error(e);
  eot::Packed P;
  e = eot::pack_both(X, Y, n, m, d, passes, workspace, L, &P, s);
  for (int32_t it = 0; it < iters && e == cudaSuccess; ++it) {
    e = eot::update(P.x, P.y, P.d_pad, g, log_b, P.kb, P.part, f, eps, passes, fault, s);
    if (e == cudaSuccess)
      e = eot::update(P.y, P.x, P.d_pad, f, log_a, P.kb, P.part, g, eps, passes, fault, s);
  }
  return b4::record_cuda_error(e);
}
