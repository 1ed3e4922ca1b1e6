// Deterministic dQ of the flash-attention backward (sm_103a: tcgen05 + TMEM
// + TMA), head_dim 64 and 128.
//
// The SK-16 single-pass FA Grad article (section 1) names a deterministic
// reduction order as the reason to leave the single pass with atomic dQ
// write-back and recompute instead.  Here the key-block-outer kernel then
// computes dK and dV only, and this kernel computes dQ with the loop order
// turned around: a CTA owns one (sequence, query head, 128-row query block)
// and sweeps the key blocks the mask band reaches, so that every dQ row is
// summed by one CTA, in ascending key-block order, in tensor memory:
//   C1   S    = Q K_j^T      (queries on TMEM lanes, 128 key columns)
//        dP   = dO V_j^T     (two alternating 128-column buffers)
//   V1   P    = exp2(S*scale*log2e - (m*log2e + log2 l))   (= exp(S*scale-m)/l)
//        dS   = P * (dP - D)          masked entries exactly 0
//        dS  -> bf16 into the first 32 of each warpgroup's 64 columns of the
//               dP buffer (the A operand of the next MMA, read from TMEM)
//   C2   acc += dS K_j       (fp32 in TMEM, d columns)
// and the unscaled sum is stored once into dq_acc (section 3.1 steps 1-5
// and 8; section 4.2: bf16 operands, fp32 scores and accumulation; scale is
// applied by fa_bwd_dq_finalize as in the atomic mode).  No CTA waits on
// another and nothing is added atomically, so the result does not depend on
// the schedule.  The recomputed S and dP cost 4 of the backward's 10
// matmul units (6 here against 4 saved in the key-block-outer kernel: 7/5
// of the minimum work in all).
//
// Warp roles (384 threads): warp 0 TMA producer (Q and dO once, then K in a
// 3-stage ring and V in a 2- or 3-stage ring; zeroes tail rows), warp 1
// TMEM allocator and MMA issuer, warps 4-11 two softmax warpgroups (thread =
// query row; warpgroup g owns key columns [64g, 64g + 64) of every block)
// and the epilogue.  Every wait is bounded (see sm103.cuh).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "sm103.cuh"

namespace fa {

__device__ int g_dq_status = 0;

namespace {

constexpr int kThreads = 384;
constexpr uint32_t kRegLaunch = 65536 / kThreads / 8 * 8;   // 168
constexpr uint32_t kRegOther = 80;      // warps 0-3
constexpr uint32_t kRegSoftmax = 200;   // warps 4-11
static_assert(128 * kRegOther + 256 * kRegSoftmax <= kThreads * kRegLaunch, "register budgets exceed the launch");
constexpr int BQ = 128;                 // query rows per CTA
constexpr int BK = 128;                 // key rows per block
constexpr uint32_t CHUNK = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128 B)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_DP0 = 128;       // two dP buffers: [128, 256) and [256, 384)
constexpr uint32_t COL_ACC = 384;       // dQ accumulator, d columns
constexpr int KS = 3;                   // K stages
template <int D>
constexpr int kVStages = (D == 64) ? 3 : 2;

enum {
  B_Q_FULL = 0, B_Q_READY,
  B_K_FULL0, B_K_READY0 = B_K_FULL0 + 3, B_K_EMPTY0 = B_K_READY0 + 3,   // up to 3 K stages
  B_V_FULL0 = B_K_EMPTY0 + 3, B_V_EMPTY0 = B_V_FULL0 + 3,
  B_S_FULL = B_V_EMPTY0 + 3, B_P_DONE, B_DP_FULL0, B_DP_FULL1, B_DS_READY0, B_DS_READY1, B_DQ_DONE0, B_DQ_DONE1,
  B_ACC_FULL,
  B_TEARDOWN, NUM_BARS
};

template <int D>
struct Layout {
  static constexpr uint32_t TILE = 128 * D * 2;   // [128 rows, D] bf16
  static constexpr int NCH = D / 64;
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t DO = TILE;
  static constexpr uint32_t K = 2 * TILE;                   // KS stages
  static constexpr uint32_t V = K + KS * TILE;              // kVStages stages
  static constexpr uint32_t BARS = V + kVStages<D> * TILE;
  static constexpr uint32_t MISC = BARS + NUM_BARS * 8;     // abort flag, TMEM address
  static constexpr uint32_t BYTES = MISC + 16;
  static_assert(COL_ACC + D <= TMEM_COLS, "tensor memory budget");
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int t) {
  return sw128_desc(tile + (t >> 2) * CHUNK + (t & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int t) {
  return sw128_desc(tile + t * 2048, CHUNK, 1024);
}
__device__ __forceinline__ constexpr uint64_t step_kmajor(int t) { return ((t >> 2) * CHUNK + (t & 3) * 32) >> 4; }
__device__ __forceinline__ constexpr uint64_t step_mnmajor(int t) { return (t * 2048) >> 4; }

// N K-steps of 16 with both operands K-major in shared memory (S, dP).
template <int N>
__device__ __forceinline__ void mmas_kk(uint32_t d, uint32_t a_tile, uint32_t b_tile, uint32_t idesc) {
  const uint64_t a0 = desc_kmajor(a_tile, 0), b0 = desc_kmajor(b_tile, 0);
#pragma unroll 4
  for (int t = 0; t < N; ++t) mma_ss(d, a0 + step_kmajor(t), b0 + step_kmajor(t), idesc, t > 0);
}
// acc (+)= dS K: A (dS, bf16 pairs) from TMEM, K step t at column
// 64*(t/4) + 8*(t%4); B = K tile read MN-major (head dims contiguous).
// (dS staged in shared memory instead, so that both operands come from
// there, measured slower: the softmax then waits for the previous product
// to have read the single buffer.)
__device__ __forceinline__ void mmas_dq(uint32_t d, uint32_t a_tmem, uint32_t k_tile, uint32_t idesc, uint32_t acc) {
  const uint64_t b0 = desc_mnmajor(k_tile, 0);
#pragma unroll 4
  for (int t = 0; t < BK / 16; ++t)
    mma_ts(d, a_tmem + (t >> 2) * 64 + (t & 3) * 8, b0 + step_mnmajor(t), idesc, acc | (t > 0));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Zero rows [first, 128) of a [128, D] tile with the 32 lanes of one warp.
template <int D>
__device__ __forceinline__ void zero_rows(uint32_t tile, int first, int lane) {
  constexpr int NCH = D / 64;
  const int nrows = 128 - first;
  for (int e = lane; e < nrows * NCH * 8; e += 32) {
    const int row = first + e / (NCH * 8);
    const int rem = e % (NCH * 8);
    st_shared_v4(tile + (rem / 8) * CHUNK + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
  }
}

// P phase of one softmax thread: query row r, this warpgroup's 64 key
// columns of S in TMEM (taddr = the row's lane, first column).  P =
// 2^(S*scale*log2e - lse2) (= exp(S*scale - m) / l); with MASK, entries
// outside the row's visible run of key columns [c_lo, c_lo + span) are 0.
// MASK is a template parameter so that full blocks run a loop without any
// per-element mask work.
template <bool MASK>
__device__ __forceinline__ void softmax_p(uint32_t taddr, float sl2, float neg_lse2, float (&P)[64], int kc0, int c_lo,
                                          int span) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t v[32];
    tmem_ld32(taddr + half * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int c2 = 0; c2 < 16; ++c2) {
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[2 * c2]), __uint_as_float(v[2 * c2 + 1])),
                                  make_float2(sl2, sl2), make_float2(neg_lse2, neg_lse2));
      float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
      if (MASK) {
        const int col = kc0 + half * 32 + 2 * c2;
        p0 = (static_cast<unsigned>(col - c_lo) < static_cast<unsigned>(span)) ? p0 : 0.f;
        p1 = (static_cast<unsigned>(col + 1 - c_lo) < static_cast<unsigned>(span)) ? p1 : 0.f;
      }
      P[half * 32 + 2 * c2] = p0;
      P[half * 32 + 2 * c2 + 1] = p1;
    }
  }
}

// dS phase: dS = P * (dP - D) from dP in TMEM (taddr), rounded to bf16 and
// stored as pairs into the first 32 of the 64 columns just read.
template <bool MASK>
__device__ __forceinline__ void softmax_ds(uint32_t taddr, float neg_D, const float (&P)[64]) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t v[32];
    tmem_ld32(taddr + half * 32, v);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int c2 = 0; c2 < 16; ++c2) {
      const int c0 = half * 32 + 2 * c2;
      // dS = P * (dP - D), two at a time (packed fp32 add and multiply)
      float2 ds = __fmul2_rn(make_float2(P[c0], P[c0 + 1]),
                             __fadd2_rn(make_float2(__uint_as_float(v[2 * c2]), __uint_as_float(v[2 * c2 + 1])),
                                        make_float2(neg_D, neg_D)));
      if (MASK) {   // P is 0 where masked, but dP there may be anything (NaN padding)
        ds.x = (P[c0] != 0.f) ? ds.x : 0.f;
        ds.y = (P[c0 + 1] != 0.f) ? ds.y : 0.f;
      }
      pk[c2] = pack_bf16x2(ds.x, ds.y);
    }
    // the first 16 (then 32) columns of this half were already read
    tmem_st16(taddr + half * 16, pk);
  }
}

__device__ __forceinline__ int floordiv(long long a, int b) {
  long long q = a / b;
  if ((a % b) != 0 && a < 0) --q;
  return static_cast<int>(q);
}

// Launch order (x: query block, y: query head, z: sequence).  Under a causal
// mask later query blocks see more keys and go first; chunked as in the
// forward-statistics kernel when the blocks' key ranges are uneven.
template <bool kChunked>
__device__ __forceinline__ void dq_block_of(const BwdParams& p, int& x, int& h, int& b) {
  if constexpr (!kChunked) {
    x = p.causal ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
    h = blockIdx.y;
    b = blockIdx.z;
  } else {
    const int nx = static_cast<int>(gridDim.x);
    const int lin = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    const int units = p.heads * p.batch;
    const int per_chunk = p.head_chunk * nx;
    const int ch = lin / per_chunk;
    const int r = lin - ch * per_chunk;
    const int g = min(p.head_chunk, units - ch * p.head_chunk);
    const int t = r / g;
    const int unit = ch * p.head_chunk + (r - t * g);
    x = nx - 1 - t;
    h = unit % p.heads;
    b = unit / p.heads;
  }
}

template <int D, bool kChunked>
__global__ void __launch_bounds__(kThreads, 1) dq_kernel(const __grid_constant__ BwdParams p) {
  using L = Layout<D>;
  constexpr int VS = kVStages<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int qb, h, b;
  dq_block_of<kChunked>(p, qb, h, b);
  const int H = p.heads;
  const int hk = h / (H / p.heads_kv);
  const int q_start = p.cu_q[b], s1 = p.cu_q[b + 1] - q_start;
  const int kv_start = p.cu_kv[b], s2 = p.cu_kv[b + 1] - kv_start;
  if (qb * BQ >= s1) return;                          // CTA-uniform, before any barrier
  const int q_valid = min(BQ, s1 - qb * BQ);
  // Mask band: query i sees key j iff j <= i + off (causal) and
  // j > i + off - W (window W > 0); key blocks this query block reaches:
  // [kb0, kb1].
  const int off = p.bottom_right ? s2 - s1 : 0;
  const int W = p.window;
  const int n_kb = (s2 + BK - 1) / BK;
  const long long q0 = static_cast<long long>(qb) * BQ;
  const int kb1 = p.causal ? min(n_kb - 1, floordiv(q0 + BQ - 1 + off, BK)) : n_kb - 1;
  const int kb0 = (p.causal && W > 0) ? max(0, floordiv(q0 + off - W + 1, BK)) : 0;
  const int n = kb1 - kb0 + 1;
  const long long rs = static_cast<long long>(H) * D;   // query-side row stride (elements)

  if (n <= 0) {
    // no row of this block sees a key: its dQ is 0
    for (int e = threadIdx.x; e < q_valid * (D / 4); e += kThreads) {
      const int r = e / (D / 4), c = (e % (D / 4)) * 4;
      st_global_v4(p.dq_acc + (q_start + qb * BQ + r) * rs + h * D + c, 0u, 0u, 0u, 0u);
    }
    return;
  }
  if (sbase & 1023) {                                 // swizzled tiles need 1 KB alignment
    if (threadIdx.x == 0) atomicCAS(&g_dq_status, 0, 99);
    return;
  }

  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC + 4);
  const uint32_t bars = sbase + L::BARS;
  auto bar = [&](int i) { return bars + 8u * i; };
  int* status = &g_dq_status;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_READY), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(B_K_FULL0 + s), 1);
      mbar_init(bar(B_K_READY0 + s), 1);
      mbar_init(bar(B_K_EMPTY0 + s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar(B_V_FULL0 + s), 1);
      mbar_init(bar(B_V_EMPTY0 + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_P_DONE), 256);
    mbar_init(bar(B_DP_FULL0), 1);
    mbar_init(bar(B_DP_FULL1), 1);
    // one per dP buffer: the MMA warp issues dP_{j+1} before it waits for
    // dS_j, so with a single barrier the softmax could complete dS_{j+1}
    // (its next phase) before that wait had seen dS_j
    mbar_init(bar(B_DS_READY0), 256);
    mbar_init(bar(B_DS_READY1), 256);
    mbar_init(bar(B_DQ_DONE0), 1);
    mbar_init(bar(B_DQ_DONE1), 1);
    mbar_init(bar(B_ACC_FULL), 1);
    mbar_init(bar(B_TEARDOWN), 1);
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    setmaxnreg_to<kRegOther, kRegLaunch>();
    const int q_row0 = q_start + qb * BQ;
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(bar(B_Q_FULL), 2 * L::TILE);
      for (int c = 0; c < L::NCH; ++c) {
        tma_load_2d(sbase + L::Q + c * CHUNK, &p.tm_q, h * D + c * 64, q_row0, bar(B_Q_FULL));
        tma_load_2d(sbase + L::DO + c * CHUNK, &p.tm_do, h * D + c * 64, q_row0, bar(B_Q_FULL));
      }
    }
    __syncwarp();
    bool ok = true, q_seen = false;
    int issued_k = 0, seen_k = 0, issued_v = 0;
    for (int j = 0; ok && j < n; ++j) {
      const int kb = kb0 + j;
      const int row = kv_start + kb * BK;
      const int sk = j % KS, sv = j % VS;
      if (j >= KS && !mbar_wait(bar(B_K_EMPTY0 + sk), ((j / KS) - 1) & 1, abort, status)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_K_FULL0 + sk), L::TILE);
        for (int c = 0; c < L::NCH; ++c)
          tma_load_2d(sbase + L::K + sk * L::TILE + c * CHUNK, &p.tm_k, hk * D + c * 64, row, bar(B_K_FULL0 + sk));
      }
      issued_k = j + 1;
      if (j >= VS && !mbar_wait(bar(B_V_EMPTY0 + sv), ((j / VS) - 1) & 1, abort, status)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_V_FULL0 + sv), L::TILE);
        for (int c = 0; c < L::NCH; ++c)
          tma_load_2d(sbase + L::V + sv * L::TILE + c * CHUNK, &p.tm_v, hk * D + c * 64, row, bar(B_V_FULL0 + sv));
      }
      issued_v = j + 1;
      if (j == 0) {
        // Q and dO rows past the sequence end (other data or NaN padding)
        // would reach the scores and dP of real keys through the MMAs
        if (!mbar_wait(bar(B_Q_FULL), 0, abort, status)) { ok = false; break; }
        q_seen = true;
        if (q_valid < BQ) {
          zero_rows<D>(sbase + L::Q, q_valid, lane);
          zero_rows<D>(sbase + L::DO, q_valid, lane);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_Q_READY));
      }
      // Key rows past the sequence end: their score columns are masked, but
      // they are also the B operand of acc += dS K, where 0 * NaN = NaN.
      if (!mbar_wait(bar(B_K_FULL0 + sk), (j / KS) & 1, abort, status)) { ok = false; break; }
      seen_k = j + 1;
      const int kv_valid = min(BK, s2 - kb * BK);
      if (kv_valid < BK) {
        zero_rows<D>(sbase + L::K + sk * L::TILE, kv_valid, lane);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_K_READY0 + sk));
    }
    // every load issued must land before the CTA exits, also after an abort
    volatile int no_abort = 0;
    for (int jj = max(seen_k, issued_k - KS); jj < issued_k; ++jj)
      mbar_wait(bar(B_K_FULL0 + jj % KS), (jj / KS) & 1, &no_abort, status);
    for (int jj = max(0, issued_v - VS); jj < issued_v; ++jj)
      mbar_wait(bar(B_V_FULL0 + jj % VS), (jj / VS) & 1, &no_abort, status);
    if (!q_seen) mbar_wait(bar(B_Q_FULL), 0, &no_abort, status);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_to<kRegOther, kRegLaunch>();
    constexpr uint32_t ID_S = idesc_bf16(128, BK, 0, 0);    // S, dP: both K-major
    constexpr uint32_t ID_DQ = idesc_bf16(128, D, 0, 1);    // acc += dS K: B (K) MN-major
    const uint32_t sQ = sbase + L::Q, sDO = sbase + L::DO;
    auto issue_dp = [&](int j) {   // dP_j into buffer j & 1 (V_j landed, buffer free)
      const int sv = j % VS;
      if (elect_one()) {
        mmas_kk<D / 16>(tmem + COL_DP0 + (j & 1) * 128, sDO, sbase + L::V + sv * L::TILE, ID_S);
        mma_commit(bar(B_DP_FULL0 + (j & 1)));
        mma_commit(bar(B_V_EMPTY0 + sv));   // dP was V_j's only use
      }
      __syncwarp();
    };
    // Issue order per key block j: S_{j+1} as soon as the softmax has read
    // S_j, then dP_{j+1} (its buffer held dS_{j-1}, long consumed), then
    // acc += dS_j K_j once dS_j is written.  The softmax needs S_{j+1} right
    // after dS_j and dP_{j+1} right after P_{j+1}, so both are queued on the
    // tensor pipe ahead of the dQ product, which nothing waits for.
    bool ok = mbar_wait(bar(B_Q_READY), 0, abort, status) && mbar_wait(bar(B_K_READY0), 0, abort, status);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        mmas_kk<D / 16>(tmem + COL_S, sQ, sbase + L::K, ID_S);
        mma_commit(bar(B_S_FULL));
      }
      __syncwarp();
      ok = mbar_wait(bar(B_V_FULL0), 0, abort, status);
      if (ok) {
        tc_fence_after();
        issue_dp(0);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      if (j + 1 < n) {
        // S_{j+1} overwrites S_j: the softmax must have read it
        const int sk1 = (j + 1) % KS;
        if (!mbar_wait(bar(B_P_DONE), j & 1, abort, status) ||
            !mbar_wait(bar(B_K_READY0 + sk1), ((j + 1) / KS) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          mmas_kk<D / 16>(tmem + COL_S, sQ, sbase + L::K + sk1 * L::TILE, ID_S);
          mma_commit(bar(B_S_FULL));
        }
        __syncwarp();
        // dP_{j+1} into buffer (j+1) & 1 once acc += dS_{j-1} K_{j-1} has read it
        if ((j >= 1 && !mbar_wait(bar(B_DQ_DONE0 + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort, status)) ||
            !mbar_wait(bar(B_V_FULL0 + (j + 1) % VS), ((j + 1) / VS) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        issue_dp(j + 1);
      }
      // acc += dS_j K_j, dS_j read from dP buffer j & 1
      if (!mbar_wait(bar(B_DS_READY0 + (j & 1)), (j >> 1) & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      const int sk = j % KS;
      if (elect_one()) {
        mmas_dq(tmem + COL_ACC, tmem + COL_DP0 + (j & 1) * 128, sbase + L::K + sk * L::TILE, ID_DQ, j > 0);
        mma_commit(bar(B_DQ_DONE0 + (j & 1)));
        mma_commit(bar(B_K_EMPTY0 + sk));    // the dQ product was K_j's last use
      }
      __syncwarp();
    }
    ok = __all_sync(0xffffffffu, ok);
    if (elect_one()) mma_commit(bar(ok ? B_ACC_FULL : B_TEARDOWN));
    __syncwarp();
    if (!ok) {
      // aborted: wait (bounded) for every MMA issued so far before TMEM is freed
      volatile int no_abort = 0;
      mbar_wait(bar(B_TEARDOWN), 0, &no_abort, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS
    setmaxnreg_to<kRegSoftmax, kRegLaunch>();
    const int wg = (warp - 4) >> 2;              // key columns [64 wg, 64 wg + 64)
    const int quarter = warp & 3;                // TMEM lane quarter
    const int r = quarter * 32 + lane;           // query row in the block
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const long long i_loc = q0 + r;              // query index in its sequence
    // This row's statistics, negated for the FMA / add below: exp(x*scale - m)/l
    // = 2^(x*scale*log2e - (m*log2e + log2 l)).  Rows past the sequence end
    // see no key (span 0 below), so their values never reach a result.
    float neg_lse2 = 0.f, neg_D = 0.f;
    if (r < q_valid) {
      const long long idx = static_cast<long long>(q_start + qb * BQ + r) * H + h;
      const float mv = __ldg(p.m + idx);
      neg_lse2 = -(mv * 1.4426950408889634f + (p.stats_lse ? 0.f : __log2f(__ldg(p.l + idx))));
      neg_D = -__ldg(p.D + idx);
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int kb = kb0 + j;
      // visible key columns of this row in block kb: [c_lo, c_lo + span)
      const long long d0 = i_loc + off - static_cast<long long>(kb) * BK;   // last visible column
      int c_lo = 0, c_end = min(BK, s2 - kb * BK);
      if (p.causal) {
        c_end = static_cast<int>(max(0LL, min(static_cast<long long>(c_end), d0 + 1)));
        if (W > 0) c_lo = static_cast<int>(max(0LL, min(static_cast<long long>(BK), d0 - W + 1)));
      }
      const int span = (r < q_valid) ? max(0, c_end - c_lo) : 0;
      const bool need_mask = __any_sync(0xffffffffu, c_lo > wg * 64 || c_lo + span < wg * 64 + 64);
      if (!mbar_wait(bar(B_S_FULL), j & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      float P[64];
      const uint32_t t_s = tmem + lane_addr + COL_S + wg * 64;
      if (need_mask)
        softmax_p<true>(t_s, sl2, neg_lse2, P, wg * 64, c_lo, span);
      else
        softmax_p<false>(t_s, sl2, neg_lse2, P, wg * 64, c_lo, span);
      tc_fence_before();
      mbar_arrive(bar(B_P_DONE));                  // S may be overwritten
      if (!mbar_wait(bar(B_DP_FULL0 + (j & 1)), (j >> 1) & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_dp = tmem + lane_addr + COL_DP0 + (j & 1) * 128 + wg * 64;
      if (need_mask)
        softmax_ds<true>(t_dp, neg_D, P);
      else
        softmax_ds<false>(t_dp, neg_D, P);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_DS_READY0 + (j & 1)));
    }
    // ------------------------------------------------------------ epilogue
    // Warpgroup g stores head dims [g D/2, (g+1) D/2) of its rows.
    if (__all_sync(0xffffffffu, ok && mbar_wait(bar(B_ACC_FULL), 0, abort, status))) {
      tc_fence_after();
      if (q_valid == BQ) {
        // A whole query block: each warp stages its 32 rows x D/2 columns as
        // 128B-swizzled [32 x 32] fp32 boxes in the Q / dO tiles, which no
        // MMA reads any more, and stores them with TMA (coalesced, instead of
        // 16-byte pieces of 32 rows per warp store).  A partial block is
        // written per row below, so that no row of the next sequence is
        // touched.
        const uint32_t box0 = sbase + L::Q + (wg * 4 + quarter) * (D / 64) * 4096;
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + COL_ACC + wg * (D / 2) + ch * 32, v);
          tmem_ld_wait();
          const uint32_t row = box0 + ch * 4096 + lane * 128;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            st_shared_v4(row + ((g ^ (lane & 7)) << 4), v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int ch = 0; ch < D / 64; ++ch)
            tma_store_2d(&p.tm_dq, box0 + ch * 4096, h * D + wg * (D / 2) + ch * 32, q_start + qb * BQ + quarter * 32);
          bulk_commit();
          bulk_wait_read0();   // the boxes are read before the CTA exits
        }
        __syncwarp();
      } else {
        float* dst = p.dq_acc + (q_start + qb * BQ + r) * rs + h * D + wg * (D / 2);
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + COL_ACC + wg * (D / 2) + ch * 32, v);
          tmem_ld_wait();
          if (r < q_valid) {
#pragma unroll
            for (int g = 0; g < 8; ++g) st_global_v4(dst + ch * 32 + g * 4, v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
          }
        }
      }
    }
  } else {
    setmaxnreg_to<kRegOther, kRegLaunch>();   // warps 2, 3 only wait at the final barrier
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Chunk of the launch order: 1 (query block fastest) unless a causal mask
// makes the blocks' key ranges differ enough (longest > 1.5 x mean, for the
// longest sequences) for the order to matter; then chunks whose key-side
// bytes (K and V of one key/value head, shared by its query heads) take
// about a quarter of L2.
int dq_head_chunk(const BwdParams& p, int batch, int n_qb, int max_kv, int head_dim) {
  constexpr long long kChunkBytes = 32ll << 20;
  if (!p.causal || n_qb <= 1 || max_kv <= 0) return 1;
  const long long s1 = static_cast<long long>(n_qb) * BQ, s2 = max_kv;
  const long long off = p.bottom_right ? s2 - s1 : 0;
  const long long n_kb = (s2 + BK - 1) / BK;
  auto fdiv = [](long long a, long long b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
  long long total = 0, longest = 0;
  for (long long x = 0; x < n_qb; ++x) {
    const long long q0 = x * BQ;
    const long long kb1 = std::min(n_kb - 1, fdiv(q0 + BQ - 1 + off, BK));
    const long long kb0 = p.window > 0 ? std::max(0LL, fdiv(q0 + off - p.window + 1, BK)) : 0;
    const long long n = std::max(0LL, kb1 - kb0 + 1);
    total += n;
    longest = std::max(longest, n);
  }
  if (2 * longest * n_qb <= 3 * total) return 1;
  const long long unit_bytes = std::max(1LL, s2 * head_dim * 4 / std::max(1, p.heads / std::max(1, p.heads_kv)));
  return static_cast<int>(std::max(1LL, std::min<long long>(static_cast<long long>(p.heads) * batch, kChunkBytes / unit_bytes)));
}

template <int D>
cudaError_t launch_d(const BwdParams& p, int batch, int max_kv, cudaStream_t s) {
  constexpr uint32_t bytes = Layout<D>::BYTES;
  static_assert(bytes <= 232448, "shared memory budget");
  static std::atomic<unsigned long long> smem_set{0}, smem_set_chunked{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(dq_kernel<D, false>), (int)bytes, smem_set);
  if (e == cudaSuccess) e = set_smem_once(reinterpret_cast<const void*>(dq_kernel<D, true>), (int)bytes, smem_set_chunked);
  if (e != cudaSuccess) return e;
  const int n_qb = p.max_q_blocks;
  if (static_cast<long long>(n_qb) * p.heads * batch > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  BwdParams q = p;
  q.batch = batch;
  q.head_chunk = dq_head_chunk(p, batch, n_qb, max_kv, D);
  dim3 grid(n_qb, p.heads, batch);
  if (q.head_chunk > 1)
    dq_kernel<D, true><<<grid, kThreads, bytes, s>>>(q);
  else
    dq_kernel<D, false><<<grid, kThreads, bytes, s>>>(q);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq(const BwdParams& p, int head_dim, int batch, int max_kv, cudaStream_t s) {
  if (batch <= 0 || p.max_q_blocks <= 0) return cudaSuccess;
  return head_dim == 64 ? launch_d<64>(p, batch, max_kv, s) : launch_d<128>(p, batch, max_kv, s);
}

int dq_read_and_clear_status(cudaStream_t s, int* status) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_dq_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_dq_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return static_cast<int>(e);
}

}  // namespace fa
