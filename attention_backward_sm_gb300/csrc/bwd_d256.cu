// Single-pass flash-attention backward for head_dim 256 (sm_103a: tcgen05 +
// TMEM + TMA).  Same computation as the head_dim 64/128 kernel (the SK-16
// single-pass FA Grad article, sections 3, 3.1, 4.1 and 4.2; the key-block
// outer loop of section 1), with a different split of the work, forced by
// the on-chip budgets: the dK and dV accumulators of a 128-row key block
// at d = 256 would take all 512 TMEM columns, and the K, V, Q, dO tiles
// 256 KB of shared memory.
//
// Two CTAs share one (sequence, key/value head, 128-row key block); CTA
// c in {0, 1} owns head-dimension half c of dK, dV and dQ.  Each computes
// the full scores and dP itself (a contraction over all 256 dimensions), so
// no data moves between the two; the cost is computing S and dP twice,
// 7/5 of the minimum matmul work.  Per 64-row query block i:
//   S^T  = K Q_i^T                  (M = 128 keys, N = 64 queries, K = 256)
//   dP^T = V dO_i^T                 V is kept in TMEM as the A operand
//   P, dS as in the 64/128 kernel (keys on TMEM lanes)
//   dV_c += P^T dO_i[:, half c]     (A = P from TMEM)
//   dK_c += dS^T Q_i[:, half c]
//   dQ_c^T = K_c^T dS^T             (M = 128 head dims, N = 64 queries);
//                                   staged transposed in shared memory and
//                                   added into dq_acc with TMA reduce-add
// TMEM: V [0,128) (bf16 pairs), S^T [128,192) (P overwrites the first 16
// columns of each softmax warpgroup's 32), dP^T [192,256) (reused for
// dQ_c^T), dV_c [256,384), dK_c [384,512).
// Shared memory: K 64 KB, Q and dO two stages of 32 KB each (V passes
// through the dO stages once on its way to TMEM), dS 16 KB, dQ staging
// 16 KB, statistics.
//
// Warp roles (512 threads): warp 0 TMA producer of K and V, warp 3 of Q and
// the row statistics, warp 2 of dO, warp 1 TMEM allocator and MMA issuer,
// warps 4-11 two softmax warpgroups (32 query columns each; warpgroup 0
// also moves V into TMEM; at the end dV_c / dK_c), warps 12-15 dQ
// write-back (lane = head dimension).  Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"
#include "sm103.cuh"

namespace fa {

__device__ int g_bwd256_status = 0;

namespace {

constexpr int D = 256;
constexpr int HALF = 128;                // head dimensions per CTA
constexpr int BM = 128;                  // key rows per CTA
constexpr int BN = 64;                   // query rows per block
constexpr int kThreads = 512;
constexpr uint32_t kRegLaunch = 65536 / kThreads;
constexpr uint32_t kRegOther = 56;
constexpr uint32_t kRegSoftmax = 152;
constexpr uint32_t kRegDrain = 152;
static_assert(128 * kRegOther + 256 * kRegSoftmax + 128 * kRegDrain <= 65536, "register budgets exceed the launch");
constexpr uint32_t CHUNK_K = BM * 128;   // 64-column chunk of a 128-row tile
constexpr uint32_t CHUNK_Q = BN * 128;   // 64-column chunk of a 64-row tile
constexpr uint32_t TILE_K = BM * D * 2;  // 64 KB
constexpr uint32_t TILE_Q = BN * D * 2;  // 32 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_V = 0;
constexpr uint32_t COL_S = 128;
constexpr uint32_t COL_DP = 192;
constexpr uint32_t COL_DV = 256;
constexpr uint32_t COL_DK = 384;

enum {
  B_KV_FULL = 0, B_KV_READY, B_V_DONE,
  B_Q_FULL0, B_Q_FULL1, B_Q_READY0, B_Q_READY1, B_Q_EMPTY0, B_Q_EMPTY1,
  B_DO_FULL0, B_DO_FULL1, B_DO_READY0, B_DO_READY1, B_DO_EMPTY0, B_DO_EMPTY1,
  B_S_FULL, B_DP_FULL, B_P_READY, B_P_USED, B_DS_READY, B_DS_FREE, B_DQ_FULL, B_DQ_EMPTY, B_ACC_FULL,
  B_TEARDOWN, B_EPI0, B_EPI1, NUM_BARS
};

struct Layout {
  static constexpr uint32_t K = 0;
  static constexpr uint32_t Q = TILE_K;                 // 2 stages
  static constexpr uint32_t DO = Q + 2 * TILE_Q;        // 2 stages; V on its way to TMEM
  static constexpr uint32_t DS = DO + 2 * TILE_Q;       // [128 keys, 64 queries] bf16
  static constexpr uint32_t DQST = DS + BM * BN * 2;    // 4 boxes of [32 queries, 32 dims] fp32
  static constexpr uint32_t STATS = DQST + 4 * 4096;    // per stage: lse2[64], D[64]
  static constexpr uint32_t BARS = STATS + 2 * 2 * BN * 4;
  static constexpr uint32_t MISC = BARS + NUM_BARS * 8;
  static constexpr uint32_t BYTES = MISC + 16;
};
static_assert(Layout::DO + 2 * TILE_Q >= Layout::DO + TILE_K, "V staging fits in the dO stages");

// 16-element K step t of a K-major tile with 64-column chunks `chunk` apart
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int t, uint32_t chunk) {
  return sw128_desc(tile + (t >> 2) * chunk + (t & 3) * 32, 16, 1024);
}
// rows 16t..16t+15 of an MN-major tile with 64-column chunks `chunk` apart
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int t, uint32_t chunk) {
  return sw128_desc(tile + t * 2048, chunk, 1024);
}

// The same descriptors stepped by constants: the start address is the
// descriptor's low 14 bits (addr >> 4) and every step stays inside its tile,
// so the issuing warp builds a group's descriptors once and adds offsets.
__device__ __forceinline__ constexpr uint64_t step_k(int t, uint32_t chunk) {
  return ((t >> 2) * chunk + (t & 3) * 32) >> 4;
}
__device__ __forceinline__ constexpr uint64_t step_mn(int t) { return (t * 2048) >> 4; }

__device__ __forceinline__ int floordiv(long long a, int b) {
  long long q = a / b;
  if ((a % b) != 0 && a < 0) --q;
  return static_cast<int>(q);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t a) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Zero rows [first, rows) of a tile of 4 chunks (`chunk` apart) with one warp.
__device__ __forceinline__ void zero_rows(uint32_t tile, int first, int rows, uint32_t chunk, int lane) {
  const int n = (rows - first) * 4 * 8;
  for (int e = lane; e < n; e += 32) {
    const int row = first + e / 32, rem = e % 32;
    st_shared_v4(tile + (rem / 8) * chunk + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
  }
}

template <bool kChunked>
__global__ void __launch_bounds__(kThreads, 1) bwd256_kernel(const __grid_constant__ BwdParams p) {
  using L = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Launch order as in the 64/128 kernel.  head_chunk = 1: grid (key block,
  // key/value head, 2 x sequence + head-dimension half).  head_chunk > 1:
  // (sequence, key/value head) units in chunks, key block slow within a
  // chunk, the two head-dimension halves of a key block side by side.
  //
  // Deterministic mode (unchunked): a CTA's dQ additions wait for those of
  // the key blocks before it in the order of the tickets, which are the
  // CTAs before it in this launch order.  So that every CTA waited for has
  // certainly started, whatever order the hardware starts CTAs in, the
  // position in the launch order is taken from a global counter when the CTA
  // starts instead of from its block index.
  int kvb, hk, b, c;                                 // c: head-dimension half
  if constexpr (!kChunked) {
    int bx = blockIdx.x, by = blockIdx.y, bz = blockIdx.z;
    if (p.work_counter != nullptr) {
      int* item_slot = reinterpret_cast<int*>(smem + Layout::MISC + 8);
      if (threadIdx.x == 0) *item_slot = atomicAdd(p.work_counter, 1);
      __syncthreads();
      const int item = *item_slot;
      bx = item % static_cast<int>(gridDim.x);
      by = (item / static_cast<int>(gridDim.x)) % static_cast<int>(gridDim.y);
      bz = item / static_cast<int>(gridDim.x * gridDim.y);
    }
    kvb = p.kv_reverse ? static_cast<int>(gridDim.x) - 1 - bx : bx;
    hk = by;
    b = bz >> 1;
    c = bz & 1;
  } else {
    const int lin = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    const int units = p.heads_kv * p.batch;
    const int per_chunk = p.head_chunk * 2 * p.grid_kv;
    const int ch = lin / per_chunk;
    const int r = lin - ch * per_chunk;
    const int g = min(p.head_chunk, units - ch * p.head_chunk);
    const int x = r / g;
    const int unit = ch * p.head_chunk + (r - x * g);
    c = x & 1;
    kvb = x >> 1;
    hk = unit % p.heads_kv;
    b = unit / p.heads_kv;
  }
  const int H = p.heads;
  const int G = p.heads / p.heads_kv;
  const int q_start = p.cu_q[b], s1 = p.cu_q[b + 1] - q_start;
  const int kv_start = p.cu_kv[b], s2 = p.cu_kv[b + 1] - kv_start;
  if (kvb * BM >= s2) return;                       // CTA-uniform, before any barrier
  if (sbase & 1023) {
    if (threadIdx.x == 0) atomicCAS(&g_bwd256_status, 0, 99);
    return;
  }
  const int kv_valid = min(BM, s2 - kvb * BM);
  const int n_qb = (s1 + BN - 1) / BN;
  // Mask band (as in the 64/128 kernel): query i sees key j iff j <= i + off
  // (causal) and j > i + off - W (window); visited query blocks [qb0, qb_hi].
  const int off = p.bottom_right ? s2 - s1 : 0;
  const int W = p.window;
  const int qb0 = p.causal ? max(0, floordiv(static_cast<long long>(kvb) * BM - off, BN)) : 0;
  const int qb_hi = (p.causal && W > 0) ? min(n_qb - 1, floordiv(static_cast<long long>(kvb) * BM + BM - 2 - off + W, BN))
                                        : n_qb - 1;
  const int n_qit = max(0, qb_hi - qb0 + 1);
  const int n_it = G * n_qit;
  const int n_kvb = (s2 + BM - 1) / BM;
  const int nq_div = max(1, n_qit);
  auto qb_of = [&](int k) { return qb0 + k % nq_div; };
  auto hq_of = [&](int k) { return hk * G + k / nq_div; };
  const long long rs_kv = static_cast<long long>(p.heads_kv) * D;

  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC + 4);
  const uint32_t bars = sbase + L::BARS;
  auto bar = [&](int i) { return bars + 8u * i; };
  float* st_lse = reinterpret_cast<float*>(smem + L::STATS);          // [2][64]
  float* st_D = reinterpret_cast<float*>(smem + L::STATS + 512);      // [2][64]
  int* status = &g_bwd256_status;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(B_KV_FULL), 1);
    mbar_init(bar(B_KV_READY), 1);
    mbar_init(bar(B_V_DONE), 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_Q_FULL0 + s), 1);
      mbar_init(bar(B_Q_READY0 + s), 1);
      mbar_init(bar(B_Q_EMPTY0 + s), 1);
      mbar_init(bar(B_DO_FULL0 + s), 1);
      mbar_init(bar(B_DO_READY0 + s), 1);
      mbar_init(bar(B_DO_EMPTY0 + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_DP_FULL), 1);
    mbar_init(bar(B_P_READY), 256);
    mbar_init(bar(B_P_USED), 1);
    mbar_init(bar(B_DS_READY), 256);
    mbar_init(bar(B_DS_FREE), 1);
    mbar_init(bar(B_DQ_FULL), 1);
    mbar_init(bar(B_DQ_EMPTY), 128);
    mbar_init(bar(B_ACC_FULL), 1);
    mbar_init(bar(B_TEARDOWN), 1);
    mbar_init(bar(B_EPI0), 128);   // dV_c / dK_c tile staged by its warpgroup
    mbar_init(bar(B_EPI1), 128);
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
    // ------------------------------------------------------------ K / V producer
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
        mbar_arrive_expect_tx(bar(B_KV_FULL), 2 * TILE_K);
        for (int ch = 0; ch < 4; ++ch) {
          tma_load_2d(sbase + L::K + ch * CHUNK_K, &p.tm_k, hk * D + ch * 64, kv_start + kvb * BM, bar(B_KV_FULL));
          tma_load_2d(sbase + L::DO + ch * CHUNK_K, &p.tm_v, hk * D + ch * 64, kv_start + kvb * BM, bar(B_KV_FULL));
        }
      }
      __syncwarp();
      int pend_kv = 1;
      bool ok = mbar_wait(bar(B_KV_FULL), 0, abort, status);
      if (ok) {
        pend_kv = 0;
        // key rows past the sequence: dQ^T contracts over keys, and dS = 0
        // there does not cancel a NaN
        if (kv_valid < BM) {
          zero_rows(sbase + L::K, kv_valid, BM, CHUNK_K, lane);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_KV_READY));
      }
      volatile int no_abort = 0;
      if (pend_kv) mbar_wait(bar(B_KV_FULL), 0, &no_abort, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dO producer
    // (its own warp, so that Q and dO loads are issued independently)
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      int pend_do = -1;
      uint32_t par_do = 0;
      for (int k = 0; k < n_it; ++k) {
        const int s = k & 1;
        const uint32_t prev = ((k >> 1) - 1) & 1;
        const int qb = qb_of(k);
        const int q_valid = min(BN, s1 - qb * BN);
        // the dO stages hold V until warpgroup 0 has moved it into TMEM
        if (k == 0 && !mbar_wait(bar(B_V_DONE), 0, abort, status)) break;
        if (k >= 2 && !mbar_wait(bar(B_DO_EMPTY0 + s), prev, abort, status)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_DO_FULL0 + s), TILE_Q);
          for (int ch = 0; ch < 4; ++ch)
            tma_load_2d(sbase + L::DO + s * TILE_Q + ch * CHUNK_Q, &p.tm_do, hq_of(k) * D + ch * 64,
                        q_start + qb * BN, bar(B_DO_FULL0 + s));
        }
        pend_do = s;
        par_do = (k >> 1) & 1;
        if (!mbar_wait(bar(B_DO_FULL0 + s), (k >> 1) & 1, abort, status)) break;
        pend_do = -1;
        if (q_valid < BN) {
          zero_rows(sbase + L::DO + s * TILE_Q, q_valid, BN, CHUNK_Q, lane);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DO_READY0 + s));
      }
      volatile int no_abort = 0;
      if (pend_do >= 0) mbar_wait(bar(B_DO_FULL0 + pend_do), par_do, &no_abort, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, BN, 0, 0);     // S^T, dP^T
      constexpr uint32_t ID_KV = idesc_bf16(128, HALF, 0, 1);  // dV_c, dK_c: B MN-major
      constexpr uint32_t ID_DQ = idesc_bf16(128, BN, 1, 1);    // dQ_c^T: both MN-major
      const uint32_t t_v = tmem + COL_V, t_s = tmem + COL_S, t_dp = tmem + COL_DP;
      const uint32_t t_dv = tmem + COL_DV, t_dk = tmem + COL_DK;
      const uint32_t sK = sbase + L::K, sDS = sbase + L::DS;
      const uint32_t sKc = sK + 2 * c * CHUNK_K;               // this CTA's half of K
      bool ok = mbar_wait(bar(B_KV_READY), 0, abort, status) && mbar_wait(bar(B_Q_READY0), 0, abort, status);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          const uint64_t a0 = desc_k(sK, 0, CHUNK_K), b0 = desc_k(sbase + L::Q, 0, CHUNK_Q);
#pragma unroll 4
          for (int t = 0; t < D / 16; ++t)
            mma_ss(t_s, a0 + step_k(t, CHUNK_K), b0 + step_k(t, CHUNK_Q), ID_S, t > 0);
          mma_commit(bar(B_S_FULL));
        }
        __syncwarp();
        ok = mbar_wait(bar(B_V_DONE), 0, abort, status);
      }
      for (int k = 0; ok && k < n_it; ++k) {
        const int s = k & 1;
        const uint32_t ph = k & 1;
        const uint32_t sQ = sbase + L::Q + s * TILE_Q, sDO = sbase + L::DO + s * TILE_Q;
        // dP^T into the dP columns, free once the previous dQ_c^T is read out
        if (k > 0 && !mbar_wait(bar(B_DQ_EMPTY), (k - 1) & 1, abort, status)) { ok = false; break; }
        if (!mbar_wait(bar(B_DO_READY0 + s), (k >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t b0 = desc_k(sDO, 0, CHUNK_Q);
#pragma unroll 4
          for (int t = 0; t < D / 16; ++t) mma_ts(t_dp, t_v + t * 8, b0 + step_k(t, CHUNK_Q), ID_S, t > 0);
          mma_commit(bar(B_DP_FULL));
        }
        __syncwarp();
        // dV_c += P^T dO_i[:, half c]; P of query step t sits at column
        // 32*(t/2) + 8*(t%2) (each warpgroup packs its 32 columns' P into
        // the first 16 of them)
        if (!mbar_wait(bar(B_P_READY), ph, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t b0 = desc_mn(sDO + 2 * c * CHUNK_Q, 0, CHUNK_Q);
#pragma unroll
          for (int t = 0; t < BN / 16; ++t)
            mma_ts(t_dv, t_s + (t >> 1) * 32 + (t & 1) * 8, b0 + step_mn(t), ID_KV, (k > 0) | (t > 0));
          mma_commit(bar(B_P_USED));
          mma_commit(bar(B_DO_EMPTY0 + s));
        }
        __syncwarp();
        // next scores (need Q_{i+1} and P_i consumed) or this block's dK /
        // dQ (need dS_i), whichever is ready first; dK / dQ when both are
        {
          bool need_s = (k + 1 < n_it), need_c2 = true;
          const int s1n = (k + 1) & 1;
          const uint32_t qpar = ((k + 1) >> 1) & 1;
          const unsigned long long t0 = globaltimer();
          while (need_s || need_c2) {
            bool s_ready = need_s && mbar_test(bar(B_Q_READY0 + s1n), qpar) && mbar_test(bar(B_P_USED), ph);
            bool c_ready = need_c2 && mbar_test(bar(B_DS_READY), ph);
            s_ready = __shfl_sync(0xffffffffu, s_ready, 0);
            c_ready = __shfl_sync(0xffffffffu, c_ready, 0);
            if (s_ready && !c_ready) {
              tc_fence_after();
              if (elect_one()) {
                const uint32_t sQn = sbase + L::Q + s1n * TILE_Q;
                const uint64_t a0 = desc_k(sK, 0, CHUNK_K), b0 = desc_k(sQn, 0, CHUNK_Q);
#pragma unroll 4
                for (int t = 0; t < D / 16; ++t)
                  mma_ss(t_s, a0 + step_k(t, CHUNK_K), b0 + step_k(t, CHUNK_Q), ID_S, t > 0);
                mma_commit(bar(B_S_FULL));
              }
              __syncwarp();
              need_s = false;
            } else if (c_ready) {
              tc_fence_after();
              if (elect_one()) {
                // dK_c += dS^T Q_i[:, half c]   (A = dS, K-major over queries)
                const uint64_t a0 = desc_k(sDS, 0, CHUNK_K), b0 = desc_mn(sQ + 2 * c * CHUNK_Q, 0, CHUNK_Q);
#pragma unroll
                for (int t = 0; t < BN / 16; ++t)
                  mma_ss(t_dk, a0 + step_k(t, CHUNK_K), b0 + step_mn(t), ID_KV, (k > 0) | (t > 0));
                // dQ_c^T = K_c^T dS^T into the dP columns (both MN-major, K = keys)
                const uint64_t a1 = desc_mn(sKc, 0, CHUNK_K), b1 = desc_mn(sDS, 0, CHUNK_K);
#pragma unroll 4
                for (int t = 0; t < BM / 16; ++t) mma_ss(t_dp, a1 + step_mn(t), b1 + step_mn(t), ID_DQ, t > 0);
                mma_commit(bar(B_DQ_FULL));
                mma_commit(bar(B_Q_EMPTY0 + s));
                mma_commit(bar(B_DS_FREE));
              }
              __syncwarp();
              need_c2 = false;
            } else {
              const bool give_up = *abort || (globaltimer() - t0 > kWaitLimitNs);
              if (__shfl_sync(0xffffffffu, give_up, 0)) {
                if (lane == 0 && !*abort) {
                  atomicCAS(status, 0, kStatusTimeout);
                  *abort = 1;
                }
                ok = false;
                break;
              }
              // (polled without a sleep: a 32 ns sleep here cost 2.6 %)
            }
          }
          if (!ok) break;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (elect_one()) mma_commit(bar(ok ? B_ACC_FULL : B_TEARDOWN));
      __syncwarp();
      if (!ok) {
        volatile int no_abort = 0;
        mbar_wait(bar(B_TEARDOWN), 0, &no_abort, status);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax / dS
    setmaxnreg_to<kRegSoftmax, kRegLaunch>();
    const int wg = (warp - 4) >> 2;          // query columns [32 wg, 32 wg + 32)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // key row (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    if (wg == 0 && n_it > 0) {
      // V (staged in the dO stages by the producer) into TMEM columns
      // [0, 128): row r, bf16 pairs in order
      ok = mbar_wait(bar(B_KV_FULL), 0, abort, status);
      if (__all_sync(0xffffffffu, ok)) {
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t w[32];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 u = ld_shared_v4(sbase + L::DO + ch * CHUNK_K + r * 128 + ((g ^ (r & 7)) << 4));
            w[4 * g] = u.x;
            w[4 * g + 1] = u.y;
            w[4 * g + 2] = u.z;
            w[4 * g + 3] = u.w;
          }
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            w0[e] = w[e];
            w1[e] = w[16 + e];
          }
          tmem_st16(tmem + lane_addr + COL_V + ch * 32, w0);
          tmem_st16(tmem + lane_addr + COL_V + ch * 32 + 16, w1);
        }
        tmem_st_wait();
        fence_proxy_async_smem();   // the reads above come before TMA rewrites the stages
        tc_fence_before();
        mbar_arrive(bar(B_V_DONE));
      } else {
        ok = false;
      }
    }
    for (int k = 0; ok && k < n_it; ++k) {
      const int s = k & 1;
      const uint32_t ph = k & 1;
      const int qb = qb_of(k);
      int c_lo = 0, c_end = min(BN, s1 - qb * BN);
      if (p.causal) {
        const long long d0 = static_cast<long long>(kvb) * BM + r - off - static_cast<long long>(qb) * BN;
        c_lo = static_cast<int>(max(0LL, min(d0, static_cast<long long>(BN))));
        if (W > 0) c_end = static_cast<int>(max(0LL, min(static_cast<long long>(c_end), d0 + W)));
      }
      const int span = (r < kv_valid) ? max(0, c_end - c_lo) : 0;
      const int qc0 = wg * 32;
      const bool need_mask = __any_sync(0xffffffffu, c_lo > qc0 || c_lo + span < qc0 + 32);
      if (!mbar_wait(bar(B_Q_READY0 + s), (k >> 1) & 1, abort, status)) { ok = false; break; }
      const float4* lse4 = reinterpret_cast<const float4*>(st_lse + s * BN + qc0);
      const float4* dvec4 = reinterpret_cast<const float4*>(st_D + s * BN + qc0);
      float4 lv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) lv[i] = lse4[i];
      if (!mbar_wait(bar(B_S_FULL), ph, abort, status)) { ok = false; break; }
      tc_fence_after();
      float P[32];
      {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + COL_S + qc0, v);
        tmem_ld_wait();
        uint32_t pk[16];
        // masked and unmasked blocks as separate instantiations: no
        // per-element mask work where every column is visible
        auto p_loop = [&](auto mask_tag) {
          constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float la[4] = {lv[c4].x, lv[c4].y, lv[c4].z, lv[c4].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = c4 * 4 + e;
              float pv = ex2_approx(fmaf(__uint_as_float(v[col]), sl2, -la[e]));
              if (MASK) {
                const bool vis = static_cast<unsigned>(qc0 + col - c_lo) < static_cast<unsigned>(span);
                pv = vis ? pv : 0.f;
              }
              P[col] = pv;
            }
          }
        };
        if (need_mask)
          p_loop(std::true_type{});
        else
          p_loop(std::false_type{});
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(P[2 * j], P[2 * j + 1]);
        tmem_st16(tmem + lane_addr + COL_S + qc0, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(B_P_READY));

      float4 dv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) dv[i] = dvec4[i];
      if (!mbar_wait(bar(B_DP_FULL), ph, abort, status)) { ok = false; break; }
      if (k > 0 && !mbar_wait(bar(B_DS_FREE), (k - 1) & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + COL_DP + qc0, v);
        tmem_ld_wait();
        uint32_t pk[16];
        auto ds_loop = [&](auto mask_tag) {
          constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float da[4] = {dv[c4].x, dv[c4].y, dv[c4].z, dv[c4].w};
            float ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = c4 * 4 + e;
              ds[e] = P[col] * (__uint_as_float(v[col]) - da[e]);
              if (MASK) ds[e] = (P[col] != 0.f) ? ds[e] : 0.f;   // dP may hold garbage where masked
            }
            pk[2 * c4] = pack_bf16x2(ds[0], ds[1]);
            pk[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
          }
        };
        if (need_mask)
          ds_loop(std::true_type{});
        else
          ds_loop(std::false_type{});
        const uint32_t ds_row = sbase + L::DS + r * 128;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int gg = wg * 4 + g;   // 16-byte granule of the 128-byte row
          st_shared_v4(ds_row + ((gg ^ (r & 7)) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_DS_READY));
    }
    // ------------------------------------------------------------ dV_c / dK_c epilogue
    const int kv_row = kv_start + kvb * BM + r;
    uint16_t* out = (wg == 0) ? p.dv : p.dk;
    const float mul = (wg == 0) ? 1.f : p.scale;
    uint8_t* dst = reinterpret_cast<uint8_t*>(out + static_cast<long long>(kv_row) * rs_kv + hk * D + c * HALF);
    if (n_it == 0) {
      if (r < kv_valid)
        for (int cc = 0; cc < HALF; cc += 8) st_global_v4(dst + cc * 2, 0u, 0u, 0u, 0u);
    } else if (__all_sync(0xffffffffu, ok && mbar_wait(bar(B_ACC_FULL), 0, abort, status))) {
      tc_fence_after();
      const uint32_t col0 = (wg == 0) ? COL_DV : COL_DK;
      if (kv_valid == BM) {
        // A whole key block: dV_c (warpgroup 0) / dK_c (1) staged as bf16 in
        // two 64-column chunks of the K tile, which no MMA reads any more,
        // and written by TMA; a partial block is written per row below, so
        // that no row of the next sequence is touched.
        const uint32_t tile = sbase + L::K + wg * 2 * CHUNK_K;
        const uint32_t row = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll 1
        for (int ch = 0; ch < HALF / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + col0 + ch * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(mul * __uint_as_float(v[g * 8 + 2 * e]), mul * __uint_as_float(v[g * 8 + 2 * e + 1]));
            const int u = (ch & 1) * 4 + g;   // 16-byte unit within the 128-byte row of a 64-column chunk
            st_shared_v4(row + (ch >> 1) * CHUNK_K + ((u ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_EPI0 + wg));
        // One thread per warpgroup waits (bounded) for the other 127 rows.
        if (quarter == 0 && lane == 0 && mbar_wait(bar(B_EPI0 + wg), 0, abort, status)) {
          for (int cc = 0; cc < 2; ++cc)
            tma_store_2d((wg == 0) ? &p.tm_dv : &p.tm_dk, tile + cc * CHUNK_K, hk * D + c * HALF + cc * 64,
                         kv_start + kvb * BM);
          bulk_commit();
          bulk_wait_read0();   // the tile is read before the CTA exits
        }
      } else {
#pragma unroll 1
        for (int ch = 0; ch < HALF / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + col0 + ch * 32, v);
          tmem_ld_wait();
          if (r < kv_valid) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(mul * __uint_as_float(v[g * 8 + 2 * e]), mul * __uint_as_float(v[g * 8 + 2 * e + 1]));
              st_global_v4(dst + (ch * 32 + g * 8) * 2, w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ_c write-back
    setmaxnreg_to<kRegDrain, kRegLaunch>();
    const int quarter = warp & 3;            // head dims [32 quarter, +32) of half c: one staging box
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t slot = sbase + L::DQST + quarter * 4096;
    const bool det = p.dq_mode != 0;
    bool issued = false;
    for (int k = 0; k < n_it; ++k) {
      const int qb = qb_of(k);
      const int hq = hq_of(k);
      const int y0 = q_start + qb * BN;
      const int x = hq * D + c * HALF + quarter * 32;
      int* ticket = det ? p.tickets + ((static_cast<long long>(b * H + hq) * p.max_q_blocks + qb) * 2 + c) * 4 + quarter
                        : nullptr;
      if (!mbar_wait(bar(B_DQ_FULL), k & 1, abort, status)) break;
      tc_fence_after();
      uint32_t va[32], vb[32];
      tmem_ld32(tmem + lane_addr + COL_DP, va);        // queries 0..31 of the block
      tmem_ld32(tmem + lane_addr + COL_DP + 32, vb);   // queries 32..63
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_DQ_EMPTY));
      bool turn = true;
      if (lane == 0 && det) {
        const long long q0 = static_cast<long long>(qb) * BN;
        const int kb_hi = p.causal ? min(n_kvb - 1, floordiv(q0 + BN - 1 + off, BM)) : n_kvb - 1;
        const int kb_lo = (p.causal && W > 0) ? max(0, floordiv(q0 + off - W + 1, BM)) : 0;
        const int before = p.kv_reverse ? kb_hi - kvb : kvb - kb_lo;
        turn = wait_counter(ticket, before, abort, status);
        fence_proxy_async_global();
      }
      turn = __shfl_sync(0xffffffffu, turn, 0);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (issued) {
          if (lane == 0) bulk_wait_read0();   // the box's previous contents have been read
          __syncwarp();
        }
        // transpose: lane = head dim, 32 queries -> rows of a [32, 32] fp32
        // box with 128-byte swizzle
#pragma unroll
        for (int qq = 0; qq < 32; ++qq) {
          const uint32_t val = half ? vb[qq] : va[qq];
          st_shared_b32(slot + qq * 128 + ((((lane >> 2) ^ (qq & 7))) << 4) + (lane & 3) * 4, val);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && turn) {
          tma_reduce_add_2d(&p.tm_dq, slot, x, y0 + half * 32);
          bulk_commit();
        }
        issued = issued || turn;
      }
      if (lane == 0 && det && turn) {
        bulk_wait_all0();
        fence_proxy_async_global();
        __threadfence();
        atomicAdd(ticket, 1);
      }
      if (!turn) break;
      __syncwarp();
    }
    if (lane == 0 && issued) bulk_wait_all0();
  } else {
    // ------------------------------------------------------------ Q producer (warp 3)
    // (its own warp, so that the first Q block loads alongside K and V)
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      // a load issued but not seen complete must land before the CTA exits
      int pend_q = -1;
      uint32_t par_q = 0;
      bool ok = true;
      float nm[2], nl[2], nd[2], rm[2], rl[2], rd[2];
      auto load_stats = [&](int k, float (&a)[2], float (&bb)[2], float (&cc)[2]) {
        const int qb = qb_of(k);
        const int q_valid = min(BN, s1 - qb * BN);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int r = lane + 32 * j;
          a[j] = 0.f;
          bb[j] = 1.f;
          cc[j] = 0.f;
          if (k < n_it && r < q_valid) {
            const long long idx = static_cast<long long>(q_start + qb * BN + r) * H + hq_of(k);
            a[j] = __ldg(p.m + idx);
            if (!p.stats_lse) bb[j] = __ldg(p.l + idx);
            cc[j] = __ldg(p.D + idx);
          }
        }
      };
      load_stats(0, nm, nl, nd);
      for (int k = 0; ok && k < n_it; ++k) {
        const int s = k & 1;
        const uint32_t prev = ((k >> 1) - 1) & 1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          rm[j] = nm[j];
          rl[j] = nl[j];
          rd[j] = nd[j];
        }
        load_stats(k + 1, nm, nl, nd);
        const int qb = qb_of(k);
        const int hq = hq_of(k);
        const int q_row0 = q_start + qb * BN;
        const int q_valid = min(BN, s1 - qb * BN);
        if (k >= 2 && !mbar_wait(bar(B_Q_EMPTY0 + s), prev, abort, status)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_Q_FULL0 + s), TILE_Q);
          for (int ch = 0; ch < 4; ++ch)
            tma_load_2d(sbase + L::Q + s * TILE_Q + ch * CHUNK_Q, &p.tm_q, hq * D + ch * 64, q_row0,
                        bar(B_Q_FULL0 + s));
        }
        pend_q = s;
        par_q = (k >> 1) & 1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          st_lse[s * BN + lane + 32 * j] = rm[j] * 1.4426950408889634f + (p.stats_lse ? 0.f : __log2f(rl[j]));
          st_D[s * BN + lane + 32 * j] = rd[j];
        }
        if (!mbar_wait(bar(B_Q_FULL0 + s), (k >> 1) & 1, abort, status)) break;
        pend_q = -1;
        if (q_valid < BN) {
          zero_rows(sbase + L::Q + s * TILE_Q, q_valid, BN, CHUNK_Q, lane);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_Q_READY0 + s));
      }
      volatile int no_abort = 0;
      if (pend_q >= 0) mbar_wait(bar(B_Q_FULL0 + pend_q), par_q, &no_abort, status);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_bwd256(const BwdParams& p, int batch, int max_kv_blocks, cudaStream_t s) {
  if (batch <= 0 || max_kv_blocks <= 0) return cudaSuccess;
  constexpr uint32_t bytes = Layout::BYTES;
  static_assert(bytes <= 232448, "shared memory budget");
  static std::atomic<unsigned long long> smem_set{0}, smem_set_chunked{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(bwd256_kernel<false>), (int)bytes, smem_set);
  if (e == cudaSuccess) e = set_smem_once(reinterpret_cast<const void*>(bwd256_kernel<true>), (int)bytes, smem_set_chunked);
  if (e != cudaSuccess) return e;
  if (2LL * max_kv_blocks * p.heads_kv * batch > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  BwdParams q = p;
  q.batch = batch;
  q.grid_kv = max_kv_blocks;
  q.head_chunk = launch_head_chunk(p, batch, max_kv_blocks, BM, BN, D);
  dim3 grid(max_kv_blocks, p.heads_kv, 2 * batch);
  if (q.head_chunk > 1)
    bwd256_kernel<true><<<grid, kThreads, bytes, s>>>(q);
  else
    bwd256_kernel<false><<<grid, kThreads, bytes, s>>>(q);
  return cudaGetLastError();
}

int bwd256_read_and_clear_status(cudaStream_t s, int* status) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_bwd256_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_bwd256_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return static_cast<int>(e);
}

}  // namespace fa
