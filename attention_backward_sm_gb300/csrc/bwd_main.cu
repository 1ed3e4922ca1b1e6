// Single-pass flash-attention backward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes follows the SK-16 single-pass FA Grad article: section 3
// (skeleton C1 -> V1 -> C2 -> V2), section 3.1 (the eight per-block steps),
// section 4.1 (m and l are consumed, never recomputed) and section 4.2
// (bf16 operands, fp32 scores/softmax, P and dS rounded to bf16 before the
// second group of matmuls, fp32 accumulation of dK, dV, dQ).  The loop order
// is the key-block-outer one that section 1 names as best for dK/dV: a CTA
// owns one (sequence, head, 128-row key block), keeps dK and dV in tensor
// memory across its whole query sweep and adds each dQ partial into an
// fp32 accumulator in global memory (section 3, V2 atomic write-back,
// restricted to dQ).
//
// Per query block i (128 rows), with the key block j fixed (128 rows):
//   C1   S^T  = K_j Q_i^T              (TMEM cols [0,128), fp32)
//        dP^T = V_j dO_i^T             (TMEM cols [128,256))
//   V1   P    = exp2(S*scale*log2e - (m*log2e + log2 l))  (= exp(S*scale-m)/l)
//        dS   = P * (dP - D)           masked entries exactly 0
//        P  -> bf16 into TMEM cols [0,32) and [64,96) (A operand of dV)
//        dS -> bf16 into shared memory (operand of dK and dQ)
//   C2   dV_j += P^T dO_i              (TMEM cols [256, 256+d))
//        dK_j += dS^T Q_i              (TMEM cols [256+d, 256+2d))
//        dQ_i partial = dS K_j         (query rows on lanes; reuses the dP columns)
//   V2   dq_acc[rows of i] += partial  (TMA tensor reduce-add from a swizzled
//                                      shared-memory copy; scale applied later)
// Transposed scores put key rows on TMEM lanes, so the softmax threads own
// whole key rows and P / dS come out already in the layouts the C2 MMAs
// want.  The MMA order inside one query block is dP_i, dV_i, S_{i+1},
// dK_i, dQ_i: the next block's scores are computed while the softmax
// warps derive dS_i.
//
// Warp roles (512 threads; registers per thread set per warpgroup: 56 for
// warps 0-3, 152 for the softmax warpgroups, 152 for the write-back, which
// holds a whole 128-column dQ partial; the sum is exactly the 65536 the
// block is launched with):
//   warp 0      TMA producer of K and V (once per CTA); d = 128 without
//               the dQ partials: then also of the per-row stats
//   warp 3      TMA producer of Q and the per-row stats (2- or 3-stage
//               ring), so that the first Q block loads alongside K and V
//               (d = 128 without a mask: from the third block on, the Q
//               load itself is issued by write-back warp 12, see below)
//   warp 2      TMA producer of dO (2-stage ring)
//               (each producer zeroes tile rows past a sequence end)
//   warp 1      TMEM allocator and MMA issuer (one elected lane issues)
//   warps 4-11  two softmax warpgroups, each owning 64 of the 128 query
//               columns for all 128 key rows; at the end dV (4-7), dK (8-11)
//   warps 12-15 dQ write-back: TMEM -> shared memory (d = 128: the block's
//               Q and dO buffers, which the MMAs are done with; d = 64: a
//               staging area of its own) -> TMA reduce-add
// The dK / dV epilogue of a whole key block at d = 128 goes through the dead
// K / V tiles and TMA stores; otherwise each thread stores its own row.
// Every mbarrier wait is bounded (see sm103.cuh); on a timeout the CTA
// records FA_ERR_TIMEOUT in the status word, drains and frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "sm103.cuh"

namespace fa {

__device__ int g_bwd_status = 0;

namespace {

constexpr int kThreads = 512;
// Registers per thread: the block launches with 65536 / 512 = 128 and each
// warpgroup then moves to its own budget.
constexpr uint32_t kRegLaunch = 65536 / kThreads;
constexpr uint32_t kRegOther = 56;     // warps 0-3: producers and MMA issuer
constexpr uint32_t kRegSoftmax = 152;  // warps 4-11
constexpr uint32_t kRegDrain = 152;    // warps 12-15
static_assert(128 * kRegOther + 256 * kRegSoftmax + 128 * kRegDrain <= 65536, "register budgets exceed the launch");
constexpr int BM = 128;   // key rows per CTA
constexpr int BN = 128;   // query rows per block
constexpr uint32_t CHUNK = 128 * 128;   // one TMA box: 128 rows x 64 bf16 (128 B)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_DP = 128;
constexpr uint32_t COL_DV = 256;

// mbarrier slots
enum {
  B_KV_FULL = 0, B_KV_READY,
  B_Q_FULL0, B_Q_READY0 = B_Q_FULL0 + 3, B_Q_EMPTY0 = B_Q_READY0 + 3,   // up to 3 Q stages
  B_DO_FULL0 = B_Q_EMPTY0 + 3,
  B_DO_FULL1, B_DO_READY0, B_DO_READY1, B_DO_EMPTY0, B_DO_EMPTY1,
  B_S_FULL, B_DP_FULL, B_P_READY, B_P_USED, B_DS_READY, B_DS_FREE, B_DQ_FULL, B_DQ_EMPTY, B_ACC_FULL,
  B_TEARDOWN, B_EPI0, B_EPI1, B_Q_ISSUED0, B_Q_ISSUED1, B_ST_READY0, B_ST_READY1, B_ST_READY2, NUM_BARS
};

// Where a dQ partial lives on its way to TMA.  d = 128: tensor memory is
// full (S, dP, dV, dK take 128 columns each), so the partial is computed
// into the dP columns, and shared memory is full too, so it is staged half in
// the block's own Q buffer (dead once dK has run) and half in its dO buffer
// (dead after dV).  d = 64: the partial has 64 tensor-memory columns of its
// own, so the next dP does not wait for it to be read out, and a 32 KB
// staging area of its own, so no operand buffer waits for TMA to read it.
template <int D>
constexpr bool kOwnDQ = (D == 64);
// Q stages (with their row statistics).  A Q load is issued once the
// stage's previous block has run dK and takes a few thousand cycles to land
// behind the dQ reduce-adds on the SM's TMA engine; with d = 64 there is room
// for a third stage, so the load has two blocks' time instead of one.
template <int D>
constexpr int kQStages = kOwnDQ<D> ? 3 : 2;

template <int D>
struct Layout {
  static constexpr uint32_t TILE = 128 * D * 2;   // [128 rows, D] bf16
  static constexpr int NCH = D / 64;              // 64-column chunks per tile
  static constexpr uint32_t K = 0;
  static constexpr uint32_t V = TILE;
  static constexpr uint32_t Q = 2 * TILE;         // kQStages stages
  static constexpr uint32_t DO = Q + kQStages<D> * TILE;   // 2 stages
  static constexpr uint32_t DS = DO + 2 * TILE;   // [128 key rows, 128 query cols] bf16 = 32 KB
  static constexpr uint32_t STG = DS + 32768;     // d = 64: dQ staging, [128 rows, 64] fp32 as 32x32 boxes
  static constexpr uint32_t STATS = STG + (kOwnDQ<D> ? 32768 : 0);   // lse2[stage][128], then D[stage][128] (fp32)
  static constexpr uint32_t STATS_D = STATS + kQStages<D> * 128 * 4;
  static constexpr uint32_t BARS = STATS + kQStages<D> * 2 * 128 * 4;
  static constexpr uint32_t MISC = BARS + NUM_BARS * 8;   // abort flag, TMEM address
  static constexpr uint32_t BYTES = MISC + 16;
  static constexpr uint32_t COL_DK = COL_DV + D;
  static constexpr uint32_t COL_DQ = kOwnDQ<D> ? COL_DV + 2 * D : COL_DP;   // dQ partial
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int t) {
  // 16-element K step t inside a [rows, K] tile stored as 64-column chunks
  return sw128_desc(tile + (t >> 2) * CHUNK + (t & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int t) {
  // rows 16t..16t+15 of a [K rows, MN] tile; MN chunks of 64 are CHUNK apart
  return sw128_desc(tile + t * 2048, CHUNK, 1024);
}

// MMA groups over N 16-element K steps, issued by one thread.  The
// descriptors of a group are built once and stepped by constants (the start
// address sits in the descriptor's low 14 bits as addr >> 4, and every step
// stays inside the tile), so each MMA costs the issuing warp a 64-bit add.
// acc: whether the first step accumulates into D.
__device__ __forceinline__ constexpr uint64_t step_kmajor(int t) { return ((t >> 2) * CHUNK + (t & 3) * 32) >> 4; }
__device__ __forceinline__ constexpr uint64_t step_mnmajor(int t) { return (t * 2048) >> 4; }
template <int N>
__device__ __forceinline__ void mmas_kk(uint32_t d, uint32_t a_tile, uint32_t b_tile, uint32_t idesc, uint32_t acc) {
  const uint64_t a0 = desc_kmajor(a_tile, 0), b0 = desc_kmajor(b_tile, 0);
#pragma unroll 4
  for (int t = 0; t < N; ++t) mma_ss(d, a0 + step_kmajor(t), b0 + step_kmajor(t), idesc, acc | (t > 0));
}
template <int N>
__device__ __forceinline__ void mmas_km(uint32_t d, uint32_t a_tile, uint32_t b_tile, uint32_t idesc, uint32_t acc) {
  const uint64_t a0 = desc_kmajor(a_tile, 0), b0 = desc_mnmajor(b_tile, 0);
#pragma unroll 4
  for (int t = 0; t < N; ++t) mma_ss(d, a0 + step_kmajor(t), b0 + step_mnmajor(t), idesc, acc | (t > 0));
}
template <int N>
__device__ __forceinline__ void mmas_mm(uint32_t d, uint32_t a_tile, uint32_t b_tile, uint32_t idesc, uint32_t acc) {
  const uint64_t a0 = desc_mnmajor(a_tile, 0), b0 = desc_mnmajor(b_tile, 0);
#pragma unroll 4
  for (int t = 0; t < N; ++t) mma_ss(d, a0 + step_mnmajor(t), b0 + step_mnmajor(t), idesc, acc | (t > 0));
}
// A from TMEM: P of K step t sits at column 64*(t/4) + 8*(t%4) (each softmax
// warpgroup keeps its 64 query columns' P in the first 32 of its 64 columns).
template <int N>
__device__ __forceinline__ void mmas_tm(uint32_t d, uint32_t a_tmem, uint32_t b_tile, uint32_t idesc, uint32_t acc) {
  const uint64_t b0 = desc_mnmajor(b_tile, 0);
#pragma unroll 4
  for (int t = 0; t < N; ++t)
    mma_ts(d, a_tmem + (t >> 2) * 64 + (t & 3) * 8, b0 + step_mnmajor(t), idesc, acc | (t > 0));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Zero rows [first, 128) of a [128, D] tile (all chunks) with the 32 lanes
// of one warp.  Each row of a chunk is one contiguous 128-byte line.
template <int D>
__device__ __forceinline__ void zero_rows(uint32_t tile, int first, int lane) {
  constexpr int NCH = D / 64;
  const int nrows = 128 - first;
  for (int e = lane; e < nrows * NCH * 8; e += 32) {
    const int row = first + e / (NCH * 8);
    const int rem = e % (NCH * 8);
    const int ch = rem / 8, g = rem % 8;
    st_shared_v4(tile + ch * CHUNK + row * 128 + g * 16, 0u, 0u, 0u, 0u);
  }
}

// P phase of one softmax thread: key row r, this warpgroup's 64 query
// columns.  Reads S^T from TMEM (taddr = row's lane, first column), forms
// P = 2^(S*scale*log2e - lse2) (= exp(S*scale - m) / l), zeroes masked
// entries when MASK, and stores P as bf16 into the first 32 of the 64
// columns just read.  MASK is a template parameter so that full blocks run
// a loop without any per-element mask work.  Every mask (tails, causal
// in either alignment, sliding window) leaves key row r a single run of
// visible query columns of the tile: [c_lo, c_lo + span) (span <= 0: none).
// lse4: the 64 per-column values -lse2 in shared memory; pre: the first 32
// of them, read earlier.  The second 32 are read while the first TMEM load
// is in flight.
template <bool MASK>
__device__ __forceinline__ void softmax_p(uint32_t taddr, const float4* lse4, const float4 (&pre)[8], float sl2,
                                          float (&P)[64], int qc0, int c_lo, int span) {
  float4 nxt[8];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t v[32];
    tmem_ld32(taddr + half * 32, v);
    if (half == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) nxt[i] = lse4[8 + i];
    }
    tmem_ld_wait();
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
      const float4 lv = half == 0 ? pre[c4] : nxt[c4];   // -lse2 of 4 columns
      // exponent arguments two at a time (packed fp32 FMA)
      const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(v[c4 * 4]), __uint_as_float(v[c4 * 4 + 1])),
                                    make_float2(sl2, sl2), make_float2(lv.x, lv.y));
      const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(v[c4 * 4 + 2]), __uint_as_float(v[c4 * 4 + 3])),
                                    make_float2(sl2, sl2), make_float2(lv.z, lv.w));
      const float xs[4] = {x01.x, x01.y, x23.x, x23.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = half * 32 + c4 * 4 + e;
        float pv = ex2_approx(xs[e]);
        if (MASK) {
          const bool vis = static_cast<unsigned>(qc0 + col - c_lo) < static_cast<unsigned>(span);
          pv = vis ? pv : 0.f;
        }
        P[col] = pv;
      }
    }
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(P[half * 32 + 2 * j], P[half * 32 + 2 * j + 1]);
    tmem_st16(taddr + half * 16, pk);
  }
  tmem_st_wait();
}

// dS phase of one softmax thread: dS = P * (dP - D) from dP^T in TMEM,
// rounded to bf16 and written as row r of the 128B-swizzled dS tile.
// dvec4: the 64 per-column values -D in shared memory; pre: the first 32.
template <bool MASK>
__device__ __forceinline__ void softmax_ds(uint32_t taddr, const float4* dvec4, const float4 (&pre)[8],
                                           const float (&P)[64], uint32_t ds_row, int r) {
  float4 nxt[8];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t v[32];
    tmem_ld32(taddr + half * 32, v);
    if (half == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) nxt[i] = dvec4[8 + i];
    }
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
      const float4 dv4 = half == 0 ? pre[c4] : nxt[c4];   // -D of 4 columns
      const int c0 = half * 32 + c4 * 4;
      // dS = P * (dP - D), two at a time (packed fp32 add and multiply)
      const float2 d01 = __fmul2_rn(make_float2(P[c0], P[c0 + 1]),
                                    __fadd2_rn(make_float2(__uint_as_float(v[c4 * 4]), __uint_as_float(v[c4 * 4 + 1])),
                                               make_float2(dv4.x, dv4.y)));
      const float2 d23 = __fmul2_rn(make_float2(P[c0 + 2], P[c0 + 3]),
                                    __fadd2_rn(make_float2(__uint_as_float(v[c4 * 4 + 2]), __uint_as_float(v[c4 * 4 + 3])),
                                               make_float2(dv4.z, dv4.w)));
      float ds[4] = {d01.x, d01.y, d23.x, d23.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // P is already 0 where masked, but dP may hold garbage there.
        if (MASK) ds[e] = (P[c0 + e] != 0.f) ? ds[e] : 0.f;
      }
      pk[2 * c4] = pack_bf16x2(ds[0], ds[1]);
      pk[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int gg = half * 4 + g;            // 16-byte granule within the 128-byte row
      st_shared_v4(ds_row + ((gg ^ (r & 7)) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
    }
  }
}

// Floor of a / b for b > 0 and any sign of a.
__device__ __forceinline__ int floordiv(long long a, int b) {
  long long q = a / b;
  if ((a % b) != 0 && a < 0) --q;
  return static_cast<int>(q);
}

// kDQ: also compute the dQ partials and add them into dq_acc (any order);
// without it the kernel computes dK and dV only (the deterministic mode,
// whose dQ comes from dq_kernel), and the dP columns, the Q buffers and
// the dO buffers are released as soon as the MMAs are done with them.
template <int D, bool kChunked, bool kDQ>
__global__ void __launch_bounds__(kThreads, 1) bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = Layout<D>;
  // dP columns, Q and dO buffers free of dQ partials (d = 64 keeps its
  // partial in columns and a staging area of its own)
  constexpr bool kSep = kOwnDQ<D> || !kDQ;
  // d = 128 with the dQ partial staged in the Q / dO buffers, no mask: the
  // Q load of block k + NQS is issued by a write-back warp once TMA has read
  // the half staged in that Q buffer and before the half staged in the dO
  // buffer is reduce-added, so that it does not queue behind 32 KB of
  // write-out on the SM's TMA engine (cfg3-nc +0.7 %; under a causal mask
  // the later release of the dO buffer cost 2 %, so masked sweeps keep the
  // producer's own order)
  const bool q_by_drain = kDQ && !kOwnDQ<D> && !p.causal;
  // d = 128 without the dQ partials (the deterministic mode): the row
  // statistics come from the K / V producer, idle once K and V have landed,
  // so that the Q producer issues each Q load without waiting on the
  // statistics' global loads (cfg3 +2.7 %, cfg3-nc +2.3 %; with the dQ
  // partials, and at d = 64, the Q producer keeping them measured faster)
  constexpr bool kStatsW0 = !kDQ && D == 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Launch order.  Unchunked (head_chunk = 1): the grid is (key block,
  // key/value head, sequence), key block fastest.  Chunked: the linear block
  // index takes the (sequence, key/value head) units in chunks of head_chunk
  // with the key block as the slow index within a chunk, so under a causal
  // mask the long sweeps of the low key blocks start first and the short ones
  // fill the tail, while the chunk's query-side data stays in L2.
  int kvb, hk, b;
  if constexpr (!kChunked) {
    kvb = static_cast<int>(blockIdx.x);
    hk = blockIdx.y;
    b = blockIdx.z;
  } else {
    const int lin = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    const int units = p.heads_kv * p.batch;
    const int per_chunk = p.head_chunk * p.grid_kv;
    const int ch = lin / per_chunk;
    const int r = lin - ch * per_chunk;
    const int g = min(p.head_chunk, units - ch * p.head_chunk);
    const int x = r / g;
    const int unit = ch * p.head_chunk + (r - x * g);
    kvb = x;
    hk = unit % p.heads_kv;
    b = unit / p.heads_kv;
  }
  // Grouped-query attention: the CTA owns key/value head hk, shared by the
  // G query heads hk*G .. hk*G+G-1, and sweeps the query blocks of each of
  // them in turn; dK and dV accumulate over the whole group in TMEM.
  const int H = p.heads;                            // query heads
  const int G = p.heads / p.heads_kv;
  const int q_start = p.cu_q[b], s1 = p.cu_q[b + 1] - q_start;
  const int kv_start = p.cu_kv[b], s2 = p.cu_kv[b + 1] - kv_start;
  if (kvb * BM >= s2) return;                       // CTA-uniform, before any barrier
  if (sbase & 1023) {                               // swizzled tiles need 1 KB alignment
    if (threadIdx.x == 0) atomicCAS(&g_bwd_status, 0, 99);
    return;
  }
  const int kv_valid = min(BM, s2 - kvb * BM);
  const int n_qb = (s1 + BN - 1) / BN;
  // Mask band: query i sees key j iff j <= i + off (causal) and
  // j > i + off - W (window W > 0); off = s2 - s1 for the bottom-right
  // alignment, else 0.  A tile (query block, key block) is visited iff the
  // band meets it; this key block's visited query blocks are [qb0, qb_hi].
  const int off = p.bottom_right ? s2 - s1 : 0;
  const int W = p.window;
  const int qb0 = p.causal ? max(0, floordiv(static_cast<long long>(kvb) * BM - off, BN)) : 0;
  const int qb_hi = (p.causal && W > 0) ? min(n_qb - 1, floordiv(static_cast<long long>(kvb) * BM + BM - 2 - off + W, BN))
                                        : n_qb - 1;
  const int n_qit = max(0, qb_hi - qb0 + 1);        // query blocks per query head
  const int n_it = G * n_qit;                       // iterations of the sweep
  const int nq_div = max(1, n_qit);                 // divisor that stays valid when there is no work
  auto qb_of = [&](int k) { return qb0 + k % nq_div; };
  auto hq_of = [&](int k) { return hk * G + k / nq_div; };
  const long long rs_kv = static_cast<long long>(p.heads_kv) * D;   // key-side row stride (elements)

  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC + 4);
  const uint32_t bars = sbase + L::BARS;
  auto bar = [&](int i) { return bars + 8u * i; };
  float* st_lse = reinterpret_cast<float*>(smem + L::STATS);          // [kQStages][128]
  float* st_D = reinterpret_cast<float*>(smem + L::STATS_D);          // [kQStages][128]
  // Raw row statistics (m, l, D) of a block are loaded one block ahead
  // into registers (lane + 32 j holds row j of the lane) and only combined
  // (lse2 = m*log2(e) + log2(l)) when stored, so that their latency hides
  // behind the waits of the current block.
  auto load_stats = [&](int k, float (&a)[4], float (&b)[4], float (&c)[4]) {
    const int qb = qb_of(k);
    const int q_valid = min(BN, s1 - qb * BN);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = lane + 32 * j;
      a[j] = 0.f;
      b[j] = 1.f;
      c[j] = 0.f;
      if (k < n_it && r < q_valid) {
        const long long idx = static_cast<long long>(q_start + qb * BN + r) * H + hq_of(k);
        a[j] = __ldg(p.m + idx);
        if (!p.stats_lse) b[j] = __ldg(p.l + idx);
        c[j] = __ldg(p.D + idx);
      }
    }
  };
  auto store_stats = [&](int s, const float (&a)[4], const float (&b)[4], const float (&c)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // log2 of the softmax denominator, exp(x - m) / l = 2^(x*log2e - lse2),
      // stored negated: the softmax adds them with packed FMAs / adds
      st_lse[s * 128 + lane + 32 * j] = -(a[j] * 1.4426950408889634f + (p.stats_lse ? 0.f : __log2f(b[j])));
      st_D[s * 128 + lane + 32 * j] = -c[j];
    }
  };
  constexpr int NQS = kQStages<D>;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(B_KV_FULL), 1);
    mbar_init(bar(B_KV_READY), 1);
    for (int s = 0; s < NQS; ++s) {
      mbar_init(bar(B_Q_FULL0 + s), 1);
      mbar_init(bar(B_Q_READY0 + s), 1);
      mbar_init(bar(B_ST_READY0 + s), 1);   // (kStatsW0) the stage's row statistics written
      // released by the four write-back warps where they stage a dQ half in
      // it (d = 128), else by the MMA commit after the block's last use
      mbar_init(bar(B_Q_EMPTY0 + s), kSep ? 1 : 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_DO_FULL0 + s), 1);
      mbar_init(bar(B_DO_READY0 + s), 1);
      mbar_init(bar(B_DO_EMPTY0 + s), kSep ? 1 : 4);
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
    mbar_init(bar(B_EPI0), 128);   // dV / dK tile staged by its warpgroup
    mbar_init(bar(B_EPI1), 128);
    // (d = 128, atomic, no mask) the next Q load is issued; two, by block
    // parity, so that warp 12 cannot complete the phase of block i + 1
    // before warps 13-15 have waited for that of block i
    mbar_init(bar(B_Q_ISSUED0), 1);
    mbar_init(bar(B_Q_ISSUED1), 1);
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
  int* status = &g_bwd_status;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
        mbar_arrive_expect_tx(bar(B_KV_FULL), 2 * L::TILE);
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_2d(sbase + L::K + c * CHUNK, &p.tm_k, hk * D + c * 64, kv_start + kvb * BM, bar(B_KV_FULL));
          tma_load_2d(sbase + L::V + c * CHUNK, &p.tm_v, hk * D + c * 64, kv_start + kvb * BM, bar(B_KV_FULL));
        }
      }
      __syncwarp();
      // (kStatsW0) the row statistics are loaded here.
      float rm[4], rl[4], rd[4], nm[4], nl[4], nd[4];
      if (kStatsW0) load_stats(0, nm, nl, nd);
      // Loads issued but not yet seen complete must land before the CTA
      // exits, even on the abort path: remember their barriers and parities.
      int pend_kv = 1;
      bool ok = mbar_wait(bar(B_KV_FULL), 0, abort, status);
      if (ok) {
        pend_kv = 0;
        if (kv_valid < BM) {
          zero_rows<D>(sbase + L::K, kv_valid, lane);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_KV_READY));
      }
      if (kStatsW0 && ok) {
        for (int k = 0; k < n_it; ++k) {
          const int s = k % NQS;
          // the stage's statistics slot is free once its previous block's dK
          // has run (the release of its Q buffer)
          if (k >= NQS && !mbar_wait(bar(B_Q_EMPTY0 + s), ((k / NQS) - 1) & 1, abort, status)) break;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            rm[j] = nm[j];
            rl[j] = nl[j];
            rd[j] = nd[j];
          }
          load_stats(k + 1, nm, nl, nd);
          store_stats(s, rm, rl, rd);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_ST_READY0 + s));
        }
      }
      volatile int no_abort = 0;
      if (pend_kv) mbar_wait(bar(B_KV_FULL), 0, &no_abort, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dO producer
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      int pend_do = -1;
      uint32_t par_do = 0;
      for (int k = 0; k < n_it; ++k) {
        const int s = k & 1;
        const uint32_t prev = ((k >> 1) - 1) & 1;
        const int qb = qb_of(k);
        const int q_valid = min(BN, s1 - qb * BN);
        if (k >= 2 && !mbar_wait(bar(B_DO_EMPTY0 + s), prev, abort, status)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_DO_FULL0 + s), L::TILE);
          for (int c = 0; c < L::NCH; ++c)
            tma_load_2d(sbase + L::DO + s * L::TILE + c * CHUNK, &p.tm_do, hq_of(k) * D + c * 64,
                        q_start + qb * BN, bar(B_DO_FULL0 + s));
        }
        pend_do = s;
        par_do = (k >> 1) & 1;
        if (!mbar_wait(bar(B_DO_FULL0 + s), (k >> 1) & 1, abort, status)) break;
        pend_do = -1;
        if (q_valid < BN) {
          zero_rows<D>(sbase + L::DO + s * L::TILE, q_valid, lane);
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
    // The whole warp runs the schedule and waits; one elected lane issues.
    if (n_it > 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);     // S^T, dP^T: K-major x K-major
      constexpr uint32_t ID_KV = idesc_bf16(128, D, 0, 1);      // dV, dK: B (dO / Q) MN-major
      constexpr uint32_t ID_DQ = idesc_bf16(128, D, 1, 1);      // dQ = dS K: both MN-major
      const uint32_t t_s = tmem + COL_S, t_dp = tmem + COL_DP;
      const uint32_t t_dv = tmem + COL_DV, t_dk = tmem + L::COL_DK, t_dq = tmem + L::COL_DQ;
      const uint32_t sK = sbase + L::K, sV = sbase + L::V, sDS = sbase + L::DS;
      bool ok = mbar_wait(bar(B_KV_READY), 0, abort, status) && mbar_wait(bar(B_Q_READY0), 0, abort, status);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          mmas_kk<D / 16>(t_s, sK, sbase + L::Q, ID_S, 0);
          mma_commit(bar(B_S_FULL));
        }
        __syncwarp();
      }
      bool dp_issued = false;   // (d = 64) dP^T of block k issued during block k-1
      for (int k = 0; ok && k < n_it; ++k) {
        const int s = k & 1;
        const uint32_t ph = k & 1;
        const int qs = k % NQS;
        const uint32_t sQ = sbase + L::Q + qs * L::TILE, sDO = sbase + L::DO + s * L::TILE;
        if (!dp_issued) {
          // dP^T into the dP columns.  d = 128: they also carry the dQ
          // partial, so they are free once the previous partial is read out.
          // d = 64: free once the softmax has read dP of the previous block
          // (its dS was seen ready before that block's dK / dQ were issued).
          if (!kSep && k > 0 && !mbar_wait(bar(B_DQ_EMPTY), (k - 1) & 1, abort, status)) { ok = false; break; }
          if (!mbar_wait(bar(B_DO_READY0 + s), (k >> 1) & 1, abort, status)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
            mmas_kk<D / 16>(t_dp, sV, sDO, ID_S, 0);
            mma_commit(bar(B_DP_FULL));
          }
          __syncwarp();
        }
        dp_issued = false;
        // dV += P^T dO with P (bf16) read from TMEM.
        if (!mbar_wait(bar(B_P_READY), ph, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          mmas_tm<BN / 16>(t_dv, t_s, sDO, ID_KV, k > 0);
          mma_commit(bar(B_P_USED));
          if (kSep) mma_commit(bar(B_DO_EMPTY0 + s));   // dP and dV were the dO block's uses
        }
        __syncwarp();
        // Independent groups follow dV_i: the next block's S^T (needs
        // Q_{i+1} loaded and dV_i done, since it overwrites the P columns)
        // and this block's dK / dQ (need dS_i).  Issue whichever group's
        // inputs are ready first.  d = 128: dK / dQ first when both are,
        // because the dQ partial gates the next dP through the write-back.
        // d = 64: S^T first (the softmax needs it next), and the next
        // block's dP^T (needs dO_{i+1} and dS_i, i.e. dP_i read) ahead of
        // dK / dQ, which also wait for the previous dQ partial to be read
        // out of its columns.
        {
          bool need_s = (k + 1 < n_it), need_c2 = true, need_dp = kSep && (k + 1 < n_it);
          const int s1n = (k + 1) & 1;                    // dO stage of the next block
          const uint32_t dpar = ((k + 1) >> 1) & 1;
          const int q1n = (k + 1) % NQS;                  // its Q stage
          const uint32_t qpar = ((k + 1) / NQS) & 1;
          const unsigned long long t0 = globaltimer();
          while (need_s || need_c2) {
            bool s_ready = need_s && mbar_test(bar(B_Q_READY0 + q1n), qpar) && mbar_test(bar(B_P_USED), ph);
            bool c_ready = need_c2 && mbar_test(bar(B_DS_READY), ph);
            bool d_ready = false;
            if (kSep) {
              d_ready = need_dp && c_ready && mbar_test(bar(B_DO_READY0 + s1n), dpar);
              if (kDQ) c_ready = c_ready && (k == 0 || mbar_test(bar(B_DQ_EMPTY), (k - 1) & 1));
            }
            s_ready = __shfl_sync(0xffffffffu, s_ready, 0);
            c_ready = __shfl_sync(0xffffffffu, c_ready, 0);
            d_ready = __shfl_sync(0xffffffffu, d_ready, 0);
            if (kSep && s_ready) {
              tc_fence_after();
              if (elect_one()) {
                mmas_kk<D / 16>(t_s, sK, sbase + L::Q + q1n * L::TILE, ID_S, 0);
                mma_commit(bar(B_S_FULL));
              }
              __syncwarp();
              need_s = false;
            } else if (kSep && d_ready) {
              tc_fence_after();
              if (elect_one()) {
                mmas_kk<D / 16>(t_dp, sV, sbase + L::DO + s1n * L::TILE, ID_S, 0);
                mma_commit(bar(B_DP_FULL));
              }
              __syncwarp();
              need_dp = false;
              dp_issued = true;
            } else if (s_ready && !c_ready) {
              tc_fence_after();
              if (elect_one()) {
                mmas_kk<D / 16>(t_s, sK, sbase + L::Q + q1n * L::TILE, ID_S, 0);
                mma_commit(bar(B_S_FULL));
              }
              __syncwarp();
              need_s = false;
            } else if (c_ready) {
              // dK += dS^T Q and the dQ partial, both from dS in shared memory.
              tc_fence_after();
              if (elect_one()) {
                mmas_km<BN / 16>(t_dk, sDS, sQ, ID_KV, k > 0);
                if (kDQ) {
                  mmas_mm<BM / 16>(t_dq, sDS, sK, ID_DQ, 0);
                  mma_commit(bar(B_DQ_FULL));
                }
                mma_commit(bar(B_DS_FREE));
                if (kSep) mma_commit(bar(B_Q_EMPTY0 + qs));   // dK was the Q block's last use
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
              // (polled without a sleep: a 32 ns sleep here cost 3 % at d = 64)
            }
          }
          if (!ok) break;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (elect_one()) mma_commit(bar(ok ? B_ACC_FULL : B_TEARDOWN));
      __syncwarp();
      if (!ok) {
        // Aborted: wait (bounded) for every MMA issued so far before TMEM is freed.
        volatile int no_abort = 0;
        mbar_wait(bar(B_TEARDOWN), 0, &no_abort, status);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax / dS
    setmaxnreg_to<kRegSoftmax, kRegLaunch>();
    const int wg = (warp - 4) >> 2;          // 0: query columns 0-63, 1: 64-127
    const int quarter = warp & 3;            // TMEM lane quarter
    const int r = quarter * 32 + lane;       // key row within the block
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int k = 0; k < n_it; ++k) {
      const uint32_t ph = k & 1;
      const int qb = qb_of(k);
      // visible query columns of key row r in this tile: [c_lo, c_lo + span)
      int c_lo = 0, c_end = min(BN, s1 - qb * BN);
      if (p.causal) {
        const long long d0 = static_cast<long long>(kvb) * BM + r - off - static_cast<long long>(qb) * BN;
        c_lo = static_cast<int>(max(0LL, min(d0, static_cast<long long>(BN))));
        if (W > 0) c_end = static_cast<int>(max(0LL, min(static_cast<long long>(c_end), d0 + W)));
      }
      const int span = (r < kv_valid) ? max(0, c_end - c_lo) : 0;
      const bool need_mask = __any_sync(0xffffffffu, c_lo > wg * 64 || c_lo + span < wg * 64 + 64);
      const int qs = k % NQS;
      // the row statistics of this block are in shared memory
      if (!mbar_wait(bar((kStatsW0 ? B_ST_READY0 : B_Q_READY0) + qs), (k / NQS) & 1, abort, status)) { ok = false; break; }
      // The 64 per-column statistics are read into registers before the
      // scores are waited for: shared-memory loads queue behind the MMAs'
      // operand reads, so their latency is hidden here rather than inside
      // the exp loop.
      const float4* lse4 = reinterpret_cast<const float4*>(st_lse + qs * 128 + wg * 64);
      const float4* dvec4 = reinterpret_cast<const float4*>(st_D + qs * 128 + wg * 64);
      float4 lsev[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) lsev[i] = lse4[i];
      if (!mbar_wait(bar(B_S_FULL), ph, abort, status)) { ok = false; break; }
      tc_fence_after();
      float P[64];
      const uint32_t t_srow = tmem + lane_addr + COL_S + wg * 64;
      if (need_mask)
        softmax_p<true>(t_srow, lse4, lsev, sl2, P, wg * 64, c_lo, span);
      else
        softmax_p<false>(t_srow, lse4, lsev, sl2, P, wg * 64, c_lo, span);
      tc_fence_before();
      mbar_arrive(bar(B_P_READY));

      float4 dv4v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) dv4v[i] = dvec4[i];
      if (!mbar_wait(bar(B_DP_FULL), ph, abort, status)) { ok = false; break; }
      // The dS buffer is free once the previous block's dK / dQ MMAs ran.
      if (k > 0 && !mbar_wait(bar(B_DS_FREE), (k - 1) & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ds_row = sbase + L::DS + wg * CHUNK + (r >> 3) * 1024 + (r & 7) * 128;
      const uint32_t t_dprow = tmem + lane_addr + COL_DP + wg * 64;
      if (need_mask)
        softmax_ds<true>(t_dprow, dvec4, dv4v, P, ds_row, r);
      else
        softmax_ds<false>(t_dprow, dvec4, dv4v, P, ds_row, r);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_DS_READY));
    }
    // ------------------------------------------------------------ dK / dV epilogue
    const int kv_row = kv_start + kvb * BM + r;
    uint16_t* out = (wg == 0) ? p.dv : p.dk;
    const float mul = (wg == 0) ? 1.f : p.scale;
    uint8_t* dst = reinterpret_cast<uint8_t*>(out + static_cast<long long>(kv_row) * rs_kv + hk * D);
    if (n_it == 0) {
      if (r < kv_valid)
        for (int c = 0; c < D; c += 8) st_global_v4(dst + c * 2, 0u, 0u, 0u, 0u);
    } else if (__all_sync(0xffffffffu, ok && mbar_wait(bar(B_ACC_FULL), 0, abort, status))) {
      tc_fence_after();
      const uint32_t col0 = (wg == 0) ? COL_DV : L::COL_DK;
      if (D == 128 && kv_valid == BM) {
        // A whole key block at d = 128: staged as bf16 in the V (dV) / K (dK)
        // tile, which no MMA reads any more, and written by TMA in 64-column
        // boxes (each thread's own row would otherwise leave as 16-byte pieces
        // of 32 different rows per warp store; 5.2 -> 3.7 us per CTA).  A
        // partial block is written per row below, so that no row of the next
        // sequence is touched; so is d = 64, where the staged store measured
        // 1.5 % slower overall.
        const uint32_t tile = sbase + ((wg == 0) ? L::V : L::K);
        const uint32_t row = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + col0 + ch * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              w[j] = pack_bf16x2(mul * __uint_as_float(v[8 * g + 2 * j]), mul * __uint_as_float(v[8 * g + 2 * j + 1]));
            const int u = (ch & 1) * 4 + g;   // 16-byte unit within the 128-byte row of a 64-column chunk
            st_shared_v4(row + (ch >> 1) * CHUNK + ((u ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_EPI0 + wg));
        // One thread per warpgroup waits (bounded) for the other 127 rows.
        if (quarter == 0 && lane == 0 && mbar_wait(bar(B_EPI0 + wg), 0, abort, status)) {
          for (int c = 0; c < L::NCH; ++c)
            tma_store_2d((wg == 0) ? &p.tm_dv : &p.tm_dk, tile + c * CHUNK, hk * D + c * 64, kv_start + kvb * BM);
          bulk_commit();
          bulk_wait_read0();   // the tile is read before the CTA exits
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + col0 + ch * 32, v);
          tmem_ld_wait();
          if (r < kv_valid) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint32_t w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                w[j] = pack_bf16x2(mul * __uint_as_float(v[8 * g + 2 * j]), mul * __uint_as_float(v[8 * g + 2 * j + 1]));
              st_global_v4(dst + (ch * 32 + g * 8) * 2, w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ write-back
    setmaxnreg_to<kRegDrain, kRegLaunch>();
    if constexpr (kDQ) {
      // TMEM lanes are query rows.  The partial of block k leaves as
      // 128B-swizzled [32 x 32] fp32 boxes reduce-added into dq_acc by TMA.
      // d = 128: first half of the columns staged in block k's Q buffer (dead
      // once dK_k has run), second half in its dO buffer (dead after dV_k),
      // each released to its owner once TMA has read it.  d = 64: both halves
      // in this warp's part of the staging area.  Both halves are in flight at
      // once; the SM's write-out bandwidth sets the pace.
      const int quarter = warp & 3;
      const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
      constexpr int NC = D / 32;              // 32-column chunks: 2 or 4
      constexpr int BPH = NC / 2;             // boxes per warp per half: 1 or 2
      auto stage_box = [&](uint32_t box, const uint32_t (&v)[32]) {
        const uint32_t row = box + lane * 128;
  #pragma unroll
        for (int g = 0; g < 8; ++g)
          st_shared_v4(row + ((g ^ (lane & 7)) << 4), v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
      };
      bool issued = false;
      int last_q = -1;   // (warp 12) the last block whose Q load this warp issued

      for (int k = 0; k < n_it; ++k) {
        const int s = k & 1;
        const int qb = qb_of(k);
        const int hq = hq_of(k);
        const int y = q_start + qb * BN + quarter * 32;
        // d = 128: the partial is staged in this block's own Q and dO buffers,
        // which the MMAs no longer read once dQ_i is complete; each goes back
        // to its owner once TMA has read it.  d = 64: in this warp's 8 KB of
        // the staging area, reused once TMA has read the previous partial.
        const uint32_t slot_a = kOwnDQ<D> ? sbase + L::STG + quarter * 8192
                                          : sbase + L::Q + (k % NQS) * L::TILE + quarter * (L::TILE / 4);
        const uint32_t slot_b = kOwnDQ<D> ? slot_a + 4096 : sbase + L::DO + s * L::TILE + quarter * (L::TILE / 4);
        if (!mbar_wait(bar(B_DQ_FULL), k & 1, abort, status)) break;
        tc_fence_after();
        uint32_t va[32], vb[32], vc[32], vd[32];
        tmem_ld32(tmem + lane_addr + L::COL_DQ + 0, va);
        tmem_ld32(tmem + lane_addr + L::COL_DQ + 32, vb);
        if (BPH == 2) {
          tmem_ld32(tmem + lane_addr + L::COL_DQ + 64, vc);
          tmem_ld32(tmem + lane_addr + L::COL_DQ + 96, vd);
        }
        tmem_ld_wait();
        // every TMEM column of this partial has been read
        tc_fence_before();
        mbar_arrive(bar(B_DQ_EMPTY));
        if (kOwnDQ<D>) {
          if (lane == 0 && issued) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
        }
        stage_box(slot_a, va);
        if (BPH == 2) stage_box(slot_a + 4096, vb);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_2d(&p.tm_dq, slot_a, hq * D + 0, y);
          if (BPH == 2) tma_reduce_add_2d(&p.tm_dq, slot_a + 4096, hq * D + 32, y);
          bulk_commit();
          issued = true;
        }
        if (BPH == 2) {
          stage_box(slot_b, vc);
          stage_box(slot_b + 4096, vd);
        } else {
          stage_box(slot_b, vb);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (q_by_drain) {
          // the first half has been read: its Q buffer goes back, and the
          // Q load of block k + NQS (issued by warp 12 once all four halves
          // are read) enters the TMA engine ahead of the second half
          if (lane == 0) {
            bulk_wait_read0();
            mbar_arrive(bar(B_Q_EMPTY0 + k % NQS));
          }
          __syncwarp();
          const int kn = k + NQS;
          if (kn < n_it) {
            if (quarter == 0) {
              if (lane == 0) {
                if (mbar_wait(bar(B_Q_EMPTY0 + k % NQS), (k / NQS) & 1, abort, status)) {
                  const uint32_t qbuf = sbase + L::Q + (k % NQS) * L::TILE;
                  mbar_arrive_expect_tx(bar(B_Q_FULL0 + k % NQS), L::TILE);
                  for (int c = 0; c < L::NCH; ++c)
                    tma_load_2d(qbuf + c * CHUNK, &p.tm_q, hq_of(kn) * D + c * 64, q_start + qb_of(kn) * BN,
                                bar(B_Q_FULL0 + k % NQS));
                  last_q = kn;
                }
                mbar_arrive(bar(B_Q_ISSUED0 + (k & 1)));
              }
            } else if (!mbar_wait(bar(B_Q_ISSUED0 + (k & 1)), (k >> 1) & 1, abort, status)) {
              break;
            }
            __syncwarp();
          }
        }
        if (lane == 0) {
          if (BPH == 2) {
            tma_reduce_add_2d(&p.tm_dq, slot_b, hq * D + 64, y);
            tma_reduce_add_2d(&p.tm_dq, slot_b + 4096, hq * D + 96, y);
          } else {
            tma_reduce_add_2d(&p.tm_dq, slot_b, hq * D + 32, y);
          }
          bulk_commit();
          if (!kOwnDQ<D>) {
            if (!q_by_drain) {
              asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // first half read
              mbar_arrive(bar(B_Q_EMPTY0 + k % NQS));
            }
            bulk_wait_read0();                                               // second half read
            mbar_arrive(bar(B_DO_EMPTY0 + s));
          }
        }
        __syncwarp();
      }
      if (lane == 0 && issued) bulk_wait_all0();
      if (lane == 0 && last_q >= 0) {
        // Q loads this warp issued land before the CTA exits, also after an
        // abort (the Q producer then stops waiting for them)
        volatile int no_abort = 0;
        for (int b = max(NQS, last_q - NQS + 1); b <= last_q; ++b)
          mbar_wait(bar(B_Q_FULL0 + b % NQS), (b / NQS) & 1, &no_abort, status);
      }
    }
  } else {
    // ------------------------------------------------------------ Q producer (warp 3)
    setmaxnreg_to<kRegOther, kRegLaunch>();
    if (n_it > 0) {
      // a load issued but not seen complete must land before the CTA exits
      int pend_q = -1;
      uint32_t par_q = 0;
      bool ok = true;
      // (unless kStatsW0) the row statistics are loaded here as well
      float rm[4], rl[4], rd[4], nm[4], nl[4], nd[4];
      if (!kStatsW0) load_stats(0, nm, nl, nd);
      // Q with the row statistics.  K / V, Q and dO have producer warps of
      // their own, so that each stream's load is issued as soon as its stage
      // is free: loads share the SM's TMA engine with the dQ reduce-adds and
      // take over a thousand cycles to land.
      for (int k = 0; ok && k < n_it; ++k) {
        const int s = k % NQS;
        const uint32_t use = k / NQS;               // how often stage s was filled before
        const uint32_t prev = (use - 1) & 1;        // parity of this stage's previous release
        const int qb = qb_of(k);
        const int hq = hq_of(k);
        const int q_row0 = q_start + qb * BN;
        const int q_valid = min(BN, s1 - qb * BN);
        if (k >= NQS && !mbar_wait(bar(B_Q_EMPTY0 + s), prev, abort, status)) break;
        if (!q_by_drain || k < NQS) {
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q_FULL0 + s), L::TILE);
            for (int c = 0; c < L::NCH; ++c)
              tma_load_2d(sbase + L::Q + s * L::TILE + c * CHUNK, &p.tm_q, hq * D + c * 64, q_row0, bar(B_Q_FULL0 + s));
          }
          pend_q = s;
          par_q = use & 1;
        }
        if constexpr (!kStatsW0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            rm[j] = nm[j];
            rl[j] = nl[j];
            rd[j] = nd[j];
          }
          load_stats(k + 1, nm, nl, nd);
          store_stats(s, rm, rl, rd);
        }
        if (!mbar_wait(bar(B_Q_FULL0 + s), use & 1, abort, status)) break;
        pend_q = -1;
        if (q_valid < BN) {
          zero_rows<D>(sbase + L::Q + s * L::TILE, q_valid, lane);
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

template <int D, bool kDQ>
cudaError_t launch_d(const BwdParams& p, int batch, int max_kv_blocks, cudaStream_t s) {
  constexpr uint32_t bytes = Layout<D>::BYTES;
  static_assert(bytes <= 232448, "shared memory budget");
  static std::atomic<unsigned long long> smem_set{0}, smem_set_chunked{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(bwd_kernel<D, false, kDQ>), (int)bytes, smem_set);
  if (e == cudaSuccess)
    e = set_smem_once(reinterpret_cast<const void*>(bwd_kernel<D, true, kDQ>), (int)bytes, smem_set_chunked);
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(max_kv_blocks) * p.heads_kv * batch > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  BwdParams q = p;
  q.batch = batch;
  q.grid_kv = max_kv_blocks;
  // neither variant orders its CTAs' work: the launch order is free
  BwdParams any_order = p;
  any_order.dq_mode = 0;
  q.head_chunk = launch_head_chunk(any_order, batch, max_kv_blocks, BM, BN, D);
  dim3 grid(max_kv_blocks, p.heads_kv, batch);
  if (q.head_chunk > 1)
    bwd_kernel<D, true, kDQ><<<grid, kThreads, bytes, s>>>(q);
  else
    bwd_kernel<D, false, kDQ><<<grid, kThreads, bytes, s>>>(q);
  return cudaGetLastError();
}

}  // namespace

// Whether the key blocks' query sweeps differ enough in length for the
// launch order to matter: the longest sweep against the mean, for the
// longest sequence (lengths rounded up to whole blocks) and the mask's band.
static bool causal_sweeps_uneven(const BwdParams& p, int n_kvb, int bm, int bn) {
  const long long s1 = static_cast<long long>(p.max_q_blocks) * bn, s2 = static_cast<long long>(n_kvb) * bm;
  const long long off = p.bottom_right ? s2 - s1 : 0;
  auto fdiv = [](long long a, long long b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
  long long total = 0, longest = 0;
  for (long long kvb = 0; kvb < n_kvb; ++kvb) {
    const long long lo = std::max(0LL, fdiv(kvb * bm - off, bn));
    const long long hi = p.window > 0 ? std::min<long long>(p.max_q_blocks - 1, fdiv(kvb * bm + bm - 2 - off + p.window, bn))
                                      : p.max_q_blocks - 1;
    const long long n = std::max(0LL, hi - lo + 1);
    total += n;
    longest = std::max(longest, n);
  }
  return 2 * longest * n_kvb > 3 * total;   // longest > 1.5 x mean
}

int launch_head_chunk(const BwdParams& p, int batch, int n_kvb, int bm, int bn, int head_dim) {
  // Key blocks fast (chunk 1) unless a causal mask makes the sweeps uneven
  // and dQ is reduced in any order; then heavy-first, in chunks whose
  // query-side bytes (Q, dO in bf16 and the fp32 dQ accumulator of one
  // query head per unit) take about a quarter of L2.
  constexpr long long kChunkBytes = 32ll << 20;
  if (!p.causal || p.dq_mode != 0 || !causal_sweeps_uneven(p, n_kvb, bm, bn)) return 1;
  const long long unit_bytes = static_cast<long long>(p.max_q_blocks) * bn * head_dim * 8;
  return static_cast<int>(std::max(1LL, std::min<long long>(static_cast<long long>(p.heads_kv) * batch, kChunkBytes / unit_bytes)));
}

cudaError_t launch_bwd_main(const BwdParams& p, int head_dim, int batch, int max_kv_blocks, bool with_dq,
                            cudaStream_t s) {
  if (batch <= 0 || max_kv_blocks <= 0) return cudaSuccess;
  if (with_dq)
    return head_dim == 64 ? launch_d<64, true>(p, batch, max_kv_blocks, s) : launch_d<128, true>(p, batch, max_kv_blocks, s);
  return head_dim == 64 ? launch_d<64, false>(p, batch, max_kv_blocks, s) : launch_d<128, false>(p, batch, max_kv_blocks, s);
}

namespace {

// Waits, through the kernels' own bounded mbarrier wait, on a barrier that
// nothing arrives on: the wait gives up after its time limit (1 s here,
// shorter than the kernels' own) and records the timeout code in the
// status word, and the kernel returns normally.
__global__ void wait_timeout_kernel() {
  __shared__ __align__(8) uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&never), 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&never), 0, &abort_flag, &g_bwd_status, 1000000000ull);
}

}  // namespace

cudaError_t launch_wait_timeout(cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

int bwd_read_and_clear_status(cudaStream_t s, int* status) {
  int zero = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return static_cast<int>(e);
  e = cudaMemcpyFromSymbol(status, g_bwd_status, sizeof(int));
  if (e != cudaSuccess) return static_cast<int>(e);
  e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int));
  return static_cast<int>(e);
}

}  // namespace fa
