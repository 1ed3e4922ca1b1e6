// Forward statistics on the tensor cores (sm_103a: tcgen05 + TMEM + TMA).
//
// For every query row: O = softmax(scale * Q K^T) V, m = max_j scale*S_ij and
// l = sum_j exp(scale*S_ij - m) (or the single statistic lse = m + ln l).
// The SK-16 single-pass FA Grad article (section 3.1 step 2) defines the
// backward's P from exactly these m and l and (section 5) names the
// online-softmax forward skeleton as their producer.  Masks: none, causal
// aligned top-left or bottom-right, and the causal sliding window of JAX
// dot_product_attention (sliding_window_length).
//
// One CTA owns one (sequence, query head, 128-row query block) and sweeps
// the key blocks (128 rows) the mask band reaches:
//   S_j  = Q K_j^T          tcgen05, queries on TMEM lanes, two alternating
//                           128-column buffers so that S_{j+1} is computed
//                           while the softmax works on S_j
//   P_j  = 2^(S_j*scale*log2e - m_used)   fp32, then bf16 into the first 64
//                           columns of S_j's buffer (two per column)
//   O   += P_j V_j          tcgen05 with A read from TMEM
// Online softmax with lazy rescaling: m_used (log2 units) only moves when
// the running maximum exceeds it by more than 8, so O is rescaled in TMEM
// rarely; l accumulates against m_used and is converted to the true maximum
// at the end.
//
// Warp roles (256 threads): warp 0 TMA producer (Q once, K/V in a 2-stage
// ring), warp 1 TMEM allocator and MMA issuer, warps 4-7 softmax (thread =
// query row; they also zero the value rows past a sequence end) and
// epilogue.  Every
// wait is bounded; a timeout records FA_ERR_TIMEOUT in the status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "sm103.cuh"

namespace fa {

__device__ int g_fwd_status = 0;

namespace {

constexpr int kThreads = 256;
constexpr int BQ = 128;                  // query rows per CTA
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0;           // two S buffers of BK columns, then O (d columns)
constexpr float kRescaleLog2 = 8.f;      // lazy-rescale threshold (factor 256)

enum {
  B_Q_FULL = 0, B_KV_FULL0, B_KV_FULL1, B_KV_EMPTY0, B_KV_EMPTY1,
  B_S_FULL0, B_S_FULL1, B_P_READY0, B_P_READY1, B_O_DONE, B_TEARDOWN, NUM_BARS
};

// Tiles are stored as 64-column (128-byte) chunks of `rows` rows each, as
// TMA writes them with 128-byte swizzle.  With d = 256 the key blocks are
// 64 rows, so that Q (128 x 256) and two stages of K and V fit in shared
// memory and O (256 columns) fits in TMEM beside the two score buffers.
template <int D>
struct Layout {
  static constexpr int BK = (D == 256) ? 64 : 128;   // key rows per block
  static constexpr uint32_t CHUNK_Q = 128 * 128;      // 128 rows x 128 B
  static constexpr uint32_t CHUNK_KV = BK * 128;
  static constexpr uint32_t TILE_Q = 128 * D * 2;
  static constexpr uint32_t TILE_KV = BK * D * 2;
  static constexpr int NCH = D / 64;
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = TILE_Q;                // 2 stages
  static constexpr uint32_t V = TILE_Q + 2 * TILE_KV;  // 2 stages
  static constexpr uint32_t BARS = TILE_Q + 4 * TILE_KV;
  static constexpr uint32_t MISC = BARS + NUM_BARS * 8;
  static constexpr uint32_t BYTES = MISC + 16;
  static constexpr uint32_t COL_O = 2 * BK;
  static_assert(COL_O + D <= TMEM_COLS, "tensor memory budget");
};

// 16-element K step t of a K-major tile stored in chunks of `chunk` bytes
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int t, uint32_t chunk) {
  return sw128_desc(tile + (t >> 2) * chunk + (t & 3) * 32, 16, 1024);
}
// rows 16t..16t+15 of an MN-major tile whose 64-column chunks are `chunk` apart
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int t, uint32_t chunk) {
  return sw128_desc(tile + t * 2048, chunk, 1024);
}

// The same descriptors stepped by constants (start address = low 14 bits,
// addr >> 4; every step stays inside its tile): the issuing thread builds a
// group's descriptors once and adds offsets.
__device__ __forceinline__ constexpr uint64_t step_kmajor(int t, uint32_t chunk) {
  return ((t >> 2) * chunk + (t & 3) * 32) >> 4;
}
__device__ __forceinline__ constexpr uint64_t step_mnmajor(int t) { return (t * 2048) >> 4; }

__device__ __forceinline__ int floordiv(long long a, int b) {
  long long q = a / b;
  if ((a % b) != 0 && a < 0) --q;
  return static_cast<int>(q);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Launch order of a forward grid (x: query tiles, or pairs of tiles; y: query
// head; z: sequence).  Under a causal mask later tiles see more keys and go
// first.  Chunked: the linear block index takes the (sequence, query head)
// units in chunks of head_chunk with the tile as the slow index within a
// chunk, so the long tiles of every unit of a chunk start before the short
// ones and the short ones fill the tail.
template <bool kChunked>
__device__ __forceinline__ void fwd_block_of(const FwdTcParams& p, int& x, int& h, int& b) {
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
    x = nx - 1 - t;   // chunked only under a causal mask
    h = unit % p.heads;
    b = unit / p.heads;
  }
}

template <int D, bool kChunked>
__global__ void __launch_bounds__(kThreads, 1) fwd_kernel(const __grid_constant__ FwdTcParams p) {
  using L = Layout<D>;
  constexpr int BK = L::BK;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int qb, h, b;
  fwd_block_of<kChunked>(p, qb, h, b);
  const int H = p.heads;
  const int hk = h / (H / p.heads_kv);
  const int q_start = p.cu_q[b], s1 = p.cu_q[b + 1] - q_start;
  const int kv_start = p.cu_kv[b], s2 = p.cu_kv[b + 1] - kv_start;
  if (qb * BQ >= s1) return;                          // CTA-uniform, before any barrier
  const int q_valid = min(BQ, s1 - qb * BQ);
  // Mask band: query i sees key j iff j <= i + off (causal) and
  // j > i + off - W (window W > 0).  Key blocks this query block reaches:
  // [kb0, kb1].
  const int off = p.bottom_right ? s2 - s1 : 0;
  const int W = p.window;
  const int n_kb = (s2 + BK - 1) / BK;
  const long long q0 = static_cast<long long>(qb) * BQ;
  const int kb1 = p.causal ? min(n_kb - 1, floordiv(q0 + BQ - 1 + off, BK)) : n_kb - 1;
  const int kb0 = (p.causal && W > 0) ? max(0, floordiv(q0 + off - W + 1, BK)) : 0;
  const int n = kb1 - kb0 + 1;
  const long long rs = static_cast<long long>(H) * D;

  if (n <= 0) {
    // No row of this block sees a key: O = 0, m = -inf, l = 0.
    for (int e = threadIdx.x; e < q_valid * (D / 8); e += kThreads) {
      const int r = e / (D / 8), c = (e % (D / 8)) * 8;
      st_global_v4(p.o + (q_start + qb * BQ + r) * rs + h * D + c, 0u, 0u, 0u, 0u);
    }
    for (int r = threadIdx.x; r < q_valid; r += kThreads) {
      const long long idx = static_cast<long long>(q_start + qb * BQ + r) * H + h;
      p.m[idx] = -INFINITY;
      if (!p.stats_lse) p.l[idx] = 0.f;
    }
    return;
  }
  if (sbase & 1023) {
    if (threadIdx.x == 0) atomicCAS(&g_fwd_status, 0, 99);
    return;
  }

  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC + 4);
  const uint32_t bars = sbase + L::BARS;
  auto bar = [&](int i) { return bars + 8u * i; };
  int* status = &g_fwd_status;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KV_FULL0 + s), 1);
      mbar_init(bar(B_KV_EMPTY0 + s), 1);
      mbar_init(bar(B_S_FULL0 + s), 1);
    }
    // one per score buffer: the MMA warp issues S_{j+1} before it waits for
    // P_j, so with a single barrier the softmax could complete P_{j+1} (its
    // next phase) before that wait had seen P_j
    mbar_init(bar(B_P_READY0), 128);
    mbar_init(bar(B_P_READY1), 128);
    mbar_init(bar(B_O_DONE), 1);
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
    volatile int no_abort = 0;
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(bar(B_Q_FULL), L::TILE_Q);
      for (int c = 0; c < L::NCH; ++c)
        tma_load_2d(sbase + L::Q + c * L::CHUNK_Q, &p.tm_q, h * D + c * 64, q_start + qb * BQ, bar(B_Q_FULL));
    }
    __syncwarp();
    // The producer only issues loads: the MMA warp waits for their arrival
    // itself, and the softmax warps zero a tail block's value rows.
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      const int s = j & 1;
      if (j >= 2 && !mbar_wait(bar(B_KV_EMPTY0 + s), ((j >> 1) - 1) & 1, abort, status)) { ok = false; break; }
      if (lane == 0) {
        const int row = kv_start + (kb0 + j) * BK;
        mbar_arrive_expect_tx(bar(B_KV_FULL0 + s), 2 * L::TILE_KV);
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_2d(sbase + L::K + s * L::TILE_KV + c * L::CHUNK_KV, &p.tm_k, hk * D + c * 64, row,
                      bar(B_KV_FULL0 + s));
          tma_load_2d(sbase + L::V + s * L::TILE_KV + c * L::CHUNK_KV, &p.tm_v, hk * D + c * 64, row,
                      bar(B_KV_FULL0 + s));
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    // every load issued must land before the CTA exits, also after an abort
    for (int jj = max(0, issued - 2); jj < issued; ++jj)
      mbar_wait(bar(B_KV_FULL0 + (jj & 1)), (jj >> 1) & 1, &no_abort, status);
    mbar_wait(bar(B_Q_FULL), 0, &no_abort, status);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t ID_S = idesc_bf16(128, BK, 0, 0);    // S = Q K^T, both K-major
    constexpr uint32_t ID_O = idesc_bf16(128, D, 0, 1);     // O += P V, V (B) MN-major
    const uint32_t sQ = sbase + L::Q;
    bool ok = mbar_wait(bar(B_Q_FULL), 0, abort, status) && mbar_wait(bar(B_KV_FULL0), 0, abort, status);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        const uint64_t a0 = desc_kmajor(sQ, 0, L::CHUNK_Q), b0 = desc_kmajor(sbase + L::K, 0, L::CHUNK_KV);
#pragma unroll 4
        for (int t = 0; t < D / 16; ++t)
          mma_ss(tmem + COL_S0, a0 + step_kmajor(t, L::CHUNK_Q), b0 + step_kmajor(t, L::CHUNK_KV), ID_S, t > 0);
        mma_commit(bar(B_S_FULL0));
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int s = j & 1;
      if (j + 1 < n) {
        const int s1n = (j + 1) & 1;
        // S_{j+1} overwrites P_{j-1}: wait until O += P_{j-1} V_{j-1} is done
        if (!mbar_wait(bar(B_KV_FULL0 + s1n), ((j + 1) >> 1) & 1, abort, status)) { ok = false; break; }
        if (j >= 1 && !mbar_wait(bar(B_O_DONE), (j - 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sK = sbase + L::K + s1n * L::TILE_KV;
          const uint64_t a0 = desc_kmajor(sQ, 0, L::CHUNK_Q), b0 = desc_kmajor(sK, 0, L::CHUNK_KV);
#pragma unroll 4
          for (int t = 0; t < D / 16; ++t)
            mma_ss(tmem + COL_S0 + s1n * BK, a0 + step_kmajor(t, L::CHUNK_Q), b0 + step_kmajor(t, L::CHUNK_KV), ID_S,
                   t > 0);
          mma_commit(bar(B_S_FULL0 + s1n));
        }
        __syncwarp();
      }
      if (!mbar_wait(bar(B_P_READY0 + s), (j >> 1) & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      if (elect_one()) {
        const uint32_t sV = sbase + L::V + s * L::TILE_KV;
        const uint64_t b0 = desc_mnmajor(sV, 0, L::CHUNK_KV);
#pragma unroll 4
        for (int t = 0; t < BK / 16; ++t)
          mma_ts(tmem + L::COL_O, tmem + COL_S0 + s * BK + t * 8, b0 + step_mnmajor(t), ID_O, (j > 0) | (t > 0));
        mma_commit(bar(B_O_DONE));
        mma_commit(bar(B_KV_EMPTY0 + s));
      }
      __syncwarp();
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (elect_one()) mma_commit(bar(B_TEARDOWN));
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(bar(B_TEARDOWN), 0, &no_abort, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // query row in the block (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;
    const long long i_loc = q0 + r;                    // query index in its sequence
    float m_used = -INFINITY;                          // log2 units, reference of P and l
    float mx_raw = -INFINITY;                          // running maximum of the raw scores
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int s = j & 1;
      const int kb = kb0 + j;
      // visible key columns of this row in block kb: [c_lo, c_lo + span)
      const long long d0 = i_loc + off - static_cast<long long>(kb) * BK;   // last visible column
      int c_lo = 0, c_end = min(BK, s2 - kb * BK);
      if (p.causal) {
        c_end = static_cast<int>(max(0LL, min(static_cast<long long>(c_end), d0 + 1)));
        if (W > 0) c_lo = static_cast<int>(max(0LL, min(static_cast<long long>(BK), d0 - W + 1)));
      }
      const int span = (r < q_valid) ? max(0, c_end - c_lo) : 0;
      const bool need_mask = __any_sync(0xffffffffu, c_lo > 0 || span < BK);
      if (!mbar_wait(bar(B_S_FULL0 + s), (j >> 1) & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_s = tmem + lane_addr + COL_S0 + s * BK;
      float x[BK];
      {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) {
          tmem_ld32(t_s + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
        }
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < BK; ++c)
          x[c] = (static_cast<unsigned>(c - c_lo) < static_cast<unsigned>(span)) ? x[c] : -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < BK; ++c) mx = fmaxf(mx, x[c]);
      mx_raw = fmaxf(mx_raw, mx);
      const float m_new = fmaxf(m_used, mx * sl2);
      const bool grow = m_new > m_used + kRescaleLog2;   // also true for the first visible key
      float alpha = 1.f;
      if (grow) {
        alpha = ex2_approx(m_used - m_new);   // 0 while m_used = -inf
        l_run *= alpha;
        m_used = m_new;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O holds the earlier blocks' P V: rescale the rows whose reference
        // moved, once O += P_{j-1} V_{j-1} has completed (the warp's TMEM
        // accesses are collective, so lanes that did not grow scale by 1)
        if (!mbar_wait(bar(B_O_DONE), (j - 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + L::COL_O + c * 32, v);
          tmem_ld_wait();
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            w0[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            w1[e] = __float_as_uint(__uint_as_float(v[16 + e]) * alpha);
          }
          tmem_st16(tmem + lane_addr + L::COL_O + c * 32, w0);
          tmem_st16(tmem + lane_addr + L::COL_O + c * 32 + 16, w1);
        }
        tmem_st_wait();
      }
      // a row that has seen no key yet has only masked entries (x = -inf):
      // any finite reference gives them P = 0
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      // P = 2^(x*sl2 - m_used), masked entries (x = -inf) give 0
      float sum = 0.f;
#pragma unroll
      for (int g = 0; g < BK / 32; ++g) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(fmaf(x[g * 32 + 2 * e], sl2, -mref));
          const float p1 = ex2_approx(fmaf(x[g * 32 + 2 * e + 1], sl2, -mref));
          sum += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + g * 16, pk);
      }
      l_run += sum;
      const int kv_valid = min(BK, s2 - kb * BK);
      if (kv_valid < BK) {
        // value rows past the sequence hold other data (or NaN padding) and
        // P = 0 does not cancel a NaN: zero them before O += P V reads them
        // (the scores of those key rows are masked, so K needs no fix-up)
        if (!mbar_wait(bar(B_KV_FULL0 + s), (j >> 1) & 1, abort, status)) { ok = false; break; }
        const uint32_t sV = sbase + L::V + s * L::TILE_KV;
        constexpr int G16 = D / 8;   // 16-byte granules per row
        for (int e = r; e < (BK - kv_valid) * G16; e += 128) {
          const int row = kv_valid + e / G16, g = e % G16;
          st_shared_v4(sV + (g / 8) * L::CHUNK_KV + row * 128 + (g % 8) * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_P_READY0 + s));
    }
    ok = __all_sync(0xffffffffu, ok);
    // ------------------------------------------------------------ epilogue
    if (ok && mbar_wait(bar(B_O_DONE), (n - 1) & 1, abort, status)) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      uint16_t* orow = p.o + (q_start + qb * BQ + r) * rs + h * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + L::COL_O + c * 32, v);
        tmem_ld_wait();
        if (r < q_valid) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
#pragma unroll
          for (int g = 0; g < 4; ++g)
            st_global_v4(orow + c * 32 + g * 8, pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
      }
      if (r < q_valid) {
        const long long idx = static_cast<long long>(q_start + qb * BQ + r) * H + h;
        if (l_run > 0.f) {
          if (p.stats_lse) {
            p.m[idx] = (m_used + log2f(l_run)) * 0.6931471805599453f;
          } else {
            const float m_true = mx_raw * p.scale;
            p.m[idx] = m_true;
            p.l[idx] = l_run * ex2_approx(m_used - mx_raw * sl2);
          }
        } else {
          p.m[idx] = -INFINITY;
          if (!p.stats_lse) p.l[idx] = 0.f;
        }
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

// ---------------------------------------------------------------------------
// Two query tiles per CTA (used for head_dim 128).  A CTA owns 256 query rows
// as tiles A and B that share every K / V block; each tile has one softmax
// warpgroup and one score buffer and O accumulator in TMEM (S_A, S_B, O_A,
// O_B).  The MMA warp cycles S_A, S_B, P_A V, P_B V, so one tile's matmuls
// run while the other tile's softmax works.  Both tiles visit the union of
// their key-block ranges (a block outside one tile's band is fully masked
// there).  The softmax reads its score row from TMEM twice (for the row
// maximum, then for P), which keeps a thread's live values to one 32-column
// chunk.

constexpr int kThreads2 = 384;
constexpr uint32_t kRegOther2 = 56;      // warps 0-3
constexpr uint32_t kRegSoftmax2 = 200;   // warps 4-11
static_assert(128 * kRegOther2 + 256 * kRegSoftmax2 <= 65536, "register budgets exceed the launch");

enum {
  C_Q_FULL = 0, C_KV_FULL0, C_KV_FULL1, C_KV_EMPTY0, C_KV_EMPTY1,
  C_S_FULL0, C_S_FULL1, C_P_READY0, C_P_READY1, C_O_DONE0, C_O_DONE1, C_TEARDOWN, C_NUM
};

template <int D>
struct Layout2 {
  static constexpr int BK = 128;
  static constexpr uint32_t CHUNK = 128 * 128;
  static constexpr uint32_t TILE = 128 * D * 2;
  static constexpr int NCH = D / 64;
  static constexpr uint32_t Q = 0;                  // tiles A, B
  static constexpr uint32_t K = 2 * TILE;           // 2 stages
  static constexpr uint32_t V = 4 * TILE;           // 2 stages
  static constexpr uint32_t BARS = 6 * TILE;
  static constexpr uint32_t MISC = BARS + C_NUM * 8;
  static constexpr uint32_t BYTES = MISC + 16;
  static constexpr uint32_t COL_S = 0;              // tile t: [128 t, 128 t + 128)
  static constexpr uint32_t COL_O = 256;            // tile t: [256 + D t, 256 + D t + D)
  static_assert(COL_O + 2 * D <= TMEM_COLS, "tensor memory budget");
};

template <int D, bool kChunked>
__global__ void __launch_bounds__(kThreads2, 1) fwd2_kernel(const __grid_constant__ FwdTcParams p) {
  using L = Layout2<D>;
  constexpr int BK = L::BK;
  constexpr uint32_t kRegLaunch2 = 65536 / kThreads2 / 8 * 8;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int qp, h, b;                                       // qp: pair of 128-row tiles
  fwd_block_of<kChunked>(p, qp, h, b);
  const int H = p.heads;
  const int hk = h / (H / p.heads_kv);
  const int q_start = p.cu_q[b], s1 = p.cu_q[b + 1] - q_start;
  const int kv_start = p.cu_kv[b], s2 = p.cu_kv[b + 1] - kv_start;
  const long long q0 = static_cast<long long>(qp) * 2 * BQ;
  if (q0 >= s1) return;                              // CTA-uniform, before any barrier
  const int rows = static_cast<int>(min(static_cast<long long>(2 * BQ), s1 - q0));
  const int off = p.bottom_right ? s2 - s1 : 0;
  const int W = p.window;
  const int n_kb = (s2 + BK - 1) / BK;
  const int kb1 = p.causal ? min(n_kb - 1, floordiv(q0 + 2 * BQ - 1 + off, BK)) : n_kb - 1;
  const int kb0 = (p.causal && W > 0) ? max(0, floordiv(q0 + off - W + 1, BK)) : 0;
  const int n = kb1 - kb0 + 1;
  const long long rs = static_cast<long long>(H) * D;

  if (n <= 0) {
    for (int e = threadIdx.x; e < rows * (D / 8); e += kThreads2) {
      const int r = e / (D / 8), c = (e % (D / 8)) * 8;
      st_global_v4(p.o + (q_start + q0 + r) * rs + h * D + c, 0u, 0u, 0u, 0u);
    }
    for (int r = threadIdx.x; r < rows; r += kThreads2) {
      const long long idx = (q_start + q0 + r) * H + h;
      p.m[idx] = -INFINITY;
      if (!p.stats_lse) p.l[idx] = 0.f;
    }
    return;
  }
  if (sbase & 1023) {
    if (threadIdx.x == 0) atomicCAS(&g_fwd_status, 0, 99);
    return;
  }

  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC + 4);
  const uint32_t bars = sbase + L::BARS;
  auto bar = [&](int i) { return bars + 8u * i; };
  int* status = &g_fwd_status;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(bar(C_Q_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C_KV_FULL0 + s), 1);
      mbar_init(bar(C_KV_EMPTY0 + s), 1);
      mbar_init(bar(C_S_FULL0 + s), 1);
      mbar_init(bar(C_P_READY0 + s), 128);
      mbar_init(bar(C_O_DONE0 + s), 1);
    }
    mbar_init(bar(C_TEARDOWN), 1);
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
    setmaxnreg_to<kRegOther2, kRegLaunch2>();
    volatile int no_abort = 0;
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(bar(C_Q_FULL), 2 * L::TILE);
      for (int t = 0; t < 2; ++t)
        for (int c = 0; c < L::NCH; ++c)
          tma_load_2d(sbase + L::Q + t * L::TILE + c * L::CHUNK, &p.tm_q, h * D + c * 64,
                      static_cast<int>(q_start + q0) + t * BQ, bar(C_Q_FULL));
    }
    __syncwarp();
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      const int s = j & 1;
      if (j >= 2 && !mbar_wait(bar(C_KV_EMPTY0 + s), ((j >> 1) - 1) & 1, abort, status)) { ok = false; break; }
      if (lane == 0) {
        const int row = kv_start + (kb0 + j) * BK;
        mbar_arrive_expect_tx(bar(C_KV_FULL0 + s), 2 * L::TILE);
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_2d(sbase + L::K + s * L::TILE + c * L::CHUNK, &p.tm_k, hk * D + c * 64, row, bar(C_KV_FULL0 + s));
          tma_load_2d(sbase + L::V + s * L::TILE + c * L::CHUNK, &p.tm_v, hk * D + c * 64, row, bar(C_KV_FULL0 + s));
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    for (int jj = max(0, issued - 2); jj < issued; ++jj)
      mbar_wait(bar(C_KV_FULL0 + (jj & 1)), (jj >> 1) & 1, &no_abort, status);
    mbar_wait(bar(C_Q_FULL), 0, &no_abort, status);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_to<kRegOther2, kRegLaunch2>();
    constexpr uint32_t ID_S = idesc_bf16(128, BK, 0, 0);
    constexpr uint32_t ID_O = idesc_bf16(128, D, 0, 1);
    auto issue_s = [&](int t, int stage) {
      const uint64_t a0 = desc_kmajor(sbase + L::Q + t * L::TILE, 0, L::CHUNK);
      const uint64_t b0 = desc_kmajor(sbase + L::K + stage * L::TILE, 0, L::CHUNK);
#pragma unroll 4
      for (int k = 0; k < D / 16; ++k)
        mma_ss(tmem + L::COL_S + t * 128, a0 + step_kmajor(k, L::CHUNK), b0 + step_kmajor(k, L::CHUNK), ID_S, k > 0);
      mma_commit(bar(C_S_FULL0 + t));
    };
    auto issue_pv = [&](int t, int stage, int j) {
      const uint64_t b0 = desc_mnmajor(sbase + L::V + stage * L::TILE, 0, L::CHUNK);
#pragma unroll 4
      for (int k = 0; k < BK / 16; ++k)
        mma_ts(tmem + L::COL_O + t * D, tmem + L::COL_S + t * 128 + k * 8, b0 + step_mnmajor(k), ID_O,
               (j > 0) | (k > 0));
      mma_commit(bar(C_O_DONE0 + t));
    };
    bool ok = mbar_wait(bar(C_Q_FULL), 0, abort, status) && mbar_wait(bar(C_KV_FULL0), 0, abort, status);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_s(0, 0);
        issue_s(1, 0);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int s = j & 1;
      for (int t = 0; t < 2; ++t) {
        if (!mbar_wait(bar(C_P_READY0 + t), j & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          issue_pv(t, s, j);
          if (t == 1) mma_commit(bar(C_KV_EMPTY0 + s));
        }
        __syncwarp();
      }
      if (!ok || j + 1 >= n) break;
      const int s1n = (j + 1) & 1;
      if (!mbar_wait(bar(C_KV_FULL0 + s1n), ((j + 1) >> 1) & 1, abort, status)) { ok = false; break; }
      for (int t = 0; t < 2; ++t) {
        // S_t(j+1) overwrites P_t(j): wait until P_t(j) V_j has run
        if (!mbar_wait(bar(C_O_DONE0 + t), j & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) issue_s(t, s1n);
        __syncwarp();
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (elect_one()) mma_commit(bar(C_TEARDOWN));
      __syncwarp();
      volatile int no_abort = 0;
      mbar_wait(bar(C_TEARDOWN), 0, &no_abort, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax (tile t)
    setmaxnreg_to<kRegSoftmax2, kRegLaunch2>();
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // query row in the tile (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + L::COL_S + t * 128;
    const uint32_t t_o = tmem + lane_addr + L::COL_O + t * D;
    const float sl2 = p.scale * 1.4426950408889634f;
    const long long i_loc = q0 + t * BQ + r;           // query index in its sequence
    const int q_valid = static_cast<int>(max(0LL, min(static_cast<long long>(BQ), s1 - q0 - t * BQ)));
    float m_used = -INFINITY, mx_raw = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int s = j & 1;
      const int kb = kb0 + j;
      const long long d0 = i_loc + off - static_cast<long long>(kb) * BK;
      int c_lo = 0, c_end = min(BK, s2 - kb * BK);
      if (p.causal) {
        c_end = static_cast<int>(max(0LL, min(static_cast<long long>(c_end), d0 + 1)));
        if (W > 0) c_lo = static_cast<int>(max(0LL, min(static_cast<long long>(BK), d0 - W + 1)));
      }
      const int span = (r < q_valid) ? max(0, c_end - c_lo) : 0;
      const bool need_mask = __any_sync(0xffffffffu, c_lo > 0 || span < BK);
      if (!mbar_wait(bar(C_S_FULL0 + t), j & 1, abort, status)) { ok = false; break; }
      tc_fence_after();
      // pass 1: row maximum of the visible scores
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < BK / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_s + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float x = __uint_as_float(v[e]);
          const bool vis = !need_mask || static_cast<unsigned>(c * 32 + e - c_lo) < static_cast<unsigned>(span);
          mx = fmaxf(mx, vis ? x : -INFINITY);
        }
      }
      mx_raw = fmaxf(mx_raw, mx);
      const float m_new = fmaxf(m_used, mx * sl2);
      const bool grow = m_new > m_used + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2_approx(m_used - m_new);
        l_run *= alpha;
        m_used = m_new;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        if (!mbar_wait(bar(C_O_DONE0 + t), (j - 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(t_o + c * 32, v);
          tmem_ld_wait();
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            w0[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            w1[e] = __float_as_uint(__uint_as_float(v[16 + e]) * alpha);
          }
          tmem_st16(t_o + c * 32, w0);
          tmem_st16(t_o + c * 32 + 16, w1);
        }
        tmem_st_wait();
      }
      // pass 2: P = 2^(x*sl2 - m_used) as bf16 pairs over the first 64 columns
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      float sum = 0.f;
#pragma unroll 1
      for (int c = 0; c < BK / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_s + c * 32, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c0 = c * 32 + 2 * e;
          const bool vis0 = !need_mask || static_cast<unsigned>(c0 - c_lo) < static_cast<unsigned>(span);
          const bool vis1 = !need_mask || static_cast<unsigned>(c0 + 1 - c_lo) < static_cast<unsigned>(span);
          const float p0 = vis0 ? ex2_approx(fmaf(__uint_as_float(v[2 * e]), sl2, -mref)) : 0.f;
          const float p1 = vis1 ? ex2_approx(fmaf(__uint_as_float(v[2 * e + 1]), sl2, -mref)) : 0.f;
          sum += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + c * 16, pk);   // columns [16c, 16c+16): behind every chunk still to be read
      }
      l_run += sum;
      const int kv_valid = min(BK, s2 - kb * BK);
      if (t == 0 && kv_valid < BK) {
        // value rows past the sequence (other data or NaN padding) are zeroed
        // before either tile's P V reads them (tile B's follows tile A's)
        if (!mbar_wait(bar(C_KV_FULL0 + s), (j >> 1) & 1, abort, status)) { ok = false; break; }
        const uint32_t sV = sbase + L::V + s * L::TILE;
        constexpr int G16 = D / 8;
        for (int e = r; e < (BK - kv_valid) * G16; e += 128) {
          const int row = kv_valid + e / G16, g = e % G16;
          st_shared_v4(sV + (g / 8) * L::CHUNK + row * 128 + (g % 8) * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C_P_READY0 + t));
    }
    ok = __all_sync(0xffffffffu, ok);
    // ------------------------------------------------------------ epilogue (tile t)
    if (ok && mbar_wait(bar(C_O_DONE0 + t), (n - 1) & 1, abort, status)) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      uint16_t* orow = p.o + (q_start + i_loc) * rs + h * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_o + c * 32, v);
        tmem_ld_wait();
        if (r < q_valid) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
#pragma unroll
          for (int g = 0; g < 4; ++g)
            st_global_v4(orow + c * 32 + g * 8, pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
      }
      if (r < q_valid) {
        const long long idx = (q_start + i_loc) * H + h;
        if (l_run > 0.f) {
          if (p.stats_lse) {
            p.m[idx] = (m_used + log2f(l_run)) * 0.6931471805599453f;
          } else {
            p.m[idx] = mx_raw * p.scale;
            p.l[idx] = l_run * ex2_approx(m_used - mx_raw * sl2);
          }
        } else {
          p.m[idx] = -INFINITY;
          if (!p.stats_lse) p.l[idx] = 0.f;
        }
      }
    }
  } else {
    setmaxnreg_to<kRegOther2, kRegLaunch2>();   // warps 2, 3
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Chunk of the launch order: 1 (tile fastest) unless a causal mask makes
// the tiles' key ranges differ enough (longest > 1.5 x mean, for the longest
// sequences, lengths rounded up to whole tiles) for the order to matter;
// then chunks whose key-side bytes (K and V in bf16, shared by the query
// heads of a group) take about a quarter of L2.
int fwd_head_chunk(const FwdTcParams& p, int batch, int n_x, int rows, int bk, int head_dim) {
  constexpr long long kChunkBytes = 32ll << 20;
  if (!p.causal || n_x <= 1 || p.max_kv <= 0) return 1;
  const long long s1 = static_cast<long long>(n_x) * rows, s2 = p.max_kv;
  const long long off = p.bottom_right ? s2 - s1 : 0;
  const long long n_kb = (s2 + bk - 1) / bk;
  auto fdiv = [](long long a, long long b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
  long long total = 0, longest = 0;
  for (long long x = 0; x < n_x; ++x) {
    const long long q0 = x * rows;
    const long long kb1 = std::min(n_kb - 1, fdiv(q0 + rows - 1 + off, bk));
    const long long kb0 = p.window > 0 ? std::max(0LL, fdiv(q0 + off - p.window + 1, bk)) : 0;
    const long long n = std::max(0LL, kb1 - kb0 + 1);
    total += n;
    longest = std::max(longest, n);
  }
  if (2 * longest * n_x <= 3 * total) return 1;
  const long long unit_bytes =
      std::max(1LL, s2 * head_dim * 4 / std::max(1, p.heads / std::max(1, p.heads_kv)));
  return static_cast<int>(std::max(1LL, std::min<long long>(static_cast<long long>(p.heads) * batch, kChunkBytes / unit_bytes)));
}

template <int D>
cudaError_t launch_d2(const FwdTcParams& p, int batch, int max_q_blocks, cudaStream_t s) {
  constexpr uint32_t bytes = Layout2<D>::BYTES;
  static_assert(bytes <= 232448, "shared memory budget");
  static std::atomic<unsigned long long> smem_set{0}, smem_set_chunked{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(fwd2_kernel<D, false>), (int)bytes, smem_set);
  if (e == cudaSuccess) e = set_smem_once(reinterpret_cast<const void*>(fwd2_kernel<D, true>), (int)bytes, smem_set_chunked);
  if (e != cudaSuccess) return e;
  const int n_x = (max_q_blocks + 1) / 2;                // pairs of 128-row tiles
  if (static_cast<long long>(n_x) * p.heads * batch > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  FwdTcParams q = p;
  q.batch = batch;
  q.head_chunk = fwd_head_chunk(p, batch, n_x, 2 * BQ, Layout2<D>::BK, D);
  dim3 grid(n_x, p.heads, batch);
  if (q.head_chunk > 1)
    fwd2_kernel<D, true><<<grid, kThreads2, bytes, s>>>(q);
  else
    fwd2_kernel<D, false><<<grid, kThreads2, bytes, s>>>(q);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdTcParams& p, int batch, int max_q_blocks, cudaStream_t s) {
  constexpr uint32_t bytes = Layout<D>::BYTES;
  static_assert(bytes <= 232448, "shared memory budget");
  static std::atomic<unsigned long long> smem_set{0}, smem_set_chunked{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(fwd_kernel<D, false>), (int)bytes, smem_set);
  if (e == cudaSuccess) e = set_smem_once(reinterpret_cast<const void*>(fwd_kernel<D, true>), (int)bytes, smem_set_chunked);
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(max_q_blocks) * p.heads * batch > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  FwdTcParams q = p;
  q.batch = batch;
  q.head_chunk = fwd_head_chunk(p, batch, max_q_blocks, BQ, Layout<D>::BK, D);
  dim3 grid(max_q_blocks, p.heads, batch);
  if (q.head_chunk > 1)
    fwd_kernel<D, true><<<grid, kThreads, bytes, s>>>(q);
  else
    fwd_kernel<D, false><<<grid, kThreads, bytes, s>>>(q);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_main(const FwdTcParams& p, int head_dim, int batch, int max_q_blocks, cudaStream_t s) {
  if (batch <= 0 || max_q_blocks <= 0) return cudaSuccess;
  // Two query tiles per CTA at d = 128 (the tensor-core and softmax work of
  // a key block are of similar size there); at d = 64 the softmax alone
  // bounds the kernel and one tile per CTA measured faster; at d = 256 two
  // Q tiles do not fit in shared memory.
  if (head_dim == 64) return launch_d<64>(p, batch, max_q_blocks, s);
  if (head_dim == 256) return launch_d<256>(p, batch, max_q_blocks, s);
  return launch_d2<128>(p, batch, max_q_blocks, s);
}

int fwd_read_and_clear_status(cudaStream_t s, int* status) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_fwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_fwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return static_cast<int>(e);
}

}  // namespace fa
