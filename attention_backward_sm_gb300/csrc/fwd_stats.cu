// Forward statistics (support step, not the timed path): for every query
// row, O = softmax(scale * Q K^T) V, m = max_j scale*S_ij and
// l = sum_j exp(scale*S_ij - m).  The SK-16 single-pass FA Grad article
// (section 3.1 step 2) defines P from exactly these m and l; section 5
// names the online-softmax forward skeleton as their producer.
//
// Masks: none, causal aligned top-left or bottom-right, and the causal
// sliding window (JAX dot_product_attention, sliding_window_length).
//
// One CTA computes a 64-row query block of one (sequence, query head; the
// key/value head is shared by a group of query heads) with an
// online softmax over 64-row key blocks, on the CUDA cores in fp32 (every
// product and sum in fp32, P kept in fp32).  256 threads: thread t owns
// query rows 4*(t/16) .. +3; in the score phase it owns key columns
// 4*(t%16) .. +3, in the output phase head-dim columns (d/16)*(t%16) ...
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace fa {
namespace {

constexpr int BQ = 64;
constexpr int BK = 64;
constexpr int LD = BQ + 4;   // padded leading dimension of the transposed tiles

__device__ __forceinline__ float bf2f(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t r;
  asm("{\n\t.reg .b16 h;\n\tcvt.rn.bf16.f32 h, %1;\n\tmov.b32 %0, {h, h};\n\t}" : "=r"(r) : "f"(f));
  return static_cast<uint16_t>(r & 0xFFFFu);
}

template <int D>
__global__ void __launch_bounds__(256) fwd_stats_kernel(const FwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* qT = sm;               // [D][LD]  Q block transposed
  float* kT = qT + D * LD;      // [D][LD]  K block transposed
  float* vs = kT + D * LD;      // [BK][D]
  float* pT = vs + BK * D;      // [BK][LD] P block transposed

  const int b = blockIdx.z, h = blockIdx.y, qb = blockIdx.x;
  const int q0 = p.cu_q[b], s1 = p.cu_q[b + 1] - q0;
  const int k0 = p.cu_kv[b], s2 = p.cu_kv[b + 1] - k0;
  if (qb * BQ >= s1) return;
  const int H = p.heads;
  const long long rs = static_cast<long long>(H) * D;   // query-side row stride in elements
  const long long rs_kv = static_cast<long long>(p.heads_kv) * D;
  const int hk = h / (H / p.heads_kv);                   // key/value head of this query head
  const int tid = threadIdx.x;
  const int rg = tid >> 4, cg = tid & 15;
  constexpr int OC = D / 16;   // output columns per thread

  for (int e = tid; e < BQ * D; e += 256) {
    const int r = e / D, c = e % D;
    const int qi = qb * BQ + r;
    qT[c * LD + r] = (qi < s1) ? bf2f(p.q[(q0 + qi) * rs + h * D + c]) : 0.f;
  }

  float m_run[4], l_run[4], acc[4][OC];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int c = 0; c < OC; ++c) acc[i][c] = 0.f;
  }

  // Query i sees key j iff j <= i + off (causal; off = s2 - s1 for the
  // bottom-right alignment, else 0) and j > i + off - W (window W > 0).
  // Keys any row of this block sees: [kv_begin, kv_end).
  const long long off = p.bottom_right ? static_cast<long long>(s2) - s1 : 0;
  const int W = p.window;
  long long kv_begin = 0, kv_end = s2;
  if (p.causal) {
    kv_end = min(kv_end, static_cast<long long>(qb) * BQ + BQ + off);
    if (W > 0) kv_begin = max(0LL, static_cast<long long>(qb) * BQ + off - W + 1);
  }
  const int kb_first = static_cast<int>(kv_begin / BK);
  const int kb_end = kv_end > kv_begin ? static_cast<int>((kv_end + BK - 1) / BK) : kb_first;

  for (int kb = kb_first; kb < kb_end; ++kb) {
    __syncthreads();
    for (int e = tid; e < BK * D; e += 256) {
      const int r = e / D, c = e % D;
      const int kj = kb * BK + r;
      const bool ok = kj < s2;
      const long long g = (k0 + kj) * rs_kv + hk * D + c;
      kT[c * LD + r] = ok ? bf2f(p.k[g]) : 0.f;
      vs[r * D + c] = ok ? bf2f(p.v[g]) : 0.f;
    }
    __syncthreads();

    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
    for (int c = 0; c < D; ++c) {
      const float4 qv = *reinterpret_cast<const float4*>(&qT[c * LD + rg * 4]);
      const float4 kv = *reinterpret_cast<const float4*>(&kT[c * LD + cg * 4]);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
      const float ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qa[i], ka[j], s[i][j]);
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qi = qb * BQ + rg * 4 + i;
      float x[4];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int kj = kb * BK + cg * 4 + j;
        const long long rel = static_cast<long long>(kj) - qi - off;   // j - (i + off)
        const bool ok = kj < s2 && (!p.causal || (rel <= 0 && (W <= 0 || rel > -W)));
        x[j] = ok ? s[i][j] * p.scale : -INFINITY;
        mx = fmaxf(mx, x[j]);
      }
#pragma unroll
      for (int sh = 8; sh > 0; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
      const float m_new = fmaxf(m_run[i], mx);
      // Rows that have seen no visible key yet keep m = -inf and P = 0.
      const float alpha = (m_new == -INFINITY) ? 1.f : expf(m_run[i] - m_new);
      float rsum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pj = (x[j] == -INFINITY) ? 0.f : expf(x[j] - m_new);
        rsum += pj;
        pT[(cg * 4 + j) * LD + rg * 4 + i] = pj;
      }
#pragma unroll
      for (int sh = 8; sh > 0; sh >>= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, sh);
      l_run[i] = l_run[i] * alpha + rsum;
      m_run[i] = m_new;
#pragma unroll
      for (int c = 0; c < OC; ++c) acc[i][c] *= alpha;
    }
    __syncthreads();

#pragma unroll 2
    for (int j = 0; j < BK; ++j) {
      const float4 pv = *reinterpret_cast<const float4*>(&pT[j * LD + rg * 4]);
      const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
      float va[OC];
#pragma unroll
      for (int c4 = 0; c4 < OC / 4; ++c4) {
        const float4 t = *reinterpret_cast<const float4*>(&vs[j * D + cg * OC + c4 * 4]);
        va[c4 * 4 + 0] = t.x;
        va[c4 * 4 + 1] = t.y;
        va[c4 * 4 + 2] = t.z;
        va[c4 * 4 + 3] = t.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < OC; ++c) acc[i][c] = fmaf(pa[i], va[c], acc[i][c]);
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qi = qb * BQ + rg * 4 + i;
    if (qi >= s1) continue;
    const long long row = q0 + qi;
    const float inv = (l_run[i] > 0.f) ? 1.f / l_run[i] : 0.f;
#pragma unroll
    for (int c = 0; c < OC; ++c) p.o[row * rs + h * D + cg * OC + c] = f2bf(acc[i][c] * inv);
    if (cg == 0) {
      if (p.stats_lse) {
        p.m[row * H + h] = (l_run[i] > 0.f) ? m_run[i] + logf(l_run[i]) : -INFINITY;
      } else {
        p.m[row * H + h] = m_run[i];
        p.l[row * H + h] = l_run[i];
      }
    }
  }
}

template <int D>
constexpr size_t fwd_smem_bytes() {
  return sizeof(float) * (2 * D * LD + BK * D + BK * LD);
}

}  // namespace

cudaError_t launch_fwd_stats(const FwdParams& p, int head_dim, int batch, int max_q_blocks64, cudaStream_t s) {
  if (batch <= 0 || max_q_blocks64 <= 0) return cudaSuccess;
  dim3 grid(max_q_blocks64, p.heads, batch);
  if (head_dim == 64) {
    constexpr size_t sm = fwd_smem_bytes<64>();
    cudaError_t e = cudaFuncSetAttribute(fwd_stats_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    fwd_stats_kernel<64><<<grid, 256, sm, s>>>(p);
  } else {
    constexpr size_t sm = fwd_smem_bytes<128>();
    cudaError_t e = cudaFuncSetAttribute(fwd_stats_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    fwd_stats_kernel<128><<<grid, 256, sm, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fa
