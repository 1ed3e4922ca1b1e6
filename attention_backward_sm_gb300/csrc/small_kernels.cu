// Bandwidth-bound kernels around the backward:
//   preprocess  D = rowsum(fp32(O) * fp32(dO)), zero the fp32 dQ accumulator
//               (SK-16 single-pass FA Grad article, section 3.1 step 4 and
//               section 4.2 row "D"; section 4: atomic targets start at zero)
//   finalize    dQ = bf16(scale * accumulator) (section 3, V2 scales dq;
//               section 4.2 row dQ)
//   zero fill   padding rows of dK / dV
// Each is a grid-stride loop over 16-byte vectors, sized to a few CTAs per SM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace fa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ float dot8(uint4 a, uint4 b) {
  float s = bf_lo(a.x) * bf_lo(b.x);
  s = fmaf(bf_hi(a.x), bf_hi(b.x), s);
  s = fmaf(bf_lo(a.y), bf_lo(b.y), s);
  s = fmaf(bf_hi(a.y), bf_hi(b.y), s);
  s = fmaf(bf_lo(a.z), bf_lo(b.z), s);
  s = fmaf(bf_hi(a.z), bf_hi(b.z), s);
  s = fmaf(bf_lo(a.w), bf_lo(b.w), s);
  s = fmaf(bf_hi(a.w), bf_hi(b.w), s);
  return s;
}

// One group of D/8 lanes per (row, head): each lane dots 8 elements, the
// group reduces with shuffles.  Loop bounds are warp-uniform so every lane
// reaches every shuffle.
template <int D>
__global__ void __launch_bounds__(kThreads) preprocess_kernel(const uint16_t* __restrict__ o,
                                                              const uint16_t* __restrict__ dout,
                                                              float* __restrict__ Dout, float* __restrict__ acc,
                                                              long long rows) {
  constexpr int G = D / 8;            // lanes per (row, head)
  constexpr int PER_WARP = 32 / G;    // (row, head) pairs per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;
  const long long warp = (static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * kThreads) >> 5;
  for (long long base = warp * PER_WARP; base < rows; base += nwarps * PER_WARP) {
    const long long r = base + lane / G;
    const bool ok = r < rows;
    float s = 0.f;
    if (ok) {
      const uint4 a = ldg_stream(o + r * D + sub * 8);
      const uint4 b = ldg_stream(dout + r * D + sub * 8);
      s = dot8(a, b);
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (ok) {
      if (sub == 0) Dout[r] = s;
      float4* z = reinterpret_cast<float4*>(acc + r * D + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kThreads) finalize_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                            long long n8, float scale) {
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n8; i += stride) {
    const uint4 a = ldg_stream(acc + i * 8);
    const uint4 b = ldg_stream(acc + i * 8 + 4);
    uint4 w;
    w.x = pack2(scale * __uint_as_float(a.x), scale * __uint_as_float(a.y));
    w.y = pack2(scale * __uint_as_float(a.z), scale * __uint_as_float(a.w));
    w.z = pack2(scale * __uint_as_float(b.x), scale * __uint_as_float(b.y));
    w.w = pack2(scale * __uint_as_float(b.z), scale * __uint_as_float(b.w));
    reinterpret_cast<uint4*>(dq)[i] = w;
  }
}

__global__ void __launch_bounds__(kThreads) zero_kernel(uint4* __restrict__ p, long long n16) {
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

int grid_for(long long work_items) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 152;
  long long want = (work_items + kThreads - 1) / kThreads;
  long long cap = static_cast<long long>(sms) * 8;   // 8 CTAs of 256 threads fill an SM
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

}  // namespace

cudaError_t launch_preprocess(const uint16_t* o, const uint16_t* dout, float* D, float* dq_acc, long long rows,
                              int head_dim, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const long long lanes = rows * (head_dim / 8);
  const int grid = grid_for(lanes);
  if (head_dim == 64)
    preprocess_kernel<64><<<grid, kThreads, 0, s>>>(o, dout, D, dq_acc, rows);
  else if (head_dim == 256)
    preprocess_kernel<256><<<grid, kThreads, 0, s>>>(o, dout, D, dq_acc, rows);
  else
    preprocess_kernel<128><<<grid, kThreads, 0, s>>>(o, dout, D, dq_acc, rows);
  return cudaGetLastError();
}

cudaError_t launch_dq_finalize(const float* acc, uint16_t* dq, long long elems, float scale, cudaStream_t s) {
  if (elems <= 0) return cudaSuccess;
  const long long n8 = elems / 8;
  finalize_kernel<<<grid_for(n8), kThreads, 0, s>>>(acc, dq, n8, scale);
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(void* p, long long bytes, cudaStream_t s) {
  if (bytes <= 0) return cudaSuccess;
  const long long n16 = bytes / 16;
  zero_kernel<<<grid_for(n16), kThreads, 0, s>>>(reinterpret_cast<uint4*>(p), n16);
  return cudaGetLastError();
}

}  // namespace fa
