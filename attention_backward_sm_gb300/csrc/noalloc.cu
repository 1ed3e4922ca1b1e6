// fa_bwd_noalloc: the whole backward (preprocess -> fa_bwd -> finalize)
// for callers that cannot allocate device memory themselves.
//
// Some callers cannot call cudaMalloc or an allocating library routine:
// runtimes that own all device memory through their own planner and hand
// a kernel library nothing but its inputs and outputs, latency-critical
// serving loops in which an allocation would stall the device, and hosts
// that run under a fixed device-memory budget.  The ordinary path needs two
// caller-provided scratch buffers (D and the fp32 dQ accumulator); this
// entry point keeps them in one statically sized array that lives in this
// module for the life of the process instead.
//
// The array is shared by every call on a device and keeps the previous
// call's contents; fa_bwd_preprocess rewrites D and zeroes the accumulator
// at the start of every call, so nothing carries over.  Two calls whose
// work overlaps on the GPU (different streams, or threads that do not
// order their streams) race on the array.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fabwd.h"
#include "internal.h"

namespace {

// File-scope scratch: every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A non-null, 256-byte aligned value that stands in for the scratch
// pointers while the arguments are checked; it is never dereferenced.
float* const kStandIn = reinterpret_cast<float*>(static_cast<uintptr_t>(256));

}  // namespace

extern "C" int fa_bwd_noalloc(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* o,
                              const fa_bf16* dout, const float* m, const float* l, fa_bf16* dq, fa_bf16* dk,
                              fa_bf16* dv, const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
                              const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q,
                              int total_kv, int heads, int head_dim, int causal, float scale, fa_stream_t stream) {
  // Every check comes before the first CUDA call, so a rejected call
  // launches nothing.
  if (total_q < 0 || heads < 1)
    return fa::set_last_error(FA_ERR_INVALID_ARG, "fa_bwd_noalloc: need total_q >= 0 and heads >= 1");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fa::set_last_error(FA_ERR_UNSUPPORTED, "fa_bwd_noalloc: head_dim must be 64, 128 or 256, got %d",
                              head_dim);
  if (causal != 0 && causal != 1)
    return fa::set_last_error(FA_ERR_INVALID_ARG, "fa_bwd_noalloc: causal must be 0 or 1, got %d", causal);
  const size_t d_bytes = round256(static_cast<size_t>(total_q) * heads * sizeof(float));
  const size_t acc_bytes = static_cast<size_t>(total_q) * heads * head_dim * sizeof(float);
  if (d_bytes + acc_bytes > FA_NOALLOC_SCRATCH_BYTES)
    return fa::set_last_error(FA_ERR_INVALID_ARG,
                              "fa_bwd_noalloc: this problem needs %zu bytes of scratch (D and the fp32 dQ "
                              "accumulator: total_q*heads*(head_dim+1)*4, rounded) but the fixed array holds %zu",
                              d_bytes + acc_bytes, static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES));
  // o and dout are read by the preprocess step, dq is written by the finalize step
  const uintptr_t al = reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout) |
                       reinterpret_cast<uintptr_t>(dq);
  if (total_q > 0 && (!o || !dout || !dq))
    return fa::set_last_error(FA_ERR_INVALID_ARG, "fa_bwd_noalloc: o, dout or dq is NULL");
  if (al & 15u) return fa::set_last_error(FA_ERR_INVALID_ARG, "fa_bwd_noalloc: o, dout and dq must be 16-byte aligned");
  // everything fa_bwd checks (shapes, offsets, pointers, alignment, scale,
  // the device), with stand-ins for the scratch pointers
  int rc = fa::bwd_impl(q, k, v, dout, m, l, kStandIn, kStandIn, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host,
                        batch, total_q, total_kv, heads, heads, head_dim, causal, 0, 0, scale, FA_DQ_ATOMIC, nullptr,
                        0, reinterpret_cast<cudaStream_t>(stream), /*check_only=*/true);
  if (rc != FA_OK) return rc;
  // The array's device address in the current context, looked up on every
  // call (a host-side table lookup once the module is loaded; a cached
  // value would go stale when the caller switches contexts or resets the
  // device).  The first call in a context loads the module.
  void* base = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&base, g_noalloc_scratch);
  if (e != cudaSuccess)
    return fa::set_last_error(FA_ERR_CUDA, "fa_bwd_noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                              cudaGetErrorString(e));
  float* D = static_cast<float*>(base);
  float* acc = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + d_bytes);
  rc = fa_bwd_preprocess(o, dout, D, acc, total_q, heads, head_dim, stream);
  if (rc != FA_OK) return rc;
  rc = fa_bwd(q, k, v, dout, m, l, D, acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch, total_q,
              total_kv, heads, head_dim, causal, scale, FA_DQ_ATOMIC, nullptr, 0, stream);
  if (rc != FA_OK) return rc;
  return fa_bwd_dq_finalize(acc, dq, total_q, heads, head_dim, scale, stream);
}
