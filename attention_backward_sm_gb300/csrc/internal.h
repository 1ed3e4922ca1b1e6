// Launch interfaces shared between the C-ABI layer (api.cu) and the kernel
// translation units.  Host-only declarations; no kernel code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace fa {

// Everything the single-pass backward kernel needs, passed by value as one
// __grid_constant__ parameter (the tensor maps must live in parameter
// space for TMA).
struct BwdParams {
  CUtensorMap tm_q;   // [total_q rows, H*d cols] bf16, box 64 x 128, 128B swizzle
  CUtensorMap tm_k;   // [total_kv rows, H*d cols]
  CUtensorMap tm_v;
  CUtensorMap tm_do;  // [total_q rows, H*d cols]
  CUtensorMap tm_dq;  // dq_acc: [total_q rows, H*d cols] fp32, box 32 x 32, 128B swizzle (reduce-add target)
  CUtensorMap tm_dk;  // dk: [total_kv rows, Hkv*d cols] bf16, box 64 x 128, 128B swizzle (store target)
  CUtensorMap tm_dv;  // dv: as dk
  const float* m;
  const float* l;
  const float* D;
  float* dq_acc;
  uint16_t* dk;
  uint16_t* dv;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  int* tickets;        // deterministic mode at head_dim 256: one counter per (batch, head, 64-row query
                       // block, head-dim half, 32-dim quarter)
  int* work_counter;   // deterministic mode at head_dim 256: CTAs take their work items from it in the
                       // order they start
  int heads;           // query heads
  int heads_kv;        // key/value heads (heads is a multiple of it)
  int causal;          // 1: causal mask (top-left unless bottom_right)
  int bottom_right;    // 1: causal diagonal aligned with the last key (offset s2 - s1 per sequence)
  int window;          // > 0: sliding window, query i sees keys (i + off - window, i + off]
  int stats_lse;       // 1: m holds lse = m + ln(l) per row and l is unused
  int dq_mode;
  int max_q_blocks;    // query blocks of the longest query sequence
  int kv_reverse;      // 1: key blocks are launched from the last one down (head_dim 256, deterministic)
  int batch;           // sequences
  int grid_kv;         // key blocks of the longest key sequence (launched per head)
  int head_chunk;      // (sequence, key/value head) units per launch-order chunk
  float scale;         // softmax scale (multiplies dK in the epilogue)
  float scale_log2;    // scale * log2(e)
};

// head_dim 64 / 128 key-block-outer kernel; with_dq: also add the dQ
// partials into dq_acc (atomic mode), else dK and dV only.
cudaError_t launch_bwd_main(const BwdParams& p, int head_dim, int batch, int max_kv_blocks, bool with_dq,
                            cudaStream_t s);
// head_dim 64 / 128 deterministic dQ (dq_main.cu): stores the unscaled
// dS K sums of every query row into dq_acc, one CTA per query block.
cudaError_t launch_dq(const BwdParams& p, int head_dim, int batch, int max_kv, cudaStream_t s);
int dq_read_and_clear_status(cudaStream_t s, int* status);
// (sequence, key/value head) units per launch-order chunk of a backward grid
// with n_kvb key blocks of bm rows and query blocks of bn rows.
int launch_head_chunk(const BwdParams& p, int batch, int n_kvb, int bm, int bn, int head_dim);
// head_dim 256 (bwd_d256.cu): tm_q / tm_do with 64-row boxes, max_q_blocks in 64-row blocks
cudaError_t launch_bwd256(const BwdParams& p, int batch, int max_kv_blocks, cudaStream_t s);
int bwd256_read_and_clear_status(cudaStream_t s, int* status);
int bwd_read_and_clear_status(cudaStream_t s, int* status);
cudaError_t launch_wait_timeout(cudaStream_t s);

cudaError_t launch_preprocess(const uint16_t* o, const uint16_t* dout, float* D, float* dq_acc, long long rows,
                              int head_dim, cudaStream_t s);
cudaError_t launch_dq_finalize(const float* acc, uint16_t* dq, long long elems, float scale, cudaStream_t s);
cudaError_t launch_zero_fill(void* p, long long bytes, cudaStream_t s);

// Forward statistics on the tensor cores (fwd_main.cu).
struct FwdTcParams {
  CUtensorMap tm_q;    // [total_q, H*d] bf16, 128x64 boxes, 128-byte swizzle
  CUtensorMap tm_k;    // [total_kv, Hkv*d]
  CUtensorMap tm_v;
  uint16_t* o;
  float* m;            // m, or lse when stats_lse
  float* l;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  int heads;
  int heads_kv;
  int causal;
  int bottom_right;
  int window;
  int stats_lse;
  int max_kv;          // longest key sequence (used on the host for the launch order)
  int batch;           // sequences
  int head_chunk;      // (sequence, query head) units per launch-order chunk
  float scale;
};
cudaError_t launch_fwd_main(const FwdTcParams& p, int head_dim, int batch, int max_q_blocks, cudaStream_t s);
int fwd_read_and_clear_status(cudaStream_t s, int* status);

// Sets a kernel's dynamic shared-memory limit once per device (the first
// call with that device current); `done` is the kernel's per-device mask.
inline cudaError_t set_smem_once(const void* func, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Records a message for fa_last_error() on the calling thread and returns code.
int set_last_error(int code, const char* fmt, ...);

// Shared body of fa_bwd / fa_bwd_gqa / fa_bwd_ex / fa_bwd_lse (api.cu), with
// the arguments of fa_bwd_ex plus stats_lse (m holds lse, l unused) and
// check_only (every host-side check, nothing launched).  Returns an fa_status.
int bwd_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout, const float* m,
             const float* l, const float* D, float* dq_acc, uint16_t* dk, uint16_t* dv, const int32_t* cu_q_dev,
             const int32_t* cu_kv_dev, const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q,
             int total_kv, int heads, int heads_kv, int head_dim, int mask, int window, int stats_lse, float scale,
             int dq_mode, void* workspace, size_t workspace_bytes, cudaStream_t stream, bool check_only);

}  // namespace fa
