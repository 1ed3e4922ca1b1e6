// C-ABI layer of libfabwd.so: argument checks, TMA descriptor encoding and
// kernel launches.  Declarations and their contracts are in include/fabwd.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/fabwd.h"
#include "internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return FA_OK;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Checks host offsets: batch+1 entries, cu[0] = 0, non-decreasing,
// cu[batch] <= total.  Reports the longest sequence.
int check_offsets(const int32_t* cu, int batch, int total, const char* name, int* max_len) {
  if (cu == nullptr) return fail(FA_ERR_INVALID_ARG, "%s_host is NULL", name);
  if (cu[0] != 0) return fail(FA_ERR_INVALID_ARG, "%s_host[0] must be 0, got %d", name, cu[0]);
  int mx = 0;
  for (int b = 0; b < batch; ++b) {
    const long long len = static_cast<long long>(cu[b + 1]) - cu[b];
    if (len < 0)
      return fail(FA_ERR_INVALID_ARG, "%s_host must be non-decreasing: entry %d is %d, entry %d is %d", name, b + 1,
                  cu[b + 1], b, cu[b]);
    if (len > mx) mx = static_cast<int>(len);
  }
  if (cu[batch] > total)
    return fail(FA_ERR_INVALID_ARG, "%s_host[batch] = %d exceeds the tensor's %d rows", name, cu[batch], total);
  *max_len = mx;
  return FA_OK;
}

int check_shape(int batch, int total_q, int total_kv, int heads, int head_dim) {
  if (batch < 0) return fail(FA_ERR_INVALID_ARG, "batch must be >= 0, got %d", batch);
  if (heads < 1) return fail(FA_ERR_INVALID_ARG, "heads must be >= 1, got %d", heads);
  if (total_q < 0 || total_kv < 0) return fail(FA_ERR_INVALID_ARG, "total_q and total_kv must be >= 0");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(FA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256, got %d", head_dim);
  if (static_cast<long long>(heads) * head_dim > 65535 * 64)
    return fail(FA_ERR_UNSUPPORTED, "heads * head_dim too large for a 2-D tensor map");
  return FA_OK;
}

int check_mask(int mask, int window) {
  if (mask != FA_MASK_NONE && mask != FA_MASK_CAUSAL && mask != FA_MASK_CAUSAL_BOTTOM_RIGHT)
    return fail(FA_ERR_INVALID_ARG, "mask must be 0 (none), 1 (causal) or 2 (causal, bottom-right), got %d", mask);
  if (window < 0) return fail(FA_ERR_INVALID_ARG, "window must be >= 0, got %d", window);
  if (window > 0 && mask == FA_MASK_NONE)
    return fail(FA_ERR_INVALID_ARG, "a sliding window needs a causal mask (it sees the keys (pos - window, pos])");
  return FA_OK;
}

// A window at least as long as both sequences together excludes no key that
// the causal mask admits; it is dropped so that device arithmetic on it
// cannot overflow.
int effective_window(int window, int max_q, int max_kv) {
  return static_cast<long long>(window) >= static_cast<long long>(max_q) + max_kv ? 0 : window;
}

int check_groups(int heads, int heads_kv) {
  if (heads_kv < 1 || heads % heads_kv != 0)
    return fail(FA_ERR_INVALID_ARG, "query heads (%d) must be a positive multiple of key/value heads (%d)", heads,
                heads_kv);
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A [rows, heads*head_dim] view with 128-byte swizzle: bf16 with boxes of
// 64 columns x box_rows rows (operand tiles; rows past `rows` read as
// zero), or fp32 with 32 x 32 boxes (the dQ accumulator; rows past `rows`
// are not written).
int make_map(CUtensorMap* m, const void* base, int rows, int heads, int head_dim, const char* name,
             bool fp32 = false, int box_rows = 128) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t esize = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads) * head_dim, static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * head_dim * esize};
  cuuint32_t box[2] = {fp32 ? 32u : 64u, fp32 ? 32u : static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return FA_OK;
}

// Unique id of the calling thread's current context (0 if unavailable).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// A second stream of the device, with the events that fork it from and
// join it back into a caller's stream.  It belongs to the context that was
// current when it was made: a call from another context (or after the
// device was reset, which makes a new context) makes new ones and leaves
// the old handles alone.  Guarded by g_side_mu, which is held from the fork
// to the join so that concurrent calls cannot interleave their events.
struct SideStream {
  unsigned long long ctx_id = 0;
  cudaStream_t st = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

SideStream* side_stream_locked(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  const unsigned long long id = current_context_id();
  if (id == 0) return nullptr;
  SideStream& ss = g_side[dev];
  if (ss.st && ss.ctx_id == id) return &ss;
  SideStream fresh;
  fresh.ctx_id = id;
  if (cudaStreamCreateWithFlags(&fresh.st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
  if (cudaEventCreateWithFlags(&fresh.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&fresh.join, cudaEventDisableTiming) != cudaSuccess) {
    if (fresh.fork) cudaEventDestroy(fresh.fork);
    cudaStreamDestroy(fresh.st);
    return nullptr;
  }
  ss = fresh;
  return &ss;
}

int check_device() {
  static std::atomic<unsigned long long> ok_mask{0};   // devices already found to be sm_103
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (ok_mask.load(std::memory_order_acquire) & bit)) return FA_OK;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(FA_ERR_UNSUPPORTED, "this library is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
  if (bit) ok_mask.fetch_or(bit, std::memory_order_release);
  return FA_OK;
}

}  // namespace

namespace fa {
int set_last_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}
}  // namespace fa

extern "C" {

const char* fa_last_error(void) { return g_err; }

namespace {

// Shared body of the forward-statistics entry points; stats_lse selects
// lse = m + ln(l) written into m (l unused) instead of the pair (m, l).
int fwd_impl(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, fa_bf16* o, float* m, float* l,
             const int32_t* cu_q_dev, const int32_t* cu_kv_dev, const int32_t* cu_q_host, const int32_t* cu_kv_host,
             int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim, int mask, int window,
             int stats_lse, float scale, fa_stream_t stream) {
  int rc = check_shape(batch, total_q, total_kv, heads, head_dim);
  if (rc) return rc;
  if ((rc = check_groups(heads, heads_kv))) return rc;
  if ((rc = check_mask(mask, window))) return rc;
  if (!isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  int max_q = 0, max_kv = 0;
  if ((rc = check_offsets(cu_q_host, batch, total_q, "cu_q", &max_q))) return rc;
  if ((rc = check_offsets(cu_kv_host, batch, total_kv, "cu_kv", &max_kv))) return rc;
  if (batch == 0 || max_q == 0) return ok();
  if (!q || !k || !v || !o || !m || (!stats_lse && !l) || !cu_q_dev || !cu_kv_dev)
    return fail(FA_ERR_INVALID_ARG, "a device pointer is NULL");
  if ((rc = check_device())) return rc;
  const void* al[] = {q, k, v, o};
  for (const void* ptr : al)
    if (!aligned16(ptr)) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  fa::FwdTcParams p;
  memset(&p, 0, sizeof(p));
  // With no key rows at all no key tile is ever loaded; the query tensor
  // then stands in as a valid address for the (unused) key and value maps.
  const bool no_keys = total_kv == 0;
  if ((rc = make_map(&p.tm_q, q, total_q, heads, head_dim, "q"))) return rc;
  const int kv_box = head_dim == 256 ? 64 : 128;   // key rows per block of the forward kernel
  if ((rc = make_map(&p.tm_k, no_keys ? static_cast<const void*>(q) : k, no_keys ? total_q : total_kv,
                     no_keys ? heads : heads_kv, head_dim, "k", false, kv_box)))
    return rc;
  if ((rc = make_map(&p.tm_v, no_keys ? static_cast<const void*>(q) : v, no_keys ? total_q : total_kv,
                     no_keys ? heads : heads_kv, head_dim, "v", false, kv_box)))
    return rc;
  p.o = o;
  p.m = m;
  p.l = l;
  p.cu_q = cu_q_dev;
  p.cu_kv = cu_kv_dev;
  p.heads = heads;
  p.heads_kv = heads_kv;
  p.causal = mask != FA_MASK_NONE;
  p.bottom_right = mask == FA_MASK_CAUSAL_BOTTOM_RIGHT;
  p.window = effective_window(window, max_q, max_kv);
  p.stats_lse = stats_lse;
  p.max_kv = max_kv;
  p.scale = scale;
  cudaError_t e = fa::launch_fwd_main(p, head_dim, batch, (max_q + 127) / 128, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ok();
}

}  // namespace

int fa_fwd_stats_ex(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, fa_bf16* o, float* m, float* l,
                    const int32_t* cu_q_dev, const int32_t* cu_kv_dev, const int32_t* cu_q_host,
                    const int32_t* cu_kv_host, int batch, int total_q, int total_kv, int heads, int heads_kv,
                    int head_dim, int mask, int window, float scale, fa_stream_t stream) {
  return fwd_impl(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch, total_q, total_kv, heads,
                  heads_kv, head_dim, mask, window, 0, scale, stream);
}

int fa_fwd_lse(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, fa_bf16* o, float* lse,
               const int32_t* cu_q_dev, const int32_t* cu_kv_dev, const int32_t* cu_q_host,
               const int32_t* cu_kv_host, int batch, int total_q, int total_kv, int heads, int heads_kv,
               int head_dim, int mask, int window, float scale, fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, nullptr, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch, total_q, total_kv,
                  heads, heads_kv, head_dim, mask, window, 1, scale, stream);
}

int fa_fwd_stats_gqa(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, fa_bf16* o, float* m, float* l,
                     const int32_t* cu_q_dev, const int32_t* cu_kv_dev, const int32_t* cu_q_host,
                     const int32_t* cu_kv_host, int batch, int total_q, int total_kv, int heads, int heads_kv,
                     int head_dim, int causal, float scale, fa_stream_t stream) {
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
  return fa_fwd_stats_ex(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch, total_q, total_kv,
                         heads, heads_kv, head_dim, causal, 0, scale, stream);
}

int fa_fwd_stats(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, fa_bf16* o, float* m, float* l,
                 const int32_t* cu_q_dev, const int32_t* cu_kv_dev, const int32_t* cu_q_host,
                 const int32_t* cu_kv_host, int batch, int total_q, int total_kv, int heads, int head_dim, int causal,
                 float scale, fa_stream_t stream) {
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
  return fa_fwd_stats_ex(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch, total_q, total_kv,
                         heads, heads, head_dim, causal, 0, scale, stream);
}

int fa_bwd_preprocess(const fa_bf16* o, const fa_bf16* dout, float* D, float* dq_acc, int total_q, int heads,
                      int head_dim, fa_stream_t stream) {
  int rc = check_shape(0, total_q, 0, heads, head_dim);
  if (rc) return rc;
  if (total_q == 0) return ok();
  if (!o || !dout || !D || !dq_acc) return fail(FA_ERR_INVALID_ARG, "a device pointer is NULL");
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dq_acc))
    return fail(FA_ERR_INVALID_ARG, "o, dout and dq_acc must be 16-byte aligned");
  if ((rc = check_device())) return rc;
  cudaError_t e = fa::launch_preprocess(o, dout, D, dq_acc, static_cast<long long>(total_q) * heads, head_dim,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
  return ok();
}

size_t fa_bwd_workspace_size(const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int heads,
                             int head_dim, int causal, int dq_mode) {
  (void)cu_kv_host;
  (void)causal;
  if (check_shape(batch, 0, 0, heads, head_dim)) return 0;
  // Atomic mode, and the deterministic mode at head_dim 64 and 128 (whose
  // dQ comes from a kernel that sums every row in one CTA), need none.
  if (dq_mode == FA_DQ_ATOMIC || (dq_mode == FA_DQ_DETERMINISTIC && head_dim != 256)) {
    ok();
    return 0;
  }
  if (dq_mode != FA_DQ_DETERMINISTIC) {
    fail(FA_ERR_INVALID_ARG, "dq_mode must be 0 or 1, got %d", dq_mode);
    return 0;
  }
  if (!cu_q_host) {
    fail(FA_ERR_INVALID_ARG, "cu_q_host is NULL");
    return 0;
  }
  int max_q = 0;
  for (int b = 0; b < batch; ++b) max_q = cu_q_host[b + 1] - cu_q_host[b] > max_q ? cu_q_host[b + 1] - cu_q_host[b] : max_q;
  ok();
  // head_dim 256: one int32 counter per (batch, head, 64-row query block,
  // head-dim half, 32-dim quarter) and the work-item counter, rounded to 256 B
  const size_t n = static_cast<size_t>(batch) * heads * ((max_q + 63) / 64) * 8 + 1;
  return ((n * 4 + 255) / 256) * 256;
}

}  // extern "C"

namespace fa {

// Shared body of the backward entry points; stats_lse: m holds lse and l is
// unused.  check_only: run every host-side check (including the device
// check) and return before anything is launched.
int bwd_impl(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout, const float* m,
             const float* l, const float* D, float* dq_acc, fa_bf16* dk, fa_bf16* dv, const int32_t* cu_q_dev,
             const int32_t* cu_kv_dev, const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q,
             int total_kv, int heads, int heads_kv, int head_dim, int mask, int window, int stats_lse, float scale,
             int dq_mode, void* workspace, size_t workspace_bytes, fa_stream_t stream, bool check_only) {
  int rc = check_shape(batch, total_q, total_kv, heads, head_dim);
  if (rc) return rc;
  if ((rc = check_groups(heads, heads_kv))) return rc;
  if ((rc = check_mask(mask, window))) return rc;
  const int causal = mask != FA_MASK_NONE;
  if (dq_mode != FA_DQ_ATOMIC && dq_mode != FA_DQ_DETERMINISTIC)
    return fail(FA_ERR_INVALID_ARG, "dq_mode must be 0 or 1, got %d", dq_mode);
  if (!isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  int max_q = 0, max_kv = 0;
  if ((rc = check_offsets(cu_q_host, batch, total_q, "cu_q", &max_q))) return rc;
  if ((rc = check_offsets(cu_kv_host, batch, total_kv, "cu_kv", &max_kv))) return rc;
  const int kv_used = batch > 0 ? cu_kv_host[batch] : 0;
  const bool has_work = batch > 0 && max_kv > 0;
  if (!has_work && total_kv == kv_used) return ok();
  if ((total_kv > 0 && (!dk || !dv)) ||
      (has_work && (!k || !v || !cu_q_dev || !cu_kv_dev)) ||
      (has_work && max_q > 0 && (!q || !dout || !m || (!stats_lse && !l) || !D || !dq_acc)))
    return fail(FA_ERR_INVALID_ARG, "a device pointer is NULL");
  const void* al[] = {q, k, v, dout, dq_acc, dk, dv};
  for (const void* ptr : al)
    if (ptr && !aligned16(ptr)) return fail(FA_ERR_INVALID_ARG, "q, k, v, dout, dq_acc, dk, dv must be 16-byte aligned");
  const size_t need = fa_bwd_workspace_size(cu_q_host, cu_kv_host, batch, heads, head_dim, causal, dq_mode);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(FA_ERR_INVALID_ARG, "workspace of %zu bytes needed, got %zu", need, workspace_bytes);
  if ((rc = check_device())) return rc;
  if (check_only) return ok();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (total_kv > kv_used) {
    const long long row_bytes = static_cast<long long>(heads_kv) * head_dim * 2;
    cudaError_t e = fa::launch_zero_fill(dk + static_cast<long long>(kv_used) * heads_kv * head_dim,
                                         (total_kv - kv_used) * row_bytes, s);
    if (e == cudaSuccess)
      e = fa::launch_zero_fill(dv + static_cast<long long>(kv_used) * heads_kv * head_dim,
                               (total_kv - kv_used) * row_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "padding zero fill");
  }
  if (!has_work) return ok();
  fa::BwdParams p;
  memset(&p, 0, sizeof(p));
  // With no query rows at all no query tile is ever loaded; the key tensor
  // then stands in as a valid address for the (unused) query maps.
  const void* qbase = max_q > 0 ? static_cast<const void*>(q) : static_cast<const void*>(k);
  const void* dobase = max_q > 0 ? static_cast<const void*>(dout) : static_cast<const void*>(k);
  const int q_box = head_dim == 256 ? 64 : 128;   // query rows per block of the backward kernel
  if ((rc = make_map(&p.tm_q, qbase, max_q > 0 ? total_q : total_kv, max_q > 0 ? heads : heads_kv, head_dim, "q",
                     false, q_box)))
    return rc;
  if ((rc = make_map(&p.tm_k, k, total_kv, heads_kv, head_dim, "k"))) return rc;
  if ((rc = make_map(&p.tm_v, v, total_kv, heads_kv, head_dim, "v"))) return rc;
  if ((rc = make_map(&p.tm_do, dobase, max_q > 0 ? total_q : total_kv, max_q > 0 ? heads : heads_kv, head_dim,
                     "dout", false, q_box)))
    return rc;
  if (max_q > 0 && (rc = make_map(&p.tm_dq, dq_acc, total_q, heads, head_dim, "dq_acc", true))) return rc;
  if ((rc = make_map(&p.tm_dk, dk, total_kv, heads_kv, head_dim, "dk"))) return rc;
  if ((rc = make_map(&p.tm_dv, dv, total_kv, heads_kv, head_dim, "dv"))) return rc;
  p.m = m;
  p.l = l;
  p.D = D;
  p.dq_acc = dq_acc;
  p.dk = dk;
  p.dv = dv;
  p.cu_q = cu_q_dev;
  p.cu_kv = cu_kv_dev;
  p.heads = heads;
  p.heads_kv = heads_kv;
  p.causal = causal;
  p.bottom_right = mask == FA_MASK_CAUSAL_BOTTOM_RIGHT;
  p.window = effective_window(window, max_q, max_kv);
  p.stats_lse = stats_lse;
  p.dq_mode = dq_mode;
  p.max_q_blocks = (max_q + q_box - 1) / q_box;
  p.kv_reverse = (head_dim == 256 && dq_mode == FA_DQ_DETERMINISTIC && causal) ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.tickets = static_cast<int*>(workspace);
  if (head_dim == 256 && dq_mode == FA_DQ_DETERMINISTIC)
    p.work_counter = p.tickets + static_cast<size_t>(batch) * heads * ((max_q + 63) / 64) * 8;
  if (need > 0) {
    cudaError_t e = fa::launch_zero_fill(workspace, static_cast<long long>(need), s);
    if (e != cudaSuccess) return cuda_fail(e, "ticket reset");
  }
  cudaError_t e;
  if (head_dim == 256) {
    e = fa::launch_bwd256(p, batch, (max_kv + 127) / 128, s);
  } else if (dq_mode == FA_DQ_ATOMIC) {
    e = fa::launch_bwd_main(p, head_dim, batch, (max_kv + 127) / 128, true, s);
  } else {
    // deterministic: dK and dV from the key-block-outer kernel, dQ from the
    // query-block-outer one (each row summed by one CTA in a fixed order).
    // The two are independent: the dQ kernel runs on a second stream,
    // forked from and joined back into the caller's, so that its CTAs fill
    // the SMs the other kernel's last wave leaves idle.  Under stream
    // capture, or without a second stream, both run in order on `s`.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream* side = (cap == cudaStreamCaptureStatusNone && max_q > 0) ? side_stream_locked(dev) : nullptr;
    if (side == nullptr) {
      e = fa::launch_bwd_main(p, head_dim, batch, (max_kv + 127) / 128, false, s);
      if (e == cudaSuccess && max_q > 0) e = fa::launch_dq(p, head_dim, batch, max_kv, s);
    } else {
      e = cudaEventRecord(side->fork, s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side->st, side->fork, 0);
      if (e == cudaSuccess) {
        const cudaError_t e_dq = fa::launch_dq(p, head_dim, batch, max_kv, side->st);
        const cudaError_t e_kv = fa::launch_bwd_main(p, head_dim, batch, (max_kv + 127) / 128, false, s);
        // the caller's stream waits for the dQ kernel, whatever happened
        cudaError_t e_join = cudaEventRecord(side->join, side->st);
        if (e_join == cudaSuccess) e_join = cudaStreamWaitEvent(s, side->join, 0);
        if (e_join != cudaSuccess) cudaStreamSynchronize(side->st);
        e = e_dq != cudaSuccess ? e_dq : (e_kv != cudaSuccess ? e_kv : e_join);
      }
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "bwd launch");
  return ok();
}

}  // namespace fa

extern "C" {

using fa::bwd_impl;

int fa_bwd_ex(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout, const float* m,
              const float* l, const float* D, float* dq_acc, fa_bf16* dk, fa_bf16* dv, const int32_t* cu_q_dev,
              const int32_t* cu_kv_dev, const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q,
              int total_kv, int heads, int heads_kv, int head_dim, int mask, int window, float scale, int dq_mode,
              void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(q, k, v, dout, m, l, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch, total_q,
                  total_kv, heads, heads_kv, head_dim, mask, window, 0, scale, dq_mode, workspace, workspace_bytes,
                  stream, false);
}

int fa_bwd_lse(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout, const float* lse,
               const float* D, float* dq_acc, fa_bf16* dk, fa_bf16* dv, const int32_t* cu_q_dev,
               const int32_t* cu_kv_dev, const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q,
               int total_kv, int heads, int heads_kv, int head_dim, int mask, int window, float scale, int dq_mode,
               void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(q, k, v, dout, lse, nullptr, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch,
                  total_q, total_kv, heads, heads_kv, head_dim, mask, window, 1, scale, dq_mode, workspace,
                  workspace_bytes, stream, false);
}

int fa_bwd_gqa(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout, const float* m,
               const float* l, const float* D, float* dq_acc, fa_bf16* dk, fa_bf16* dv, const int32_t* cu_q_dev,
               const int32_t* cu_kv_dev, const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q,
               int total_kv, int heads, int heads_kv, int head_dim, int causal, float scale, int dq_mode,
               void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
  return fa_bwd_ex(q, k, v, dout, m, l, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch,
                   total_q, total_kv, heads, heads_kv, head_dim, causal, 0, scale, dq_mode, workspace,
                   workspace_bytes, stream);
}

int fa_bwd(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout, const float* m, const float* l,
           const float* D, float* dq_acc, fa_bf16* dk, fa_bf16* dv, const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
           const int32_t* cu_q_host, const int32_t* cu_kv_host, int batch, int total_q, int total_kv, int heads,
           int head_dim, int causal, float scale, int dq_mode, void* workspace, size_t workspace_bytes,
           fa_stream_t stream) {
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
  return fa_bwd_ex(q, k, v, dout, m, l, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, batch,
                   total_q, total_kv, heads, heads, head_dim, causal, 0, scale, dq_mode, workspace, workspace_bytes,
                   stream);
}

int fa_bwd_dq_finalize(const float* dq_acc, fa_bf16* dq, int total_q, int heads, int head_dim, float scale,
                       fa_stream_t stream) {
  int rc = check_shape(0, total_q, 0, heads, head_dim);
  if (rc) return rc;
  if (total_q == 0) return ok();
  if (!dq_acc || !dq) return fail(FA_ERR_INVALID_ARG, "a device pointer is NULL");
  if (!aligned16(dq_acc) || !aligned16(dq)) return fail(FA_ERR_INVALID_ARG, "dq_acc and dq must be 16-byte aligned");
  if (!isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if ((rc = check_device())) return rc;
  cudaError_t e = fa::launch_dq_finalize(dq_acc, dq, static_cast<long long>(total_q) * heads * head_dim, scale,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  return ok();
}

int fa_selftest_wait_timeout(fa_stream_t stream) {
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = fa::launch_wait_timeout(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ok();
}

int fa_check_device_status(fa_stream_t stream) {
  int st = 0, st256 = 0, st_dq = 0, st_fwd = 0;
  int e = fa::bwd_read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &st);
  if (e == 0) e = fa::bwd256_read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &st256);
  if (e == 0) e = fa::dq_read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &st_dq);
  if (e == 0) e = fa::fwd_read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &st_fwd);
  if (st == 0) st = st256;
  if (st == 0) st = st_dq;
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "fa_check_device_status");
  if (st == 4) return fail(FA_ERR_TIMEOUT, "a device-side wait in fa_bwd ran out of time (status %d)", st);
  if (st != 0) return fail(FA_ERR_CUDA, "fa_bwd recorded device status %d", st);
  if (st_fwd == 4) return fail(FA_ERR_TIMEOUT, "a device-side wait in the forward ran out of time (status %d)", st_fwd);
  if (st_fwd != 0) return fail(FA_ERR_CUDA, "the forward recorded device status %d", st_fwd);
  return ok();
}

}  // extern "C"
