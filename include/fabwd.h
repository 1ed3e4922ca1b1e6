/*
 * fabwd.h -- C ABI of libfabwd.so, a single-pass flash-attention backward
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (cited by page title and section):
 *   "PyPTO-Gym SK-16: single-pass Attention backward (FA Grad)" article,
 *   section 3 (kernel skeleton with inputs q, k, v, o, do, l, m and outputs
 *   dq, dk, dv over packed variable-length batches with cumulative offsets
 *   actual_q / actual_kv), section 3.1 (the eight per-block steps) and
 *   section 4.2 (dtype table).  For each sequence b and head h, with
 *   X = scale * Q K^T (masked entries -inf):
 *       P  = exp(X - m) / l              (m, l given, never recomputed)
 *       dP = dO V^T,  D = rowsum(O * dO), dS = P * (dP - D)
 *       dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K
 *   The causal mask is top-left aligned (key j visible to query i iff
 *   j <= i, local indices; the JAX cuDNN wrapper's MaskType.CAUSAL).
 *
 * Conventions shared by every entry point:
 *   - Tensors are packed and contiguous.  q, o, dout, dq: [total_q, H, d];
 *     k, v, dk, dv: [total_kv, H, d], or [total_kv, Hkv, d] in the entry
 *     points that take heads_kv (grouped-query attention, Hkv divides H);
 *     m, l, D: [total_q, H] (float32).
 *     Element type fa_bf16 is the raw 16-bit pattern of a bfloat16.
 *     The head h of row r sits at element offset (r * H + h) * d.
 *   - cu_q / cu_kv are int32 cumulative offsets with batch+1 entries,
 *     cu[0] = 0, non-decreasing, cu[batch] <= total.  Sequence b owns
 *     rows [cu[b], cu[b+1]).  Rows at or beyond cu[batch] are padding.
 *     Entry points that take both a device and a host copy need both to
 *     hold the same values: the host copy sizes the launch.
 *   - All device pointers are caller-owned device memory, 16-byte aligned.
 *     The library allocates no device memory on these paths.
 *   - head_dim must be 64, 128 or 256 (the JAX cuDNN wrapper's
 *     check_is_flash_attention admits head dims up to 256); heads >= 1.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *     default stream) and returns FA_OK or an error code.  Arguments are
 *     checked on the host before anything is launched; on an error nothing
 *     is launched and fa_last_error() describes the problem.
 *   - Device-side waits are bounded (20 s of wall time each).  A kernel
 *     whose internal wait runs out records FA_ERR_TIMEOUT in a device
 *     status word and returns early, leaving its outputs incomplete;
 *     fa_check_device_status() reads and clears the word.  A call's outputs
 *     are valid only once a later fa_check_device_status() has returned
 *     FA_OK (the Python binding's high-level functions do this by default).
 */
#ifndef FABWD_H
#define FABWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fa_bf16;               /* bfloat16 bit pattern */
typedef struct CUstream_st* fa_stream_t;  /* same type as cudaStream_t */

enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null pointer, bad offsets, bad sizes, misalignment */
    FA_ERR_UNSUPPORTED = 2,   /* head_dim not in {64, 128, 256}, no sm_103a device */
    FA_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
    FA_ERR_TIMEOUT = 4        /* a device-side bounded wait ran out */
};

enum fa_dq_mode {
    FA_DQ_ATOMIC = 0,         /* dQ partials added with fp32 atomics, in any order */
    FA_DQ_DETERMINISTIC = 1   /* bitwise reproducible dQ.  head_dim 64 / 128: the key-block-outer
                                 kernel computes dK and dV only, and a query-block-outer kernel sums
                                 each row of dQ in one CTA in ascending key-block order (no atomics,
                                 no waits between CTAs, no workspace).  The two kernels are
                                 independent: the dQ kernel runs on a second stream that the library
                                 keeps per device and context, forked from `stream` and joined back
                                 into it with events (calls stay ordered on `stream`; while `stream`
                                 is being captured into a graph, both run in order on it).
                                 head_dim 256: dQ partials
                                 added in a fixed key-block order through counters in
                                 fa_bwd_workspace_size() bytes of workspace */
};

/* Masks of the _ex entry points (local indices i of the query, j of the key
 * within one sequence of s1 queries and s2 keys).  JAX
 * fused_attention_stablehlo.py, MaskType and the sliding_window_length
 * argument of dot_product_attention. */
enum fa_mask {
    FA_MASK_NONE = 0,                  /* every key visible */
    FA_MASK_CAUSAL = 1,                /* top-left: j <= i (MaskType.CAUSAL) */
    FA_MASK_CAUSAL_BOTTOM_RIGHT = 2    /* diagonal through the last key: j <= i + s2 - s1
                                          (the pages define no alignment for s1 != s2;
                                          this is the other usual one) */
};

/* Forward statistics used to build consistent backward inputs (support
 * step; the SK-16 article, section 5, says the forward skeleton supplies
 * l and m).  Writes O = softmax(scale*QK^T) V (bf16), m_i = max_j of the
 * scaled scores and l_i = sum_j exp(scaled score - m_i) (float32) for every
 * row of every sequence.  Rows of a sequence with no keys get O = 0,
 * m = -inf, l = 0.  Padding rows are not written.  Runs on the tensor cores
 * (a CTA owns one 128-row query block, or two of them at head_dim 128
 * sharing each key/value tile; O accumulates in tensor memory); q, k, v
 * and o must be 16-byte aligned. */
int fa_fwd_stats(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v,
                 fa_bf16* o, float* m, float* l,
                 const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
                 const int32_t* cu_q_host, const int32_t* cu_kv_host,
                 int batch, int total_q, int total_kv, int heads, int head_dim,
                 int causal, float scale, fa_stream_t stream);

/* fa_fwd_stats for grouped-query attention: k and v have heads_kv heads
 * ([total_kv, heads_kv, d]); query head h uses key/value head
 * h / (heads / heads_kv) (consecutive groups; the JAX cuDNN wrapper's
 * q_N != kv_N case of JAX fused_attention_stablehlo.py,
 * `_dot_product_attention_bwd_cuda_lowering`).
 * heads must be a positive multiple of heads_kv.  fa_fwd_stats is this
 * call with heads_kv = heads. */
int fa_fwd_stats_gqa(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v,
                     fa_bf16* o, float* m, float* l,
                     const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
                     const int32_t* cu_q_host, const int32_t* cu_kv_host,
                     int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim,
                     int causal, float scale, fa_stream_t stream);

/* fa_fwd_stats_gqa with a mask and a sliding window: mask is an fa_mask;
 * window = W > 0 restricts a causal mask to the left window (pos - W, pos]
 * with pos = i (top-left) or i + s2 - s1 (bottom-right), i.e. query i sees
 * keys j with pos - W < j <= pos (JAX dot_product_attention,
 * sliding_window_length); window = 0 means no window, and a window needs
 * a causal mask.  Rows that see no key get O = 0, m = -inf, l = 0. */
int fa_fwd_stats_ex(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v,
                    fa_bf16* o, float* m, float* l,
                    const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
                    const int32_t* cu_q_host, const int32_t* cu_kv_host,
                    int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim,
                    int mask, int window, float scale, fa_stream_t stream);

/* fa_fwd_stats_ex writing the single softmax statistic per row instead of
 * (m, l): lse[r, h] = m + ln(l) (natural log; -inf for rows that see no
 * key).  JAX fused_attention_stablehlo.py keeps one float32 softmax_stat of
 * shape (B, N, T) between its forward and backward calls; lse is the
 * reading of what it holds.  lse: [total_q, H] float32. */
int fa_fwd_lse(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v,
               fa_bf16* o, float* lse,
               const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
               const int32_t* cu_q_host, const int32_t* cu_kv_host,
               int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim,
               int mask, int window, float scale, fa_stream_t stream);

/* Backward preprocess (section 3.1 step 4; section 4.2 row "D"):
 * D[r, h] = sum_k float(O[r,h,k]) * float(dO[r,h,k]) for every row
 * r < total_q, and dq_acc[r, h, :] = 0 (float32 accumulator of
 * [total_q, H, d]; the SK-16 host pre-zeroes its atomic targets, section 4).
 */
int fa_bwd_preprocess(const fa_bf16* o, const fa_bf16* dout, float* D, float* dq_acc,
                      int total_q, int heads, int head_dim, fa_stream_t stream);

/* Bytes of device workspace fa_bwd needs for these shapes and dq_mode
 * (0 for FA_DQ_ATOMIC).  The JAX cuDNN wrapper
 * (fused_attention_stablehlo.py, _dot_product_attention_bwd_cuda_lowering)
 * likewise returns a workspace buffer sized for the backward call, and the
 * SK-16 article (section 6) sizes the kernel's scratch with its
 * max_workspace_kb option; here the caller allocates it.  Returns 0 and
 * sets fa_last_error() on bad arguments, so check fa_last_error() when a
 * mode needs workspace. */
size_t fa_bwd_workspace_size(const int32_t* cu_q_host, const int32_t* cu_kv_host,
                             int batch, int heads, int head_dim, int causal, int dq_mode);

/* The single-pass backward (section 3: C1 -> V1 -> C2 -> V2), key-block
 * outer.  Each CTA owns one (sequence, head, 128-row key block), keeps
 * its dK and dV accumulators in tensor memory for the whole query sweep and
 * writes them once; the unscaled dS K partial of every (query block, key
 * block) pair is added into dq_acc (float32, zeroed by fa_bwd_preprocess).
 * Inputs: q, k, v, dout (bf16), m, l (the forward statistics, consumed as
 * given: section 4.1) and D from fa_bwd_preprocess.  Outputs: dk = bf16(scale
 * * dS^T Q) and dv = bf16(P^T dO) for every key row of every sequence
 * (exact zeros for keys no query sees), zeros in padding rows
 * [cu_kv[batch], total_kv).  dq_acc must then go through
 * fa_bwd_dq_finalize.  workspace: at least fa_bwd_workspace_size() bytes
 * (may be NULL when that is 0); its contents need no initialisation. */
int fa_bwd(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout,
           const float* m, const float* l, const float* D,
           float* dq_acc, fa_bf16* dk, fa_bf16* dv,
           const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
           const int32_t* cu_q_host, const int32_t* cu_kv_host,
           int batch, int total_q, int total_kv, int heads, int head_dim,
           int causal, float scale, int dq_mode,
           void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* fa_bwd for grouped-query attention: q, dout, m, l, D, dq_acc have heads
 * query heads; k, v, dk, dv have heads_kv heads ([total_kv, heads_kv, d]);
 * query head h attends with key/value head h / (heads / heads_kv).  The
 * gradients of a shared key/value head are the sums over its query heads:
 * one CTA per (sequence, key/value head, key block) sweeps the query blocks
 * of every query head of the group, accumulating dK and dV on chip.
 * fa_bwd is this call with heads_kv = heads; the workspace size is that of
 * fa_bwd with `heads` query heads. */
int fa_bwd_gqa(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout,
               const float* m, const float* l, const float* D,
               float* dq_acc, fa_bf16* dk, fa_bf16* dv,
               const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
               const int32_t* cu_q_host, const int32_t* cu_kv_host,
               int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim,
               int causal, float scale, int dq_mode,
               void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* fa_bwd_gqa with a mask and a sliding window (as in fa_fwd_stats_ex).
 * A CTA visits only the query blocks whose tiles the band of visible
 * (query, key) pairs meets; gradients of keys no query sees are exact
 * zeros.  fa_bwd and fa_bwd_gqa are this call with mask = causal and
 * window = 0.  In FA_DQ_DETERMINISTIC mode the key-block order of the dQ
 * additions is fixed for a given mask, so runs are bitwise reproducible.
 *
 * head_dim 256 (all backward entry points): the dK and dV accumulators of a
 * 128-row key block would fill the whole tensor memory, so two CTAs share
 * each (sequence, key/value head, key block), one per half of the head
 * dimension; each computes the full scores and dP and its half of dK, dV
 * and dQ, over 64-row query blocks.  In FA_DQ_DETERMINISTIC mode the
 * workspace then holds one counter per (batch, head, 64-row query block,
 * head-dim half, 32-dim quarter) and one work-item counter from which the
 * CTAs take their order as they start; fa_bwd_workspace_size accounts for
 * both. */
int fa_bwd_ex(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout,
              const float* m, const float* l, const float* D,
              float* dq_acc, fa_bf16* dk, fa_bf16* dv,
              const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
              const int32_t* cu_q_host, const int32_t* cu_kv_host,
              int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim,
              int mask, int window, float scale, int dq_mode,
              void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* fa_bwd_ex consuming the single statistic lse = m + ln(l) (as written by
 * fa_fwd_lse) instead of (m, l): P = exp(scale * S - lse).  Everything else,
 * including the workspace, is as in fa_bwd_ex. */
int fa_bwd_lse(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* dout,
               const float* lse, const float* D,
               float* dq_acc, fa_bf16* dk, fa_bf16* dv,
               const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
               const int32_t* cu_q_host, const int32_t* cu_kv_host,
               int batch, int total_q, int total_kv, int heads, int heads_kv, int head_dim,
               int mask, int window, float scale, int dq_mode,
               void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* dQ write-back (section 3, V2 applies scale to dq; section 4.2 row dQ:
 * fp32 accumulate, then bf16): dq[e] = bf16_rne(scale * dq_acc[e]) for all
 * total_q * heads * head_dim elements. */
int fa_bwd_dq_finalize(const float* dq_acc, fa_bf16* dq, int total_q, int heads,
                       int head_dim, float scale, fa_stream_t stream);

/* Bytes of the library's fixed scratch array used by fa_bwd_noalloc. */
#define FA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* The full backward (fa_bwd_preprocess -> fa_bwd in FA_DQ_ATOMIC mode ->
 * fa_bwd_dq_finalize) without any caller-provided scratch and without any
 * device allocation.  The SK-16 article has no counterpart: this is an
 * interface for callers that cannot call cudaMalloc, such as runtimes that
 * own all device memory through their own planner and give a kernel
 * library nothing but its inputs and outputs, serving loops in which an
 * allocation would stall the device, and hosts with a fixed device-memory
 * budget.  The caller passes inputs (q, k, v, o, dout, m, l, offsets) and
 * outputs (dq, dk, dv) with the layouts above; head_dim 64, 128 or 256
 * (FA_ERR_UNSUPPORTED otherwise), causal 0 or 1.  D and the fp32 dQ
 * accumulator live in one static device array of FA_NOALLOC_SCRATCH_BYTES
 * that every GPU which loads the library keeps until process exit; a
 * problem needing more (total_q * heads * (head_dim + 1) * 4 bytes,
 * rounded up) is rejected with FA_ERR_INVALID_ARG.  Every argument is
 * checked before anything is launched.  Each call looks up the array's
 * device address in the current context (cudaGetSymbolAddress), so it
 * stays valid across context switches and device resets; the first call in
 * a context loads the library's device code, so make it before any stream
 * capture.  Every call shares the array: calls whose work overlaps on the
 * GPU race, so order them on one stream.  Each call re-zeroes what must
 * start at zero. */
int fa_bwd_noalloc(const fa_bf16* q, const fa_bf16* k, const fa_bf16* v, const fa_bf16* o,
                   const fa_bf16* dout, const float* m, const float* l,
                   fa_bf16* dq, fa_bf16* dk, fa_bf16* dv,
                   const int32_t* cu_q_dev, const int32_t* cu_kv_dev,
                   const int32_t* cu_q_host, const int32_t* cu_kv_host,
                   int batch, int total_q, int total_kv, int heads, int head_dim,
                   int causal, float scale, fa_stream_t stream);

/* Diagnostic (the pages have no counterpart): launches one block that
 * waits, through the same bounded mbarrier wait the kernels use, on a
 * barrier nothing arrives on.  After its own short limit (1 s; the
 * kernels' waits give up after 20 s) it records
 * FA_ERR_TIMEOUT in the device status word and returns; nothing faults and
 * the context stays usable.  The next fa_check_device_status on `stream`
 * then returns FA_ERR_TIMEOUT.  Lets a caller test its handling of a timed
 * out kernel. */
int fa_selftest_wait_timeout(fa_stream_t stream);

/* Synchronises `stream`, then reads and clears the device status word
 * that bounded waits set.  Returns FA_OK, FA_ERR_TIMEOUT or FA_ERR_CUDA.
 * The outputs of the kernels launched before it are complete and valid
 * only when it returns FA_OK: after FA_ERR_TIMEOUT some CTAs stopped early
 * and dq_acc, dk, dv (or o, m, l) may be partial. */
int fa_check_device_status(fa_stream_t stream);

/* Message describing the last error returned on the calling thread
 * (empty string after success), in the manner of the argument validators
 * of the PyPTO block_attn_res_impl.py page (_validate_forward_inputs:
 * which argument, what was expected, what was given) and of the JAX
 * wrapper's check_layout.  The pointer stays valid until the next call on
 * the same thread. */
const char* fa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FABWD_H */
