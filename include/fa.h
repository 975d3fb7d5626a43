/*
 * fa.h - C ABI of the GB300 (sm_103a) exact attention library (libfa.so): the
 * forward with its per-row LSE, and its backward.
 *
 * The operation is the exact scaled-dot-product attention forward with a
 * per-row log-sum-exp, as defined by the FlashAttention pages:
 *
 *   "mslk/attention/flash_attn/interface.py", `_flash_attn_fwd`:
 *       O = softmax(scale * Q K^T + mask) V,  LSE = log sum_j exp(scale q.k_j)
 *       over visible keys; default scale 1/sqrt(head_dim_qk); O has q's layout
 *       with head_dim_v; LSE is fp32 (B,Hq,Sq), or (Hq,Tq) for packed varlen;
 *       causal means window_right = 0; GQA head h reads KV head h / (Hq/Hkv).
 *   "mslk/attention/flash_attn/flash_bwd_sm100.py", causal block bound:
 *       the causal diagonal is bottom-right aligned (offset Sk - Sq), and the
 *       window [i + off - window_left, i + off + window_right] is taken about it.
 *   "mslk/attention/flash_attn/interface.py", `_flash_attn_fwd_combine` and
 *   "mslk/attention/fmha/triton_splitk.py", `merge_attentions`:
 *       split-KV partials (fp32 O and LSE per split) merge by LSE weights.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers; the library allocates nothing.
 *     The caller owns every buffer, including workspace, and the stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream; inputs must stay alive and
 *     unmodified until the stream reaches the call.
 *   - bf16 tensors have a contiguous last dimension; the other strides are
 *     given in ELEMENTS. Base pointers must be 16-byte aligned and strides
 *     multiples of 8 elements (16 bytes), else FA_ERR_ALIGNMENT.
 *   - Arguments are checked before any launch: a non-zero status means that
 *     nothing was launched (except FA_ERR_LAUNCH / FA_ERR_CUDA, reported after
 *     a failed launch). No error crosses the ABI as an exception.
 *   - Device-side waits are bounded; a wait that runs out sets a device status
 *     word instead of hanging. fa_get_status() reads and clears it.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* shape / dtype-rule / null-pointer violation          */
  FA_ERR_UNSUPPORTED = 2,     /* legal input outside the compiled kernel set           */
  FA_ERR_ALIGNMENT = 3,       /* base pointer or stride not 16-byte aligned            */
  FA_ERR_WORKSPACE = 4,       /* workspace NULL or smaller than fa_workspace_size()   */
  FA_ERR_LAUNCH = 5,          /* a kernel launch failed (cudaGetLastError)            */
  FA_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device wait ran out (from fa_get_status)   */
  FA_ERR_CUDA = 7,            /* another CUDA runtime error (no device, bad stream)   */
};

/*
 * Arguments of one attention forward.
 *
 * Batched layout (cu_seqlens_q == NULL):
 *   q   (batch, seqlen_q, num_heads_q,  head_dim_qk)
 *   k   (batch, seqlen_k, num_heads_kv, head_dim_qk)   seqlen_k = cache capacity
 *   v   (batch, seqlen_k, num_heads_kv, head_dim_v)
 *   out (batch, seqlen_q, num_heads_q,  head_dim_v)    bf16, written
 *   lse (batch, num_heads_q, seqlen_q)                 fp32 contiguous, written; may be NULL
 * Packed varlen layout (cu_seqlens_q and cu_seqlens_k both non-NULL, int32 [batch+1],
 * prefix sums starting at 0; the *_batch_stride fields are ignored):
 *   q   (total_q, num_heads_q, head_dim_qk)   k, v (total_k, num_heads_kv, ...)
 *   out (total_q, num_heads_q, head_dim_v)    lse (num_heads_q, total_q)
 * seqused_k (int32 [batch], optional): only keys [0, seqused_k[b]) of sequence b
 *   exist; it overrides seqlen_k / the cu_seqlens_k length. Cache rows past
 *   seqused_k[b] may hold anything (NaN included): no arithmetic ever uses them.
 * Masks: causal != 0 forces window_right = 0. window_left / window_right = -1
 *   means unbounded on that side. Key j is visible from query row i of a
 *   sequence with Sq query rows and Sk keys iff
 *     j < Sk and (wl < 0 or j >= i + Sk - Sq - wl) and (wr < 0 or j <= i + Sk - Sq + wr).
 *   A row with no visible key gets O = 0 and LSE = -inf.
 * softmax_scale <= 0 (or NaN) selects 1/sqrt(head_dim_qk).
 * num_splits: 0 = let the library choose (fa_num_splits), 1 = no split,
 *   > 1 = split-KV with that many splits followed by the combine (<= 256).
 *   Decode shapes and fp8 caches split on the decode kernel at the
 *   boundaries of fa_split_len; prefill shapes split on the prefill kernel at
 *   whole 128-key blocks (ceil(key blocks / num_splits) blocks per split).
 * Supported (head_dim_qk, head_dim_v): (64,64), (128,128), (192,128), (256,256).
 * Element type: bf16 for q and out; k and v are bf16 unless kv_format says otherwise.
 *
 * KV-cache forms (every field below zero / NULL: a bf16 cache in the layouts above).
 *   fp8 cache ("fp8 KV-cache decode (e4m3/e5m2)" on the FlashAttention sm_120
 *   pull-request page: a bf16 query against a quantized cache with per-(batch,
 *   kv_head) k_descale / v_descale): kv_format FA_KV_E4M3 or FA_KV_E5M2; k and
 *   v hold one byte per element in that 8-bit float format, and element
 *   (b, j, g, d) of K stands for its code value x k_descale[b * num_heads_kv + g]
 *   (V likewise with v_descale; a NULL descale means 1). K/V strides are still
 *   in elements (= bytes) and must be multiples of 16. Head dims (128,128) and
 *   (256,256); batched or paged layout, not varlen.
 *   Paged cache ("mslk/attention/flash_attn/interface.py", `_flash_attn_fwd`:
 *   page_table int32 (batch, max_num_pages_per_seq), k/v (num_pages, page_size,
 *   num_heads_kv, head_dim)): page_table != NULL; k and v are pools of
 *   num_pages pages, k_batch_stride / v_batch_stride are the page strides, and
 *   key j of sequence b is row j % page_size of page
 *   page_table[b * max_pages_per_seq + j / page_size]. The key capacity is
 *   max_pages_per_seq * page_size (seqlen_k is ignored); seqused_k gives the
 *   lengths. page_size: 8, 16, 32 or a multiple of 64. Not with cu_seqlens
 *   (FA_ERR_INVALID_ARG). A page index outside [0, num_pages) reads zeros.
 *   An fp8 cache runs on the split-KV decode kernel for any number of query
 *   rows (correct for prefill shapes too, but built for few rows per KV head);
 *   a paged bf16 cache runs on the same kernels as the plain layout (decode
 *   for few rows per KV head, the tensor-memory prefill kernel otherwise).
 */
enum {
  FA_KV_BF16 = 0,   /* 2-byte bfloat16 elements                                 */
  FA_KV_E4M3 = 1,   /* 1-byte E4M3 (bias 7, no infinities), times its descale   */
  FA_KV_E5M2 = 2,   /* 1-byte E5M2 (bias 15, IEEE-style), times its descale     */
};

typedef struct fa_fwd_args {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int64_t q_batch_stride, q_row_stride, q_head_stride;
  int64_t k_batch_stride, k_row_stride, k_head_stride;
  int64_t v_batch_stride, v_row_stride, v_head_stride;
  int64_t o_batch_stride, o_row_stride, o_head_stride;
  int32_t batch;
  int32_t seqlen_q;        /* batched: query rows per sequence                 */
  int32_t seqlen_k;        /* batched: key rows (capacity) per sequence        */
  int32_t num_heads_q;
  int32_t num_heads_kv;
  int32_t head_dim_qk;
  int32_t head_dim_v;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* seqused_k;
  int32_t total_q;         /* varlen: rows of q / out                           */
  int32_t total_k;         /* varlen: rows of k / v                             */
  int32_t max_seqlen_q;    /* varlen: upper bound on any query length           */
  int32_t max_seqlen_k;    /* varlen: upper bound on any key length             */
  float softmax_scale;
  int32_t causal;
  int32_t window_left;
  int32_t window_right;
  int32_t num_splits;
  /* KV-cache forms (see above); zero / NULL for a plain bf16 cache */
  int32_t kv_format;           /* FA_KV_BF16, FA_KV_E4M3 or FA_KV_E5M2            */
  const float* k_descale;      /* fp8: fp32 [batch * num_heads_kv] or NULL (= 1)   */
  const float* v_descale;
  const int32_t* page_table;   /* int32 [batch * max_pages_per_seq] or NULL        */
  int32_t max_pages_per_seq;
  int32_t page_size;           /* keys per page                                    */
  int32_t num_pages;           /* pages in the k and v pools                       */
} fa_fwd_args;

/*
 * fa_fwd - O and LSE for args (the whole forward: split-KV plus combine when the
 * resolved split count is > 1, otherwise one kernel).
 * workspace: device buffer of at least fa_workspace_size(args) bytes, 256-byte
 * aligned; may be NULL when that size is 0. Its contents are scratch.
 * Returns FA_OK or an error code (see the enum); asynchronous on `stream`.
 */
int fa_fwd(const fa_fwd_args* args, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_splitkv - the split-KV pass alone ("interface.py", `_flash_attn_fwd`
 * with num_splits > 1: fp32 out_partial and lse_partial).
 * Split s covers key positions [s*L, (s+1)*L) of every sequence, with
 * L = fa_split_len(args, num_splits). An empty split writes O = 0, LSE = -inf.
 *   out_partial fp32 (num_splits, batch, seqlen_q, num_heads_q, head_dim_v)
 *               or   (num_splits, total_q, num_heads_q, head_dim_v), contiguous
 *   lse_partial fp32 (num_splits, batch, num_heads_q, seqlen_q)
 *               or   (num_splits, num_heads_q, total_q), contiguous
 * args->out / args->lse / args->num_splits are ignored. 1 <= num_splits <= 256.
 * workspace: as for fa_fwd (this pass needs none today; pass NULL, 0).
 */
int fa_fwd_splitkv(const fa_fwd_args* args, int num_splits, float* out_partial,
                   float* lse_partial, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_combine - merge split partials by LSE weights ("interface.py",
 * `_flash_attn_fwd_combine`; "triton_splitk.py", `merge_attentions`):
 *   M = max_s LSE_s;  LSE = M + log sum_s exp(LSE_s - M);  O = sum_s exp(LSE_s - LSE) O_s
 * Splits with LSE_s = -inf are skipped (their O_s is never read); if every split
 * is empty the row gets O = 0 and LSE = -inf.
 * Layouts: partials as in fa_fwd_splitkv (cu_seqlens_q != NULL selects the
 * packed layout with total_q rows; only its presence matters). out is bf16
 * with the given strides (elements; batch stride ignored when packed); lse is
 * fp32 (batch, num_heads, seqlen_q) or (num_heads, total_q), may be NULL.
 * head_dim_v in {64, 128, 256}; 1 <= num_splits <= 256.
 */
int fa_combine(const float* out_partial, const float* lse_partial, int num_splits,
               int batch, int seqlen_q, int num_heads, int head_dim_v,
               const int32_t* cu_seqlens_q, int total_q,
               void* out, int64_t o_batch_stride, int64_t o_row_stride, int64_t o_head_stride,
               float* lse, void* stream);

/*
 * fa_fwd_decode_noalloc - split-KV decode plus combine, like fa_fwd on a
 * decode-shaped problem, but with no workspace argument: the fp32 split
 * partials live in a fixed array inside the library (FA_NOALLOC_SCRATCH_BYTES
 * per GPU). The pages have no counterpart of this entry point. It exists for
 * callers that cannot allocate device memory at the point of the call:
 * engines whose device memory belongs to another allocator that they cannot
 * reach from the call site, and latency-critical paths that must not take the
 * driver's allocation locks or its implicit synchronisation.
 * The array is reserved on each device when the library's module is loaded
 * there, which under CUDA's default lazy module loading is the first call of
 * any entry point of this library on that device (with
 * CUDA_MODULE_LOADING=EAGER, when the library is loaded); it is held until the
 * process exits. The first call of this entry point on each device also looks
 * up the array's device address there (the device must be current).
 * The caller still passes q/k/v/out/lse in args. Only decode-shaped problems
 * (seqlen_q * Hq/Hkv <= 16) and fp8 caches are served, on the decode kernel;
 * other shapes return FA_ERR_UNSUPPORTED. args->num_splits is resolved as in
 * fa_fwd. Problems whose partials (num_splits * rows * Hq * (head_dim_v + 1)
 * floats) exceed the array return FA_ERR_WORKSPACE before anything is launched.
 * No call allocates: it calls no cudaMalloc/cudaFree or allocating library routine.
 * Every call on a device shares the one array: calls whose work overlaps on the
 * GPU (different streams without ordering between them) race and give wrong
 * results. Nothing in the array needs clearing: each call writes every partial
 * it later reads.
 */
#define FA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int fa_fwd_decode_noalloc(const fa_fwd_args* args, void* stream);

/*
 * fa_bwd - gradients dQ, dK, dV of the forward described by args, given dO
 * ("mslk/attention/flash_attn/flash_bwd_sm100.py": the preprocess forms
 * D = rowsum(dO * O); the main loop recomputes P from the stored LSE and forms
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q;
 * with GQA, dK and dV of KV head g sum over the q heads that read it).
 * args: the forward's arguments, batched or packed varlen layout (as for
 *   fa_fwd). args->out must hold the forward's O and args->lse its LSE (both
 *   read, not written).
 * dout: dO, bf16, out's shape and strides (o_*_stride).
 * dq / dk / dv: written, bf16, with q's / k's / v's shapes and strides. Keys
 *   that no query sees get dK = dV = 0; rows that see no key get dQ = 0.
 * Supported: (head_dim_qk, head_dim_v) (64,64), (128,128), (192,128) (the
 *   shape the interface page names for Blackwell) or (256,256); at the last
 *   two the dK/dV kernel runs a dV pass and a dK pass in one grid, since both
 *   accumulators do not fit tensor memory beside S and dP; causal, sliding
 *   window, GQA/MQA and varlen (cu_seqlens_q / cu_seqlens_k) as in the
 *   forward; seqused_k as in the forward ("interface.py", `_flash_attn_bwd`
 *   takes seqused_q / seqused_k): only keys [0, seqused_k[b]) exist, cache
 *   rows past them may hold anything (NaN included), and their dK and dV are
 *   written as 0 (up to seqlen_k, or the sequence's cu_seqlens_k length).
 *   A page table or an fp8 cache gives FA_ERR_UNSUPPORTED.
 * workspace: at least fa_bwd_workspace_size(args) bytes, 256-byte aligned
 *   (fp32 LSE * log2(e) and D for every padded query row). The call is
 *   deterministic: no atomics, the same inputs give the same bits.
 * Every kernel runs on `stream`, one after the other (preprocess, dK/dV, dQ).
 */
int fa_bwd(const fa_fwd_args* args, const void* dout, void* dq, void* dk, void* dv, void* workspace,
           size_t workspace_bytes, void* stream);

/*
 * fa_bwd_two_streams - fa_bwd with the dK/dV kernel on a second stream of the
 * caller's, concurrent with the dQ kernel on `stream` (the two only share
 * read-only inputs). side_stream is a cudaStream_t and fork_event /
 * join_event are cudaEvent_t (created by the caller, e.g. with
 * cudaEventDisableTiming), all passed as void*. The call records fork_event
 * on `stream` after the preprocess, makes side_stream wait for it, launches
 * dK/dV there, records join_event on side_stream and makes `stream` wait for
 * it: to the caller the whole backward is ordered on `stream`. Give
 * side_stream a higher priority than `stream`, so that the long dK/dV CTAs
 * are placed first and the short dQ CTAs fill the SMs they leave idle.
 * The library creates no stream or event. Both events are re-recorded by
 * every call: calls that share them must be issued from one host thread.
 * Returns FA_ERR_INVALID_ARG when side_stream or an event is NULL or
 * side_stream == stream; otherwise as fa_bwd.
 */
int fa_bwd_two_streams(const fa_fwd_args* args, const void* dout, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, void* stream, void* side_stream,
                       void* fork_event, void* join_event);

/* Bytes of workspace fa_bwd needs for args (0 when fa_bwd would reject args). */
size_t fa_bwd_workspace_size(const fa_fwd_args* args);

/* Bytes of workspace fa_fwd needs for args (with args->num_splits resolved as fa_fwd does). */
size_t fa_workspace_size(const fa_fwd_args* args);

/*
 * Split count fa_fwd uses when args->num_splits == 0.
 * The pages' policies, and where this one departs from them:
 *   "mslk/attention/flash_attn/interface.py", `num_splits_heuristic`: no split
 *     when a sequence has at most 4 key blocks, else
 *     min(num_SMs / total_mblocks, max_splits, key blocks), that is, split
 *     only a grid that leaves SMs idle. The prefill rule below is this one
 *     (at least 4 key blocks per split, at most 32 splits, counted in the
 *     256-row tiles of this library's prefill kernel) with one change: a grid
 *     that fills more than half of the SMs is not split, because the fp32
 *     partials and the combine cost more than the idle SMs.
 *   "mslk/attention/fmha/triton_splitk.py", `get_split_k` / `split_size`:
 *     for decode, the splits follow the key length (about Mk / 128-key
 *     chunks, halved until they fit) and each split covers
 *     ceil(Mk / split_k) keys. The decode rule below also splits by key
 *     length, with a longer chunk: about 2048 keys per split, doubled while
 *     (sequences x KV heads x row chunks x splits) < 2 x num_sms, at most 128.
 *     `num_splits_heuristic` would return 1 on a decode batch whose KV heads
 *     alone fill the SMs; with seqused_k spread 16x between sequences that
 *     leaves a long tail of the longest sequences, so the fixed key length
 *     wins there.
 * Decode-shaped problems are those with seqlen_q * Hq/Hkv <= 16. Prefill
 * shapes with a bf16 cache split into whole 128-key blocks and run on the
 * prefill kernel, merged by the combine. fp8 caches follow the decode rule.
 * num_sms <= 0 queries the current device.
 */
int fa_num_splits(const fa_fwd_args* args, int num_sms);

/*
 * Keys per split of the decode kernel and of fa_fwd_splitkv:
 * L = 64 * ceil(ceil(Kmax / num_splits) / 64), Kmax = seqlen_k (batched),
 * max_seqlen_k (varlen) or max_pages_per_seq * page_size (paged); split s
 * covers key positions [s*L, (s+1)*L). This is the split-K page's
 * `split_size` = ceil(Mk / split_k) ("mslk/attention/fmha/triton_splitk.py"),
 * rounded up to the decode kernel's 64-key tile so that no tile straddles two
 * splits. Returns 0 when args are invalid.
 */
int fa_split_len(const fa_fwd_args* args, int num_splits);

/*
 * Synchronizes `stream`, then reads and clears the device status word of the
 * current device. Returns FA_OK, or FA_ERR_DEVICE_TIMEOUT if some kernel's
 * bounded wait ran out since the last call (that kernel's outputs are invalid).
 */
int fa_get_status(void* stream);

/* Limit for every device-side wait, in nanoseconds (default 4e9 = 4 s). */
void fa_set_wait_timeout_ns(uint64_t ns);

/* Static text for a status code. */
const char* fa_status_string(int status);

/* ABI version (major*100 + minor): 200 since fa_fwd_args gained the KV-cache
 * fields, 201 since fa_bwd, 202 since fa_bwd_two_streams (fa_bwd itself runs
 * on the caller's stream alone). */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
