// fa_kernels.h - parameter blocks and launchers shared by the host API
// (fa_api.cu) and the kernel translation units. Internal to libfa.so.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Everything a forward kernel needs besides the tensor maps. Strides are in
// elements. `wr` is already 0 when the call was causal.
struct FwdParams {
  const void* q;
  void* out;
  float* lse;                    // final LSE or NULL
  float* out_partial;            // split mode: fp32 partial O
  float* lse_partial;            // split mode: fp32 partial LSE
  int64_t q_bs, q_rs, q_hs;
  int64_t o_bs, o_rs, o_hs;
  const int* cu_seqlens_q;
  const int* cu_seqlens_k;
  const int* seqused_k;
  int* tile_prefix;              // varlen prefill: [batch+1] tile prefix sums (workspace)
  int batch, seqlen_q, seqlen_k; // batched sizes (seqlen_k = capacity)
  int total_q;                   // varlen rows (LSE row stride)
  int max_seqlen_q;
  int hq, hkv, r;                // r = hq / hkv
  float scale_log2;              // softmax_scale * log2(e)
  int wl, wr;                    // -1 = unbounded
  int num_splits;                // decode grid extent over key splits (>= 1)
  int split_len;                 // keys per split (covers every key when num_splits == 1)
  int write_partial;             // decode: 1 = fp32 partials at [split], 0 = final bf16 O / LSE
  int pack;                      // prefill: 1 = tile rows are (query row, head) pairs of one KV head
  int m_blocks;                  // batched prefill: ceil(tile rows of a sequence / rows per tile)
  int num_tiles;                 // batched prefill: total work tiles
  int* status;                   // device status word
  unsigned long long timeout_ns;
  // KV-cache forms (decode kernel only)
  int kv_type;                   // 0 bf16, 1 e4m3, 2 e5m2
  const float* k_descale;        // fp8: [batch * hkv] or NULL
  const float* v_descale;
  const int* page_table;         // [batch * max_pages] or NULL
  int max_pages, page_size, num_pages;
};

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_prefill(const FwdParams& p, int dk, int dv, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mo, int num_sms, cudaStream_t stream);
cudaError_t launch_varlen_prepare(const FwdParams& p, int rows_per_tile, cudaStream_t stream);
int prefill_rows_per_tile(int dk, int dv);
bool prefill_supported(int dk, int dv);

cudaError_t launch_decode(const FwdParams& p, int dk, int dv, const CUtensorMap& mk, const CUtensorMap& mv,
                          cudaStream_t stream);
bool decode_supported(int dk, int dv);
int decode_max_rows();

// Backward (dQ, dK, dV): batched or packed varlen layout, head dims 64 or
// 128 (dk == dv). dq / dk / dv take q's / k's / v's strides, dout and out
// take the o strides. lse2 and dsum are workspace arrays: batched
// [batch][hq][sq_pad] (sq_pad = 128-row multiple of seqlen_q); varlen
// [hq][ws_rows], sequence b's rows starting at bwd_ws_row0(b) (a multiple of
// 4, and 128-row padded regions that do not overlap).
struct BwdParams {
  const void* out;
  const void* dout;
  const float* lse;              // forward LSE [batch][hq][seqlen_q], natural log
  void* dq;
  void* dk;
  void* dv;
  float* lse2;                   // LSE * log2(e); +inf where P must be 0
  float* dsum;                   // rowsum(dO * O)
  int64_t q_bs, q_rs, q_hs;
  int64_t k_bs, k_rs, k_hs;
  int64_t v_bs, v_rs, v_hs;
  int64_t o_bs, o_rs, o_hs;
  int batch, seqlen_q, seqlen_k, sq_pad;  // batched sizes (varlen: max_seqlen_q / _k, and sq_pad unused)
  int hq, hkv, r;
  float scale, scale_log2;
  int wl, wr;                    // -1 = unbounded; wr is 0 when causal
  const int* cu_seqlens_q;       // varlen: int32 [batch+1], else NULL
  const int* cu_seqlens_k;
  const int* seqused_k;          // int32 [batch] or NULL: keys [0, seqused_k[b]) exist
  int total_q;                   // varlen: rows of q (LSE row stride)
  int64_t ws_rows;               // varlen: workspace rows per head
  int tiles_fast;                // grids with the tile / key-block index in x (packed varlen)
  int* status;
  unsigned long long timeout_ns;
};
// first workspace row of sequence b (varlen): 4-aligned, and far enough past
// sequence b-1's padded region (which ends before cu_seqlens_q[b] + 132 b)
__host__ __device__ inline int64_t bwd_ws_row0(const int* cu_seqlens_q, int b) {
  return ((int64_t(cu_seqlens_q[b]) + 132 * int64_t(b) + 3) / 4) * 4;
}
// Optional second stream of the caller for the dK/dV kernel, with the two
// events that fork it from and join it back into the main stream (all three
// owned by the caller). stream == nullptr: every kernel on the main stream.
struct BwdSide {
  cudaStream_t stream;
  cudaEvent_t fork, join;
};
cudaError_t launch_bwd(const BwdParams& p, int dk, int dv, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t stream, const BwdSide& side);
bool bwd_supported(int dk, int dv);

struct CombineParams {
  const float* out_partial;
  const float* lse_partial;
  void* out;
  float* lse;
  int64_t o_bs, o_rs, o_hs;
  int num_splits;
  int batch, seqlen_q, hq, dv;
  int varlen, total_q;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

}  // namespace fa
