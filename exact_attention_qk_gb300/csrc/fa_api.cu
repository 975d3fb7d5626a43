// fa_api.cu - the C ABI of libfa.so: argument checks, TMA descriptor
// encoding, the split policy, and routing between the prefill, decode and
// combine kernels. All checks mirror `_flash_attn_fwd` on the FlashAttention
// interface page ("mslk/attention/flash_attn/interface.py"): Hq % Hkv == 0,
// head dims <= 256 and multiples of 8, int32 contiguous cu_seqlens/seqused,
// num_splits <= 256 (`_flash_attn_fwd_combine`).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_kernels.h"

namespace fa {
namespace {

__device__ int g_status[1];

std::atomic<unsigned long long> g_timeout_ns{4000000000ull};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int* status_ptr() {
  // one address per device (the symbol lives in every device's image)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static int* ptrs[64] = {nullptr};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// 4-D map (d, rows, heads, batch-or-page) with a box of (box_bytes of d,
// box_rows, 1, 1), swizzled over box_bytes (128: 64 bf16 or 128 one-byte
// elements per box row; 64: 32 bf16). Strides are in elements. Out-of-range
// coordinates read as zero (loads) or are not written (stores).
bool make_map(CUtensorMap* m, const void* base, int64_t d, int64_t rows, int64_t heads, int64_t batch,
              int64_t row_stride, int64_t head_stride, int64_t batch_stride, int box_rows, int esize = 2,
              int box_bytes = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)(row_stride * esize), (cuuint64_t)(head_stride * esize),
                           (cuuint64_t)(batch_stride * esize)};
  cuuint32_t box[4] = {(cuuint32_t)(box_bytes / esize), (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle sw = box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D bf16 map of q (or O) for pack-GQA: (d, head within the KV group, row,
// KV head, batch) with a box of (64, r, box_rows / r, 1, 1), so one box is
// box_rows tile rows ordered (query row, head) with the r heads of a row adjacent.
bool make_map_packed_q(CUtensorMap* m, const void* base, int64_t d, int64_t r, int64_t rows, int64_t hkv,
                       int64_t batch, int64_t row_stride, int64_t head_stride, int64_t batch_stride,
                       int box_rows = 128, int box_cols = 64) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[5] = {(cuuint64_t)d, (cuuint64_t)r, (cuuint64_t)rows, (cuuint64_t)hkv, (cuuint64_t)batch};
  cuuint64_t strides[4] = {(cuuint64_t)(head_stride * 2), (cuuint64_t)(row_stride * 2),
                           (cuuint64_t)(head_stride * r * 2), (cuuint64_t)(batch_stride * 2)};
  cuuint32_t box[5] = {(cuuint32_t)box_cols, (cuuint32_t)r, (cuuint32_t)(box_rows / r), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUtensorMapSwizzle sw = box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult res = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(int64_t s) { return s >= 0 && (s % 8) == 0; }
bool stride_ok_bytes(int64_t s, int esize) { return s >= 0 && (s * esize) % 16 == 0; }
bool fp8_kv(const fa_fwd_args* a) { return a->kv_format == FA_KV_E4M3 || a->kv_format == FA_KV_E5M2; }
// fp8 caches run on the decode kernel whatever the query length
bool kv_special(const fa_fwd_args* a) { return fp8_kv(a); }

struct Resolved {
  bool varlen;
  int rows_q;       // batched: seqlen_q; varlen: max_seqlen_q
  int kmax;         // batched: seqlen_k; varlen: max_seqlen_k
  int r;
  float scale;
  int wl, wr;
};

int check_args(const fa_fwd_args* a, Resolved* out) {
  if (!a) return FA_ERR_INVALID_ARG;
  const bool varlen = a->cu_seqlens_q != nullptr || a->cu_seqlens_k != nullptr;
  if (varlen && (a->cu_seqlens_q == nullptr || a->cu_seqlens_k == nullptr)) return FA_ERR_UNSUPPORTED;
  if (a->batch < 0 || a->num_heads_q <= 0 || a->num_heads_kv <= 0) return FA_ERR_INVALID_ARG;
  if (a->num_heads_q % a->num_heads_kv != 0) return FA_ERR_INVALID_ARG;
  if (a->head_dim_qk <= 0 || a->head_dim_v <= 0 || a->head_dim_qk > 256 || a->head_dim_v > 256)
    return FA_ERR_INVALID_ARG;
  if (a->head_dim_qk % 8 != 0 || a->head_dim_v % 8 != 0) return FA_ERR_INVALID_ARG;
  if (!prefill_supported(a->head_dim_qk, a->head_dim_v)) return FA_ERR_UNSUPPORTED;
  if (a->window_left < -1 || a->window_right < -1) return FA_ERR_INVALID_ARG;
  if (a->num_splits < 0 || a->num_splits > 256) return FA_ERR_INVALID_ARG;
  if (a->kv_format != FA_KV_BF16 && !fp8_kv(a)) return FA_ERR_INVALID_ARG;
  if (fp8_kv(a)) {
    if (varlen) return FA_ERR_UNSUPPORTED;
    if (!((a->head_dim_qk == 128 && a->head_dim_v == 128) || (a->head_dim_qk == 256 && a->head_dim_v == 256)))
      return FA_ERR_UNSUPPORTED;
  }
  if (a->page_table != nullptr) {
    // "page_table is not supported with cu_seqlens_k" (interface.py, _flash_attn_fwd)
    if (varlen) return FA_ERR_INVALID_ARG;
    const int ps = a->page_size;
    if (ps <= 0 || !(ps == 8 || ps == 16 || ps == 32 || ps % 64 == 0)) return FA_ERR_UNSUPPORTED;
    if (a->max_pages_per_seq <= 0 || a->num_pages <= 0) return FA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(a->max_pages_per_seq) * ps > INT32_MAX / 2) return FA_ERR_INVALID_ARG;
  }
  if (varlen) {
    if (a->total_q < 0 || a->total_k < 0 || a->max_seqlen_q < 0 || a->max_seqlen_k < 0) return FA_ERR_INVALID_ARG;
  } else {
    if (a->seqlen_q < 0 || a->seqlen_k < 0) return FA_ERR_INVALID_ARG;
  }
  Resolved r;
  r.varlen = varlen;
  r.rows_q = varlen ? a->max_seqlen_q : a->seqlen_q;
  r.kmax = varlen ? a->max_seqlen_k : a->seqlen_k;
  r.r = a->num_heads_q / a->num_heads_kv;
  if (a->page_table != nullptr) r.kmax = a->max_pages_per_seq * a->page_size;
  r.scale = (a->softmax_scale > 0.f && std::isfinite(a->softmax_scale))
                ? a->softmax_scale
                : 1.0f / std::sqrt(static_cast<float>(a->head_dim_qk));
  r.wl = a->window_left;
  r.wr = a->causal ? 0 : a->window_right;
  if (out) *out = r;
  return FA_OK;
}

int check_tensors(const fa_fwd_args* a, bool need_out) {
  if (!a->q || !a->k || !a->v) return FA_ERR_INVALID_ARG;
  if (need_out && !a->out) return FA_ERR_INVALID_ARG;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || (need_out && !aligned16(a->out)))
    return FA_ERR_ALIGNMENT;
  const bool varlen = a->cu_seqlens_q != nullptr;
  const int es = fp8_kv(a) ? 1 : 2;
  if (!stride_ok(a->q_row_stride) || !stride_ok(a->q_head_stride) || !stride_ok_bytes(a->k_row_stride, es) ||
      !stride_ok_bytes(a->k_head_stride, es) || !stride_ok_bytes(a->v_row_stride, es) ||
      !stride_ok_bytes(a->v_head_stride, es))
    return FA_ERR_ALIGNMENT;
  if (need_out && (!stride_ok(a->o_row_stride) || !stride_ok(a->o_head_stride))) return FA_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(a->k_descale) & 3u) || (reinterpret_cast<uintptr_t>(a->v_descale) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->page_table) & 3u))
    return FA_ERR_ALIGNMENT;
  if (!varlen) {
    if (!stride_ok(a->q_batch_stride) || !stride_ok_bytes(a->k_batch_stride, es) ||
        !stride_ok_bytes(a->v_batch_stride, es))
      return FA_ERR_ALIGNMENT;
    if (need_out && !stride_ok(a->o_batch_stride)) return FA_ERR_ALIGNMENT;
  }
  return FA_OK;
}

bool decode_shaped(const fa_fwd_args* a, const Resolved& r) {
  return static_cast<long long>(r.rows_q) * r.r <= decode_max_rows();
}

// Prefill packs the r q heads of a KV head into the tile rows when r > 1
// divides 128 and no sequence has more than 128 query rows.
bool pack_gqa(const Resolved& r) { return r.r > 1 && 128 % r.r == 0 && r.rows_q <= 128; }

// Prefill grid that would leave more than half of the SMs idle (few sequences
// x heads x query tiles against long keys): its keys are split so that the
// work items (tile, split) fill the GPU, at least 4 key blocks per split and
// no split empty for every tile. The combine merges the fp32 partials.
int prefill_splits(const fa_fwd_args* a, const Resolved& r, int num_sms) {
  if (kv_special(a) || decode_shaped(a, r) || r.kmax <= 0) return 1;
  if (num_sms <= 0) num_sms = device_sms();
  if (num_sms <= 0) return 1;
  const int rpt = prefill_rows_per_tile(a->head_dim_qk, a->head_dim_v);
  const bool pack = pack_gqa(r);
  const long long rows = static_cast<long long>(r.rows_q) * (pack ? r.r : 1);
  const long long tiles = static_cast<long long>(a->batch) * (pack ? a->num_heads_kv : a->num_heads_q) *
                          ((rows + rpt - 1) / rpt);
  if (tiles <= 0 || 2 * tiles > num_sms) return 1;
  const int nkb = (r.kmax + 127) / 128;
  long long ns = num_sms / tiles;
  if (ns > nkb / 4) ns = nkb / 4;
  if (ns > 32) ns = 32;
  if (ns < 2) return 1;
  const int per = static_cast<int>((nkb + ns - 1) / ns);
  return (nkb + per - 1) / per;
}

// keys per split of the prefill kernel: whole 128-key blocks
int prefill_split_len(int kmax, int ns) {
  const int nkb = (kmax + 127) / 128;
  return ((nkb + ns - 1) / ns) * 128;
}

int resolve_splits(const fa_fwd_args* a, const Resolved& r, int num_sms) {
  if (a->num_splits > 0) return a->num_splits;
  if (!decode_shaped(a, r) || r.kmax <= 0) return prefill_splits(a, r, num_sms);
  if (num_sms <= 0) num_sms = device_sms();
  constexpr int kTarget = 2048;
  int ns = (r.kmax + kTarget - 1) / kTarget;
  const long long chunks = (static_cast<long long>(r.rows_q) * r.r + decode_max_rows() - 1) / decode_max_rows();
  const long long units = static_cast<long long>(a->batch) * a->num_heads_kv * (chunks > 0 ? chunks : 1);
  while (ns < 128 && units * ns < 2LL * num_sms && r.kmax / (2 * ns) >= 512) ns *= 2;
  if (ns < 1) ns = 1;
  if (ns > 128) ns = 128;
  return ns;
}

int split_len_for(int kmax, int ns) {
  if (ns <= 1) return INT32_MAX / 2;   // one split holds every key
  const int per = (kmax + ns - 1) / ns;
  const int l = ((per + 63) / 64) * 64;
  return l > 0 ? l : 64;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t prefix_off, prefix_bytes;
  size_t opart_off, opart_bytes;
  size_t lpart_off, lpart_bytes;
  size_t total;
};

WsLayout ws_layout(const fa_fwd_args* a, const Resolved& r, int ns) {
  WsLayout w{};
  size_t off = 0;
  const bool prefill = !decode_shaped(a, r) && !kv_special(a);
  if (prefill && r.varlen) {
    w.prefix_off = off;
    w.prefix_bytes = align256(sizeof(int) * (static_cast<size_t>(a->batch) + 1));
    off += w.prefix_bytes;
  }
  if (ns > 1) {
    const size_t rows = r.varlen ? static_cast<size_t>(a->total_q)
                                 : static_cast<size_t>(a->batch) * static_cast<size_t>(a->seqlen_q);
    w.opart_off = off;
    w.opart_bytes = align256(sizeof(float) * ns * rows * a->num_heads_q * a->head_dim_v);
    off += w.opart_bytes;
    w.lpart_off = off;
    w.lpart_bytes = align256(sizeof(float) * ns * rows * a->num_heads_q);
    off += w.lpart_bytes;
  }
  w.total = off;
  return w;
}

void fill_common(FwdParams* p, const fa_fwd_args* a, const Resolved& r) {
  std::memset(p, 0, sizeof(*p));
  p->q = a->q;
  p->out = a->out;
  p->lse = a->lse;
  p->q_bs = a->q_batch_stride;
  p->q_rs = a->q_row_stride;
  p->q_hs = a->q_head_stride;
  p->o_bs = a->o_batch_stride;
  p->o_rs = a->o_row_stride;
  p->o_hs = a->o_head_stride;
  p->cu_seqlens_q = a->cu_seqlens_q;
  p->cu_seqlens_k = a->cu_seqlens_k;
  p->seqused_k = a->seqused_k;
  p->batch = a->batch;
  p->seqlen_q = r.varlen ? 0 : a->seqlen_q;
  p->seqlen_k = r.varlen ? 0 : a->seqlen_k;
  p->total_q = r.varlen ? a->total_q : 0;
  p->max_seqlen_q = r.rows_q;
  p->hq = a->num_heads_q;
  p->hkv = a->num_heads_kv;
  p->r = r.r;
  p->scale_log2 = static_cast<float>(static_cast<double>(r.scale) * 1.4426950408889634);
  p->wl = r.wl;
  p->wr = r.wr;
  p->num_splits = 1;
  p->split_len = INT32_MAX / 2;
  p->write_partial = 0;
  p->status = status_ptr();
  p->timeout_ns = g_timeout_ns.load();
  p->kv_type = a->kv_format;
  p->k_descale = a->k_descale;
  p->v_descale = a->v_descale;
  p->page_table = a->page_table;
  p->max_pages = a->max_pages_per_seq;
  p->page_size = a->page_size;
  p->num_pages = a->num_pages;
  if (a->page_table != nullptr) p->seqlen_k = r.kmax;   // key capacity of every sequence
}

bool kv_maps(const fa_fwd_args* a, const Resolved& r, int box_rows, CUtensorMap* mk, CUtensorMap* mv) {
  const int es = fp8_kv(a) ? 1 : 2;
  if (a->page_table != nullptr) {
    // pools: (d, page_size, heads, pages); a load moves a piece of one page:
    // box_rows when the page size is a multiple of it, else 64, else a page
    const int ps = a->page_size;
    const int rows = (ps % box_rows == 0) ? box_rows : (ps % 64 == 0 ? 64 : ps);
    return make_map(mk, a->k, a->head_dim_qk, a->page_size, a->num_heads_kv, a->num_pages, a->k_row_stride,
                    a->k_head_stride, a->k_batch_stride, rows, es) &&
           make_map(mv, a->v, a->head_dim_v, a->page_size, a->num_heads_kv, a->num_pages, a->v_row_stride,
                    a->v_head_stride, a->v_batch_stride, rows, es);
  }
  const int64_t rows = r.varlen ? a->total_k : a->seqlen_k;
  const int64_t nb = r.varlen ? 1 : a->batch;
  const int64_t kbs = r.varlen ? a->k_row_stride * (rows > 0 ? rows : 1) : a->k_batch_stride;
  const int64_t vbs = r.varlen ? a->v_row_stride * (rows > 0 ? rows : 1) : a->v_batch_stride;
  return make_map(mk, a->k, a->head_dim_qk, rows, a->num_heads_kv, nb, a->k_row_stride, a->k_head_stride,
                  kbs > 0 ? kbs : 16, box_rows, es) &&
         make_map(mv, a->v, a->head_dim_v, rows, a->num_heads_kv, nb, a->v_row_stride, a->v_head_stride,
                  vbs > 0 ? vbs : 16, box_rows, es);
}

int run_decode(const fa_fwd_args* a, const Resolved& r, int ns, float* opart, float* lpart, cudaStream_t st) {
  FwdParams p;
  fill_common(&p, a, r);
  p.num_splits = ns;
  p.split_len = split_len_for(r.kmax, ns);
  p.write_partial = opart != nullptr ? 1 : 0;
  p.out_partial = opart;
  p.lse_partial = lpart;
  if (!p.status) return FA_ERR_CUDA;
  CUtensorMap mk, mv;
  // decode tiles: 64 keys of bf16, 128 keys of one-byte elements
  if (!kv_maps(a, r, fp8_kv(a) ? 128 : 64, &mk, &mv)) return FA_ERR_CUDA;
  cudaError_t e = launch_decode(p, a->head_dim_qk, a->head_dim_v, mk, mv, st);
  if (e == cudaErrorInvalidConfiguration) return FA_ERR_UNSUPPORTED;   // grid beyond 65535 rows of CTAs
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int run_prefill(const fa_fwd_args* a, const Resolved& r, void* ws, const WsLayout& w, cudaStream_t st,
                int ns = 1, float* opart = nullptr, float* lpart = nullptr) {
  FwdParams p;
  fill_common(&p, a, r);
  if (!p.status) return FA_ERR_CUDA;
  if (ns > 1) {   // key splits into fp32 partials (the combine follows)
    p.num_splits = ns;
    p.split_len = prefill_split_len(r.kmax, ns);
    p.write_partial = 1;
    p.out_partial = opart;
    p.lse_partial = lpart;
  }
  const int rpt = prefill_rows_per_tile(a->head_dim_qk, a->head_dim_v);
  // Pack-GQA for short query sequences: with at most 128 query rows a head's
  // tile would be mostly empty and each K/V block would be read once per head
  p.pack = pack_gqa(r) ? 1 : 0;
  const int mult = p.pack ? r.r : 1;
  if (r.varlen) {
    p.tile_prefix = reinterpret_cast<int*>(static_cast<char*>(ws) + w.prefix_off);
    cudaError_t e = launch_varlen_prepare(p, rpt, st);
    if (e != cudaSuccess) return FA_ERR_LAUNCH;
  } else {
    p.m_blocks = (a->seqlen_q * mult + rpt - 1) / rpt;
    p.num_tiles = p.m_blocks * (p.pack ? a->num_heads_kv : a->num_heads_q) * a->batch;
  }
  CUtensorMap mq, mk, mv;
  const int64_t qrows = r.varlen ? a->total_q : a->seqlen_q;
  const int64_t qb = r.varlen ? 1 : a->batch;
  const int64_t qbs = r.varlen ? a->q_row_stride * (qrows > 0 ? qrows : 1) : a->q_batch_stride;
  // O has q's layout with head_dim_v; the kernel stores boxes of 32 rows x 32
  // columns (64-byte swizzle); packed groups of more than 32 heads are stored
  // row by row
  CUtensorMap mo;
  std::memset(&mo, 0, sizeof(mo));
  const int64_t obs = r.varlen ? a->o_row_stride * (qrows > 0 ? qrows : 1) : a->o_batch_stride;
  if (p.pack) {
    if (!make_map_packed_q(&mq, a->q, a->head_dim_qk, r.r, qrows, a->num_heads_kv, qb, a->q_row_stride,
                           a->q_head_stride, qbs > 0 ? qbs : 8) ||
        (r.r <= 32 && !make_map_packed_q(&mo, a->out, a->head_dim_v, r.r, qrows, a->num_heads_kv, qb,
                                         a->o_row_stride, a->o_head_stride, obs > 0 ? obs : 8, 32, 32)))
      return FA_ERR_CUDA;
  } else if (!make_map(&mq, a->q, a->head_dim_qk, qrows, a->num_heads_q, qb, a->q_row_stride, a->q_head_stride,
                       qbs > 0 ? qbs : 8, 128) ||
             !make_map(&mo, a->out, a->head_dim_v, qrows, a->num_heads_q, qb, a->o_row_stride, a->o_head_stride,
                       obs > 0 ? obs : 8, 32, 2, 64)) {
    return FA_ERR_CUDA;
  }
  if (!kv_maps(a, r, 128, &mk, &mv)) return FA_ERR_CUDA;
  const int sms = device_sms();
  if (sms <= 0) return FA_ERR_CUDA;
  cudaError_t e = launch_prefill(p, a->head_dim_qk, a->head_dim_v, mq, mk, mv, mo, sms, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Scratch for fa_fwd_decode_noalloc: split partials of callers that cannot
// allocate. One copy per device that loads the library; shared by every call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in for it).
void* noalloc_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static void* ptrs[64] = {nullptr};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

bool no_work(const fa_fwd_args* a, const Resolved& r) {
  if (a->batch == 0) return true;
  if (r.varlen) return a->total_q == 0;
  return a->seqlen_q == 0;
}

struct BwdWs {
  int sq_pad;         // batched: 128-row multiple of seqlen_q
  int64_t ws_rows;    // varlen: rows per q head (each sequence's padded region at bwd_ws_row0)
  size_t lse2_off, dsum_off, total;
};

BwdWs bwd_ws(const fa_fwd_args* a) {
  BwdWs w{};
  const bool varlen = a->cu_seqlens_q != nullptr;
  w.sq_pad = varlen ? 0 : ((a->seqlen_q + 127) / 128) * 128;
  // (a multiple of 32, so that every head's region starts 16-byte aligned)
  w.ws_rows = varlen ? ((static_cast<int64_t>(a->total_q) + 132 * static_cast<int64_t>(a->batch) + 4 + 31) / 32) * 32
                     : 0;
  const size_t n = varlen ? static_cast<size_t>(a->num_heads_q) * static_cast<size_t>(w.ws_rows)
                          : static_cast<size_t>(a->batch) * a->num_heads_q * w.sq_pad;
  w.lse2_off = 0;
  w.dsum_off = align256(n * sizeof(float));
  w.total = w.dsum_off + align256(n * sizeof(float));
  return w;
}

int check_bwd_args(const fa_fwd_args* a, Resolved* r) {
  const int rc = check_args(a, r);
  if (rc != FA_OK) return rc;
  if (a->page_table != nullptr || a->kv_format != FA_KV_BF16) return FA_ERR_UNSUPPORTED;
  if (!bwd_supported(a->head_dim_qk, a->head_dim_v)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_abi_version(void) { return 202; }

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case FA_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

void fa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns > 0 ? ns : 1); }

int fa_num_splits(const fa_fwd_args* a, int num_sms) {
  Resolved r;
  if (check_args(a, &r) != FA_OK) return 1;
  fa_fwd_args b = *a;
  b.num_splits = 0;
  return resolve_splits(&b, r, num_sms);
}

int fa_split_len(const fa_fwd_args* a, int num_splits) {
  Resolved r;
  if (check_args(a, &r) != FA_OK) return 0;
  return split_len_for(r.kmax, num_splits);
}

size_t fa_workspace_size(const fa_fwd_args* a) {
  Resolved r;
  if (check_args(a, &r) != FA_OK) return 0;
  const int ns = resolve_splits(a, r, 0);
  return ws_layout(a, r, ns).total;
}

int fa_fwd(const fa_fwd_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  Resolved r;
  int rc = check_args(a, &r);
  if (rc != FA_OK) return rc;
  if (no_work(a, r)) return FA_OK;
  rc = check_tensors(a, true);
  if (rc != FA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ns = resolve_splits(a, r, 0);
  const WsLayout w = ws_layout(a, r, ns);
  if (w.total > 0 && (workspace == nullptr || workspace_bytes < w.total)) return FA_ERR_WORKSPACE;
  if (w.total > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
  if (ns > 1) {
    float* opart = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.opart_off);
    float* lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.lpart_off);
    // decode shapes and fp8 caches split on the decode kernel, prefill shapes
    // on the prefill kernel (whole 128-key blocks per split)
    rc = (decode_shaped(a, r) || kv_special(a)) ? run_decode(a, r, ns, opart, lpart, st)
                                                : run_prefill(a, r, workspace, w, st, ns, opart, lpart);
    if (rc != FA_OK) return rc;
    return fa_combine(opart, lpart, ns, a->batch, r.varlen ? 0 : a->seqlen_q, a->num_heads_q, a->head_dim_v,
                      a->cu_seqlens_q, r.varlen ? a->total_q : 0, a->out, a->o_batch_stride, a->o_row_stride,
                      a->o_head_stride, a->lse, stream);
  }
  if (decode_shaped(a, r) || kv_special(a)) return run_decode(a, r, 1, nullptr, nullptr, st);
  return run_prefill(a, r, workspace, w, st);
}

int fa_fwd_splitkv(const fa_fwd_args* a, int num_splits, float* out_partial, float* lse_partial,
                   void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  Resolved r;
  int rc = check_args(a, &r);
  if (rc != FA_OK) return rc;
  if (num_splits < 1 || num_splits > 256) return FA_ERR_INVALID_ARG;
  if (no_work(a, r)) return FA_OK;
  rc = check_tensors(a, false);
  if (rc != FA_OK) return rc;
  if (!out_partial || !lse_partial) return FA_ERR_INVALID_ARG;
  if (!aligned16(out_partial) || (reinterpret_cast<uintptr_t>(lse_partial) & 3u)) return FA_ERR_ALIGNMENT;
  fa_fwd_args b = *a;
  b.out = nullptr;
  b.lse = nullptr;
  return run_decode(&b, r, num_splits, out_partial, lse_partial, static_cast<cudaStream_t>(stream));
}

int fa_combine(const float* out_partial, const float* lse_partial, int num_splits, int batch, int seqlen_q,
               int num_heads, int head_dim_v, const int32_t* cu_seqlens_q, int total_q, void* out,
               int64_t o_batch_stride, int64_t o_row_stride, int64_t o_head_stride, float* lse, void* stream) {
  if (num_splits < 1 || num_splits > 256) return FA_ERR_INVALID_ARG;
  if (batch < 0 || num_heads <= 0 || seqlen_q < 0 || total_q < 0) return FA_ERR_INVALID_ARG;
  if (head_dim_v != 64 && head_dim_v != 128 && head_dim_v != 256) return FA_ERR_UNSUPPORTED;
  const bool varlen = cu_seqlens_q != nullptr;
  const long long rows = varlen ? total_q : static_cast<long long>(batch) * seqlen_q;
  if (rows == 0) return FA_OK;
  if (!out_partial || !lse_partial || !out) return FA_ERR_INVALID_ARG;
  if (!aligned16(out_partial) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse_partial) & 3u))
    return FA_ERR_ALIGNMENT;
  if (!stride_ok(o_row_stride) || !stride_ok(o_head_stride) || (!varlen && !stride_ok(o_batch_stride)))
    return FA_ERR_ALIGNMENT;
  CombineParams p;
  p.out_partial = out_partial;
  p.lse_partial = lse_partial;
  p.out = out;
  p.lse = lse;
  p.o_bs = o_batch_stride;
  p.o_rs = o_row_stride;
  p.o_hs = o_head_stride;
  p.num_splits = num_splits;
  p.batch = batch;
  p.seqlen_q = varlen ? 0 : seqlen_q;
  p.hq = num_heads;
  p.dv = head_dim_v;
  p.varlen = varlen ? 1 : 0;
  p.total_q = varlen ? total_q : 0;
  cudaError_t e = launch_combine(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_decode_noalloc(const fa_fwd_args* a, void* stream) {
  Resolved r;
  int rc = check_args(a, &r);
  if (rc != FA_OK) return rc;
  if (no_work(a, r)) return FA_OK;
  rc = check_tensors(a, true);
  if (rc != FA_OK) return rc;
  // decode shapes and fp8 caches only, on the decode kernel (whose grid is
  // sized for few rows per KV head)
  if (!decode_shaped(a, r) && !kv_special(a)) return FA_ERR_UNSUPPORTED;
  const int ns = resolve_splits(a, r, 0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ns <= 1) return run_decode(a, r, 1, nullptr, nullptr, st);
  const size_t rows = r.varlen ? static_cast<size_t>(a->total_q)
                               : static_cast<size_t>(a->batch) * static_cast<size_t>(a->seqlen_q);
  const size_t obytes = align256(sizeof(float) * ns * rows * a->num_heads_q * a->head_dim_v);
  const size_t lbytes = align256(sizeof(float) * ns * rows * a->num_heads_q);
  if (obytes + lbytes > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  char* base = static_cast<char*>(noalloc_scratch_ptr());
  if (!base) return FA_ERR_CUDA;
  float* opart = reinterpret_cast<float*>(base);
  float* lpart = reinterpret_cast<float*>(base + obytes);
  rc = run_decode(a, r, ns, opart, lpart, st);
  if (rc != FA_OK) return rc;
  return fa_combine(opart, lpart, ns, a->batch, r.varlen ? 0 : a->seqlen_q, a->num_heads_q, a->head_dim_v,
                    a->cu_seqlens_q, r.varlen ? a->total_q : 0, a->out, a->o_batch_stride, a->o_row_stride,
                    a->o_head_stride, a->lse, stream);
}

size_t fa_bwd_workspace_size(const fa_fwd_args* a) {
  Resolved r;
  if (check_bwd_args(a, &r) != FA_OK) return 0;
  return bwd_ws(a).total;
}

static int bwd_impl(const fa_fwd_args* a, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, void* stream, const BwdSide& side) {
  Resolved r;
  int rc = check_bwd_args(a, &r);
  if (rc != FA_OK) return rc;
  // With no query rows only dK = dV = 0 is written, and with no keys only
  // dQ = 0: the tensors of the empty side are never touched and may be NULL
  // (as an empty tensor's storage is).
  const bool has_q = r.varlen ? a->total_q > 0 : a->seqlen_q > 0;
  const bool has_k = r.varlen ? a->total_k > 0 : a->seqlen_k > 0;
  if (a->batch == 0 || (!has_q && !has_k)) return FA_OK;
  fa_fwd_args c = *a;
  if (!has_q) {
    c.q = c.k;
    c.out = const_cast<void*>(c.k);
  }
  if (!has_k) c.k = c.v = c.q;
  rc = check_tensors(&c, true);
  if (rc != FA_OK) return rc;
  if ((has_q && (!a->lse || !dout || !dq)) || (has_k && (!dk || !dv))) return FA_ERR_INVALID_ARG;
  if ((has_q && (!aligned16(dout) || !aligned16(dq) || (reinterpret_cast<uintptr_t>(a->lse) & 3u))) ||
      (has_k && (!aligned16(dk) || !aligned16(dv))))
    return FA_ERR_ALIGNMENT;
  const BwdWs w = bwd_ws(a);
  if (w.total > 0 && (workspace == nullptr || workspace_bytes < w.total)) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.out = a->out;
  p.dout = dout;
  p.lse = a->lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.lse2_off);
  p.dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.dsum_off);
  p.q_bs = a->q_batch_stride;
  p.q_rs = a->q_row_stride;
  p.q_hs = a->q_head_stride;
  p.k_bs = a->k_batch_stride;
  p.k_rs = a->k_row_stride;
  p.k_hs = a->k_head_stride;
  p.v_bs = a->v_batch_stride;
  p.v_rs = a->v_row_stride;
  p.v_hs = a->v_head_stride;
  p.o_bs = a->o_batch_stride;
  p.o_rs = a->o_row_stride;
  p.o_hs = a->o_head_stride;
  p.batch = a->batch;
  p.seqlen_q = r.varlen ? a->max_seqlen_q : a->seqlen_q;
  p.seqlen_k = r.varlen ? a->max_seqlen_k : a->seqlen_k;
  p.sq_pad = w.sq_pad;
  p.cu_seqlens_q = a->cu_seqlens_q;
  p.cu_seqlens_k = a->cu_seqlens_k;
  p.seqused_k = a->seqused_k;
  p.total_q = r.varlen ? a->total_q : 0;
  p.ws_rows = w.ws_rows;
  // packed varlen: neighbouring tiles of one head in consecutive CTAs (the
  // (sequence, head) index in y, whose limit is 65535)
  p.tiles_fast = r.varlen && static_cast<int64_t>(a->batch) * a->num_heads_q <= 65535 ? 1 : 0;
  if (r.varlen) {   // batch strides are ignored in the packed layout
    p.q_bs = p.k_bs = p.v_bs = p.o_bs = 0;
  }
  p.hq = a->num_heads_q;
  p.hkv = a->num_heads_kv;
  p.r = r.r;
  p.scale = r.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(r.scale) * 1.4426950408889634);
  p.wl = r.wl;
  p.wr = r.wr;
  p.status = status_ptr();
  p.timeout_ns = g_timeout_ns.load();
  if (!p.status) return FA_ERR_CUDA;
  // batched: (d, rows, heads, batch); packed varlen: (d, total rows, heads, 1)
  // with the batch stride a stand-in (one batch)
  const int64_t sq = r.varlen ? a->total_q : a->seqlen_q, sk = r.varlen ? a->total_k : a->seqlen_k;
  const int64_t nb = r.varlen ? 1 : a->batch;
  const int64_t qbs = r.varlen ? a->q_row_stride * sq : a->q_batch_stride;
  const int64_t obs = r.varlen ? a->o_row_stride * sq : a->o_batch_stride;
  const int64_t kbs = r.varlen ? a->k_row_stride * sk : a->k_batch_stride;
  const int64_t vbs = r.varlen ? a->v_row_stride * sk : a->v_batch_stride;
  const int d = a->head_dim_qk, d_v = a->head_dim_v;
  // the maps of an empty side are stand-ins (copies of the other side's), never read
  CUtensorMap mq, mk, mv, mdo;
  if (has_q && (!make_map(&mq, a->q, d, sq, a->num_heads_q, nb, a->q_row_stride, a->q_head_stride, qbs, 128) ||
                !make_map(&mdo, dout, d_v, sq, a->num_heads_q, nb, a->o_row_stride, a->o_head_stride, obs, 128)))
    return FA_ERR_CUDA;
  if (has_k && (!make_map(&mk, a->k, d, sk, a->num_heads_kv, nb, a->k_row_stride, a->k_head_stride, kbs, 128) ||
                !make_map(&mv, a->v, d_v, sk, a->num_heads_kv, nb, a->v_row_stride, a->v_head_stride, vbs, 128)))
    return FA_ERR_CUDA;
  if (!has_q) mq = mdo = mk;
  if (!has_k) mk = mv = mq;
  cudaError_t e = launch_bwd(p, d, d_v, mq, mk, mv, mdo, static_cast<cudaStream_t>(stream), side);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd(const fa_fwd_args* a, const void* dout, void* dq, void* dk, void* dv, void* workspace,
           size_t workspace_bytes, void* stream) {
  const BwdSide none{nullptr, nullptr, nullptr};
  return bwd_impl(a, dout, dq, dk, dv, workspace, workspace_bytes, stream, none);
}

int fa_bwd_two_streams(const fa_fwd_args* a, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                       size_t workspace_bytes, void* stream, void* side_stream, void* fork_event,
                       void* join_event) {
  if (side_stream == nullptr || fork_event == nullptr || join_event == nullptr || side_stream == stream)
    return FA_ERR_INVALID_ARG;
  const BwdSide side{static_cast<cudaStream_t>(side_stream), static_cast<cudaEvent_t>(fork_event),
                     static_cast<cudaEvent_t>(join_event)};
  return bwd_impl(a, dout, dq, dk, dv, workspace, workspace_bytes, stream, side);
}

int fa_get_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

}  // extern "C"
