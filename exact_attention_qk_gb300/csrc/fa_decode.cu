// fa_decode.cu - split-KV decode forward and the LSE-weighted combine.
//
// Decode ("mslk/attention/fmha/triton_splitk.py", split-K forward; and
// "mslk/attention/flash_attn/interface.py", `_flash_attn_fwd` with
// num_splits > 1): few query rows against a long KV cache. Reading K and V
// once from HBM is the whole cost, so the kernel is built for bandwidth:
//   * one CTA per (split, KV head x row chunk, sequence); the Hq/Hkv query heads
//     that share a KV head are packed as rows of one CTA (the triton page's
//     head-swapping trick), so K/V bytes are read once per KV head;
//   * a producer warp streams 64-key K/V tiles with TMA (128-byte swizzle) into
//     a 2-deep mbarrier ring (three CTAs per SM keep enough bytes in flight);
//     cache rows at or past seqused_k are never used in arithmetic;
//   * four compute warps take 16 keys each per tile: QK^T with 16-byte swizzled
//     shared loads (conflict-free), two keys per lane so each q load feeds both,
//     packed fp32 FMA (FFMA2), online softmax in base 2 with the scale folded
//     into q, and P.V with per-lane output columns;
//   * the four warps' (m, l, O) states merge in shared memory at the end and the
//     CTA writes either the final bf16 O / fp32 LSE or the fp32 split partials.
// KV-cache forms (the fp8 KV-cache decode and paged-KV passages of the
// FlashAttention sm_120 pull-request page and of `_flash_attn_fwd`):
//   * fp8 (E4M3 / E5M2) caches move one byte per element: a 128-byte box row
//     holds 128 dims; the compute warps widen codes to fp32 in registers, the
//     K descale is folded into q and the V descale into the written O;
//   * a paged cache is read page by page: each 64-key tile looks up its page
//     (or pages, for pages under 64 keys) in the page table and loads from
//     that page's rows; an index outside the pool reads zeros.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_kernels.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kDecWarps = 4;            // compute warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kTileKeys = 64;
constexpr int kBoxBytes = kTileKeys * 128;   // one 64-element x 64-key box

// Widen four fp8 codes (one 32-bit word, lowest byte first) to fp32 pairs.
template <int KVT>
__device__ __forceinline__ void fp8x4_to_f32(uint32_t w, float2& lo, float2& hi) {
  uint32_t h0, h1;
  if constexpr (KVT == 1) {   // E4M3 -> f16 pairs (exact), then f32
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
  } else {                    // E5M2 is the upper byte of an f16
    h0 = __byte_perm(w, 0u, 0x1404);
    h1 = __byte_perm(w, 0u, 0x3424);
  }
  lo = __half22float2(*reinterpret_cast<const __half2*>(&h0));
  hi = __half22float2(*reinterpret_cast<const __half2*>(&h1));
}

template <int DK, int DV, int NR, int KVT>
struct DecodeCfg {
  static constexpr int ES = KVT ? 1 : 2;          // bytes per K/V element
  static constexpr int KCH = DK * ES / 128;       // 128-byte boxes per K row
  static constexpr int VCH = DV * ES / 128;
  static constexpr int STAGE_BYTES = (KCH + VCH) * kBoxBytes;
  // Two stages keep the CTA under 70 KB of shared memory, so three CTAs (12
  // compute warps) share an SM: the QK / softmax / PV chains are latency-bound
  // and need the extra warps more than each CTA needs a deeper ring.
  static constexpr int NSTAGE = 2;
  static constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;
  static constexpr int Q_BYTES = NR * DK * 4;
  static constexpr int P_BYTES = kDecWarps * 16 * NR * 4;
  static constexpr int MERGE_BYTES = kDecWarps * NR * (DV + 2) * 4;
  static constexpr int OFF_Q = RING_BYTES;
  static constexpr int OFF_P = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8 + 16 + 1024;   // + alignment slack
  static constexpr int E = DV / 32;                                   // output columns per lane
  static_assert(MERGE_BYTES <= RING_BYTES, "merge area reuses the ring");
  static_assert(NR * E <= 64, "accumulator budget");
};

template <int DK, int DV, int NR, int KVT>
__global__ void __launch_bounds__(kDecThreads, (NR <= 4) ? 3 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                  const FwdParams p) {
  using C = DecodeCfg<DK, DV, NR, KVT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* q_s = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* p_s = reinterpret_cast<float*>(smem + C::OFF_P);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::NSTAGE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int g = blockIdx.y % p.hkv;
  const int chunk = blockIdx.y / p.hkv;
  const int b = blockIdx.z;

  // ---- sequence geometry --------------------------------------------------------------
  const bool varlen = p.cu_seqlens_q != nullptr;
  int q_row0 = 0, k_row0 = 0, sq = p.seqlen_q, sk = p.seqlen_k;
  if (varlen) {
    q_row0 = p.cu_seqlens_q[b];
    sq = p.cu_seqlens_q[b + 1] - q_row0;
    k_row0 = p.cu_seqlens_k[b];
    sk = p.cu_seqlens_k[b + 1] - k_row0;
  }
  if (p.seqused_k) sk = p.seqused_k[b];
  if (!varlen) sk = min(sk, p.seqlen_k);           // never past the cache capacity
  const int rows = sq * p.r;                       // packed rows of this KV head
  const int prow0 = chunk * NR;
  if (prow0 >= rows) return;                       // chunk past this sequence's rows
  const int off = sk - sq;
  const bool split_mode = p.write_partial != 0;
  const int s_lo = min(sk, split * p.split_len);
  const int s_hi = min(sk, (split + 1) * p.split_len);

  // per-row visible key interval [lo, hi] (inclusive) inside this split
  int lo[NR], hi[NR];
  int klo = INT32_MAX, khi = -1;
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) {
    const int pr = prow0 + rr;
    lo[rr] = 1;
    hi[rr] = 0;
    if (pr < rows) {
      const int i = pr / p.r;
      int l = s_lo, h = s_hi - 1;
      if (p.wl >= 0) l = max(l, i + off - p.wl);
      if (p.wr >= 0) h = min(h, i + off + p.wr);
      l = max(l, 0);
      if (l <= h) {
        lo[rr] = l;
        hi[rr] = h;
        klo = min(klo, l);
        khi = max(khi, h + 1);
      }
    }
  }

  auto row_out = [&](int rr, int& i, int& h) {
    const int pr = prow0 + rr;
    i = pr / p.r;
    h = g * p.r + pr % p.r;
  };
  auto write_row = [&](int rr, int d, float o, float lse_v, bool write_lse) {
    int i, h;
    row_out(rr, i, h);
    if (split_mode) {
      const int64_t rows_total = varlen ? p.total_q : int64_t(p.batch) * p.seqlen_q;
      const int64_t ri = varlen ? int64_t(q_row0 + i) : int64_t(b) * p.seqlen_q + i;
      p.out_partial[((int64_t(split) * rows_total + ri) * p.hq + h) * DV + d] = o;
      if (write_lse) {
        const int64_t li = varlen ? (int64_t(split) * p.hq + h) * p.total_q + q_row0 + i
                                  : ((int64_t(split) * p.batch + b) * p.hq + h) * p.seqlen_q + i;
        p.lse_partial[li] = lse_v;
      }
    } else {
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
      out[(varlen ? 0 : int64_t(b) * p.o_bs) + int64_t(q_row0 + i) * p.o_rs + int64_t(h) * p.o_hs + d] =
          __float2bfloat16_rn(o);
      if (write_lse && p.lse) {
        const int64_t li = varlen ? int64_t(h) * p.total_q + q_row0 + i
                                  : (int64_t(b) * p.hq + h) * p.seqlen_q + i;
        p.lse[li] = lse_v;
      }
    }
  };

  if (khi <= klo) {   // nothing visible in this split for any row: O = 0, LSE = -inf
    for (int idx = tid; idx < NR * DV; idx += blockDim.x) {
      const int rr = idx / DV, d = idx % DV;
      if (prow0 + rr < rows) write_row(rr, d, 0.f, -INFINITY, d == 0);
    }
    return;
  }

  const int key_base = (klo / kTileKeys) * kTileKeys;
  const int ntiles = (khi - key_base + kTileKeys - 1) / kTileKeys;

  if (tid == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // q rows -> fp32 with the softmax scale (base 2) and the K descale folded in
  const float qscale = p.scale_log2 * (p.k_descale ? p.k_descale[int64_t(b) * p.hkv + g] : 1.f);
  for (int idx = tid; idx < NR * DK; idx += blockDim.x) {
    const int rr = idx / DK, d = idx % DK;
    float v = 0.f;
    if (prow0 + rr < rows) {
      int i, h;
      row_out(rr, i, h);
      const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(p.q);
      v = __bfloat162float(q[(varlen ? 0 : int64_t(b) * p.q_bs) + int64_t(q_row0 + i) * p.q_rs +
                             int64_t(h) * p.q_hs + d]) *
          qscale;
    }
    q_s[idx] = v;
  }
  __syncthreads();

  const WaitGuard guard{abort_flag, p.status, p.timeout_ns};

  if (warp == kDecWarps) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      const int kb = varlen ? 0 : b;
      constexpr int INNER = 128 / C::ES;   // elements per box row
      const bool paged = p.page_table != nullptr;
      const int rpl = paged ? min(kTileKeys, p.page_size) : kTileKeys;   // rows per load
      int t = 0;
      for (; t < ntiles; ++t) {
        const int st = t % C::NSTAGE;
        const int key = key_base + t * kTileKeys;
        if (!paged) {
          if (t >= C::NSTAGE && !mbar_wait(&empty[st], ((t / C::NSTAGE) - 1) & 1, guard)) break;
          uint8_t* dst = smem + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
          const int row = k_row0 + key;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(dst + c * kBoxBytes, &mapK, &full[st], c * INNER, row, g, kb);
#pragma unroll
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(dst + (C::KCH + c) * kBoxBytes, &mapV, &full[st], c * INNER, row, g, kb);
        } else {
          // the page of the tile's first key, read before the slot wait so
          // that its latency overlaps it (pages of 64+ keys: one per tile)
          const int pi0 = key / p.page_size;
          const int page0 = pi0 < p.max_pages ? p.page_table[int64_t(b) * p.max_pages + pi0] : p.num_pages;
          if (t >= C::NSTAGE && !mbar_wait(&empty[st], ((t / C::NSTAGE) - 1) & 1, guard)) break;
          uint8_t* dst = smem + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
          for (int sub = 0; sub < kTileKeys; sub += rpl) {
            const int kk = key + sub;
            const int pi = kk / p.page_size;
            const int page =
                sub == 0 ? page0 : (pi < p.max_pages ? p.page_table[int64_t(b) * p.max_pages + pi] : p.num_pages);
            const int r = kk - pi * p.page_size;
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(dst + c * kBoxBytes + sub * 128, &mapK, &full[st], c * INNER, r, g, page);
#pragma unroll
            for (int c = 0; c < C::VCH; ++c)
              tma_load_4d(dst + (C::KCH + c) * kBoxBytes + sub * 128, &mapV, &full[st], c * INNER, r, g, page);
          }
        }
      }
      // drain: never leave a copy in flight into shared memory of an exiting CTA
      const WaitGuard drain{abort_flag, p.status, p.timeout_ns};
      for (int u = max(0, t - C::NSTAGE); u < t; ++u) {
        const uint32_t a = smem_u32(&full[u % C::NSTAGE]);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, (u / C::NSTAGE) & 1) && global_timer_ns() - t0 < drain.timeout_ns) {
        }
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  // Lane = (key slot kq in 0..7, dim quarter qp in 0..3); each lane takes keys
  // kq and kq + 8 of its warp's 16, so every q load feeds two keys. Products
  // run as packed fp32 pairs (FFMA2); a 2-level shuffle sums the quarters.
  const int kq = lane & 7, qp = lane >> 3;
  const int kw0 = warp * 16 + kq, kw1 = kw0 + 8;   // keys inside a tile
  constexpr int E = C::E;
  constexpr int QCH = DK / 32;                     // 8-dim chunks per quarter
  float2 o[NR][E / 2];
  float m_run[NR], l_run[NR];
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) {
    m_run[rr] = -INFINITY;
    l_run[rr] = 0.f;
#pragma unroll
    for (int e = 0; e < E / 2; ++e) o[rr][e] = make_float2(0.f, 0.f);
  }
  float* pw = p_s + warp * 16 * NR;
  const int e0 = lane * E;                       // first output column of this lane
  // this lane's columns inside a V row: box, 16-byte granule, byte in it
  const int vbox = e0 * C::ES / 128, vch = (e0 * C::ES % 128) / 16, vbyte = e0 * C::ES % 16;
  const int key_end = min(sk, s_hi);             // keys at or past this are never used

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % C::NSTAGE;
    if (!mbar_wait(&full[st], (t / C::NSTAGE) & 1, guard)) {
      ok = false;
      break;
    }
    const uint8_t* stage = smem + st * C::STAGE_BYTES;
    const int tkey0 = key_base + t * kTileKeys;

    // ---- S = q K^T for two keys over this lane's quarter of the dims ----
    float2 acc0[NR], acc1[NR];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      acc0[rr] = make_float2(0.f, 0.f);
      acc1[rr] = make_float2(0.f, 0.f);
    }
    if constexpr (KVT != 0) {
      // fp8: 16 dims (one 16-byte granule) per load, DK/64 granules per quarter
#pragma unroll
      for (int c = 0; c < DK / 64; ++c) {
        const int gg = qp * (DK / 64) + c;
        const uint8_t* kb = stage + (gg >> 3) * kBoxBytes;
        const uint4 ka = *reinterpret_cast<const uint4*>(kb + kw0 * 128 + (((gg & 7) ^ (kw0 & 7)) << 4));
        const uint4 kc = *reinterpret_cast<const uint4*>(kb + kw1 * 128 + (((gg & 7) ^ (kw1 & 7)) << 4));
        float2 a[8], bb[8];
        fp8x4_to_f32<KVT>(ka.x, a[0], a[1]);
        fp8x4_to_f32<KVT>(ka.y, a[2], a[3]);
        fp8x4_to_f32<KVT>(ka.z, a[4], a[5]);
        fp8x4_to_f32<KVT>(ka.w, a[6], a[7]);
        fp8x4_to_f32<KVT>(kc.x, bb[0], bb[1]);
        fp8x4_to_f32<KVT>(kc.y, bb[2], bb[3]);
        fp8x4_to_f32<KVT>(kc.z, bb[4], bb[5]);
        fp8x4_to_f32<KVT>(kc.w, bb[6], bb[7]);
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float4 qv = *reinterpret_cast<const float4*>(q_s + rr * DK + gg * 16 + u * 4);
            const float2 q0 = make_float2(qv.x, qv.y), q1 = make_float2(qv.z, qv.w);
            acc0[rr] = __ffma2_rn(q0, a[2 * u], acc0[rr]);
            acc0[rr] = __ffma2_rn(q1, a[2 * u + 1], acc0[rr]);
            acc1[rr] = __ffma2_rn(q0, bb[2 * u], acc1[rr]);
            acc1[rr] = __ffma2_rn(q1, bb[2 * u + 1], acc1[rr]);
          }
        }
      }
    } else {
#pragma unroll
    for (int c = 0; c < QCH; ++c) {
      const int gc = qp * QCH + c;
      const uint8_t* kb = stage + (gc >> 3) * kBoxBytes;
      const uint4 ka = *reinterpret_cast<const uint4*>(kb + kw0 * 128 + (((gc & 7) ^ (kw0 & 7)) << 4));
      const uint4 kc = *reinterpret_cast<const uint4*>(kb + kw1 * 128 + (((gc & 7) ^ (kw1 & 7)) << 4));
      const float2 a0 = make_float2(bf16lo_to_f32(ka.x), bf16hi_to_f32(ka.x));
      const float2 a1 = make_float2(bf16lo_to_f32(ka.y), bf16hi_to_f32(ka.y));
      const float2 a2 = make_float2(bf16lo_to_f32(ka.z), bf16hi_to_f32(ka.z));
      const float2 a3 = make_float2(bf16lo_to_f32(ka.w), bf16hi_to_f32(ka.w));
      const float2 b0 = make_float2(bf16lo_to_f32(kc.x), bf16hi_to_f32(kc.x));
      const float2 b1 = make_float2(bf16lo_to_f32(kc.y), bf16hi_to_f32(kc.y));
      const float2 b2 = make_float2(bf16lo_to_f32(kc.z), bf16hi_to_f32(kc.z));
      const float2 b3 = make_float2(bf16lo_to_f32(kc.w), bf16hi_to_f32(kc.w));
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        const float4 qa = *reinterpret_cast<const float4*>(q_s + rr * DK + gc * 8);
        const float4 qb = *reinterpret_cast<const float4*>(q_s + rr * DK + gc * 8 + 4);
        const float2 q0 = make_float2(qa.x, qa.y), q1 = make_float2(qa.z, qa.w);
        const float2 q2 = make_float2(qb.x, qb.y), q3 = make_float2(qb.z, qb.w);
        acc0[rr] = __ffma2_rn(q0, a0, acc0[rr]);
        acc0[rr] = __ffma2_rn(q1, a1, acc0[rr]);
        acc0[rr] = __ffma2_rn(q2, a2, acc0[rr]);
        acc0[rr] = __ffma2_rn(q3, a3, acc0[rr]);
        acc1[rr] = __ffma2_rn(q0, b0, acc1[rr]);
        acc1[rr] = __ffma2_rn(q1, b1, acc1[rr]);
        acc1[rr] = __ffma2_rn(q2, b2, acc1[rr]);
        acc1[rr] = __ffma2_rn(q3, b3, acc1[rr]);
      }
    }
    }
    const int j0 = tkey0 + kw0, j1 = tkey0 + kw1;
    float s0[NR], s1[NR];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      float x0 = acc0[rr].x + acc0[rr].y, x1 = acc1[rr].x + acc1[rr].y;
      x0 += __shfl_xor_sync(0xffffffffu, x0, 8);
      x1 += __shfl_xor_sync(0xffffffffu, x1, 8);
      x0 += __shfl_xor_sync(0xffffffffu, x0, 16);
      x1 += __shfl_xor_sync(0xffffffffu, x1, 16);
      s0[rr] = (j0 >= lo[rr] && j0 <= hi[rr]) ? x0 : -INFINITY;
      s1[rr] = (j1 >= lo[rr] && j1 <= hi[rr]) ? x1 : -INFINITY;
    }
    // ---- online softmax over this warp's 16 keys (base 2) ----
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      float bm = fmaxf(s0[rr], s1[rr]);
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      const float m_new = fmaxf(m_run[rr], bm);
      float factor = 1.f, p0 = 0.f, p1 = 0.f;
      if (m_new != -INFINITY) {
        factor = ex2_approx(m_run[rr] - m_new);
        p0 = ex2_approx(s0[rr] - m_new);
        p1 = ex2_approx(s1[rr] - m_new);
      }
      m_run[rr] = m_new;
      l_run[rr] = l_run[rr] * factor + (p0 + p1);
      const float2 f2 = make_float2(factor, factor);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) o[rr][e] = __fmul2_rn(o[rr][e], f2);
      if (qp == 0) {
        pw[kq * NR + rr] = p0;
        pw[(kq + 8) * NR + rr] = p1;
      }
    }
    __syncwarp();
    // ---- O += P V over the keys this warp owns that exist ----
    const int wkey0 = tkey0 + warp * 16;
    const int kbeg = max(0, klo - wkey0);
    const int kend = min(16, key_end - wkey0);
    auto pv_key = [&](int k2) {
      const int key = warp * 16 + k2;
      const uint8_t* vp = stage + (C::KCH + vbox) * kBoxBytes + key * 128 + (((vch ^ (key & 7)) << 4) + vbyte);
      float2 vf[E / 2];
      if constexpr (KVT != 0 && E == 4) {
        fp8x4_to_f32<KVT>(*reinterpret_cast<const uint32_t*>(vp), vf[0], vf[1]);
      } else if constexpr (KVT != 0 && E == 8) {
        const uint2 w = *reinterpret_cast<const uint2*>(vp);
        fp8x4_to_f32<KVT>(w.x, vf[0], vf[1]);
        fp8x4_to_f32<KVT>(w.y, vf[2], vf[3]);
      } else if constexpr (E == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
        vf[0] = make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
      } else if constexpr (E == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(vp);
        vf[0] = make_float2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
        vf[1] = make_float2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
      } else {
        const uint4 w = *reinterpret_cast<const uint4*>(vp);
        vf[0] = make_float2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
        vf[1] = make_float2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
        vf[2] = make_float2(bf16lo_to_f32(w.z), bf16hi_to_f32(w.z));
        vf[3] = make_float2(bf16lo_to_f32(w.w), bf16hi_to_f32(w.w));
      }
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        const float pr = pw[k2 * NR + rr];
        const float2 p2 = make_float2(pr, pr);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) o[rr][e] = __ffma2_rn(p2, vf[e], o[rr][e]);
      }
    };
    if (kbeg == 0 && kend == 16) {
      // all 16 keys exist (the common case): unrolled so the shared loads overlap
#pragma unroll 4
      for (int k2 = 0; k2 < 16; ++k2) pv_key(k2);
    } else {
      for (int k2 = kbeg; k2 < kend; ++k2) pv_key(k2);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- merge the four warps' states ----
  float lsum[NR];
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) {
    float l = qp == 0 ? l_run[rr] : 0.f;
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    lsum[rr] = l;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");   // ring no longer read
  float* mg = reinterpret_cast<float*>(smem);          // [warp][rr][DV + 2]
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) {
    float* row = mg + (warp * NR + rr) * (DV + 2);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      row[e0 + 2 * e] = o[rr][e].x;
      row[e0 + 2 * e + 1] = o[rr][e].y;
    }
    if (lane == 0) {
      row[DV] = m_run[rr];
      row[DV + 1] = lsum[rr];
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
  if (!ok || *abort_flag) return;
  const float vscale = p.v_descale ? p.v_descale[int64_t(b) * p.hkv + g] : 1.f;
  for (int idx = tid; idx < NR * DV; idx += kDecWarps * 32) {
    const int rr = idx / DV, d = idx % DV;
    if (prow0 + rr >= rows) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mg[(w * NR + rr) * (DV + 2) + DV]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float* row = mg + (w * NR + rr) * (DV + 2);
        const float sc = ex2_approx(row[DV] - M);
        L += row[DV + 1] * sc;
        acc += row[d] * sc;
      }
    }
    const bool empty_row = !(L > 0.f);
    const float ov = empty_row ? 0.f : acc / L * vscale;
    const float lse_v = empty_row ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f;
    write_row(rr, d, ov, lse_v, d == 0);
  }
}

// ---- combine ----------------------------------------------------------------------------
constexpr int kCombineWarps = 8;

template <int DV>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
  constexpr int E = DV / 32;
  const int lane = threadIdx.x & 31;
  const int64_t rows_total = p.varlen ? p.total_q : int64_t(p.batch) * p.seqlen_q;
  const int64_t gw = int64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  if (gw >= rows_total * p.hq) return;
  const int64_t ri = gw / p.hq;
  const int h = static_cast<int>(gw % p.hq);
  int64_t lse_base, lse_split_stride;
  if (p.varlen) {
    lse_base = int64_t(h) * p.total_q + ri;
    lse_split_stride = int64_t(p.hq) * p.total_q;
  } else {
    const int64_t b = ri / p.seqlen_q, i = ri % p.seqlen_q;
    lse_base = (b * p.hq + h) * p.seqlen_q + i;
    lse_split_stride = int64_t(p.batch) * p.hq * p.seqlen_q;
  }
  constexpr float kLog2e = 1.4426950408889634f;
  float M = -INFINITY;
  for (int s = lane; s < p.num_splits; s += 32) M = fmaxf(M, p.lse_partial[lse_base + s * lse_split_stride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float sum = 0.f;
  if (M != -INFINITY)
    for (int s = lane; s < p.num_splits; s += 32) {
      const float l = p.lse_partial[lse_base + s * lse_split_stride];
      if (l != -INFINITY) sum += ex2_approx((l - M) * kLog2e);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const bool empty_row = (M == -INFINITY) || !(sum > 0.f);
  const float lse = empty_row ? -INFINITY : M + logf(sum);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  if (!empty_row) {
    for (int s = 0; s < p.num_splits; ++s) {
      const float l = p.lse_partial[lse_base + s * lse_split_stride];
      if (l == -INFINITY) continue;
      const float w = ex2_approx((l - lse) * kLog2e);
      const float* src = p.out_partial + ((int64_t(s) * rows_total + ri) * p.hq + h) * DV + lane * E;
      if constexpr (E == 2) {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
      } else {
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const float4 v = *reinterpret_cast<const float4*>(src + e);
          acc[e] = fmaf(w, v.x, acc[e]); acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
          acc[e + 2] = fmaf(w, v.z, acc[e + 2]); acc[e + 3] = fmaf(w, v.w, acc[e + 3]);
        }
      }
    }
  }
  int64_t obase;
  if (p.varlen) {
    obase = ri * p.o_rs + int64_t(h) * p.o_hs;
  } else {
    const int64_t b = ri / p.seqlen_q, i = ri % p.seqlen_q;
    obase = b * p.o_bs + i * p.o_rs + int64_t(h) * p.o_hs;
  }
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + obase + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    *reinterpret_cast<__nv_bfloat162*>(out + e) = __floats2bfloat162_rn(acc[e], acc[e + 1]);
  }
  if (p.lse && lane == 0) p.lse[lse_base] = lse;
}

template <int DK, int DV, int NR, int KVT>
cudaError_t launch_decode_t(const FwdParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                            cudaStream_t stream) {
  using C = DecodeCfg<DK, DV, NR, KVT>;
  auto kern = decode_kernel<DK, DV, NR, KVT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int rows = p.max_seqlen_q * p.r;
  const int chunks = (rows + NR - 1) / NR;
  dim3 grid(p.num_splits, p.hkv * chunks, p.batch);
  kern<<<grid, kDecThreads, C::SMEM, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

template <int DK, int DV, int KVT = 0>
cudaError_t launch_decode_nr(const FwdParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                             cudaStream_t stream) {
  // rows per CTA: up to 8 (more would spill the accumulators); larger row
  // counts are split into chunks of 8 over grid.y
  const int rows = p.max_seqlen_q * p.r;
  if (rows <= 1) return launch_decode_t<DK, DV, 1, KVT>(p, mk, mv, stream);
  if (rows <= 2) return launch_decode_t<DK, DV, 2, KVT>(p, mk, mv, stream);
  if (rows <= 4) return launch_decode_t<DK, DV, 4, KVT>(p, mk, mv, stream);
  return launch_decode_t<DK, DV, 8, KVT>(p, mk, mv, stream);
}

}  // namespace

bool decode_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 192 && dv == 128) ||
         (dk == 256 && dv == 256);
}

int decode_max_rows() { return 16; }

cudaError_t launch_decode(const FwdParams& p, int dk, int dv, const CUtensorMap& mk, const CUtensorMap& mv,
                          cudaStream_t stream) {
  if (p.kv_type == 1) {
    if (dk == 128 && dv == 128) return launch_decode_nr<128, 128, 1>(p, mk, mv, stream);
    if (dk == 256 && dv == 256) return launch_decode_nr<256, 256, 1>(p, mk, mv, stream);
    return cudaErrorInvalidValue;
  }
  if (p.kv_type == 2) {
    if (dk == 128 && dv == 128) return launch_decode_nr<128, 128, 2>(p, mk, mv, stream);
    if (dk == 256 && dv == 256) return launch_decode_nr<256, 256, 2>(p, mk, mv, stream);
    return cudaErrorInvalidValue;
  }
  if (dk == 64 && dv == 64) return launch_decode_nr<64, 64>(p, mk, mv, stream);
  if (dk == 128 && dv == 128) return launch_decode_nr<128, 128>(p, mk, mv, stream);
  if (dk == 192 && dv == 128) return launch_decode_nr<192, 128>(p, mk, mv, stream);
  if (dk == 256 && dv == 256) return launch_decode_nr<256, 256>(p, mk, mv, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  const int64_t rows_total = p.varlen ? p.total_q : int64_t(p.batch) * p.seqlen_q;
  const int64_t warps = rows_total * p.hq;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((warps + kCombineWarps - 1) / kCombineWarps);
  switch (p.dv) {
    case 64: combine_kernel<64><<<blocks, kCombineWarps * 32, 0, stream>>>(p); break;
    case 128: combine_kernel<128><<<blocks, kCombineWarps * 32, 0, stream>>>(p); break;
    case 256: combine_kernel<256><<<blocks, kCombineWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
