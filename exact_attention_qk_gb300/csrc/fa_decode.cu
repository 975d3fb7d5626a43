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
//   * four compute warps take 16 keys each per tile and run both products on
//     the tensor cores as warp-level m16n8k16 MMAs with fp32 accumulation:
//     S^T = K q^T (M = the warp's 16 keys, N = 8 packed query rows) and
//     O^T += V^T P^T (M = 16 output columns, N = the same 8 rows). Inside each
//     16-wide K step the fragment's k indices {2t, 2t+1, 2t+8, 2t+9} stand for
//     the four CONSECUTIVE dims (or keys) 4t..4t+3, the same on both operands,
//     so every thread reads its K elements with one 32/64-bit shared load per
//     key; the online softmax (base 2) runs on the S fragments;
//   * the four warps' (m, l, O) states merge in shared memory at the end and the
//     CTA writes either the final bf16 O / fp32 LSE or the fp32 split partials.
// KV-cache forms (the fp8 KV-cache decode and paged-KV passages of the
// FlashAttention sm_120 pull-request page and of `_flash_attn_fwd`):
//   * fp8 (E4M3 / E5M2) caches move one byte per element: a 128-byte box row
//     holds 128 dims; codes convert exactly to f16 pairs straight into the MMA
//     fragments (q is taken to f16 with a power-of-two prescale that keeps it
//     in range), the K descale scales S and the V descale the written O;
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
constexpr int kRows = 8;                     // packed query rows per CTA (the MMAs' N)

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

template <int DK, int DV, int KVT>
struct DecodeCfg {
  // keys per tile: 64 with bf16 elements; 128 with one-byte elements, so a
  // tile moves the same bytes and each warp takes two 16-key groups
  static constexpr int TK = KVT ? 128 : 64;
  static constexpr int G = TK / 64;               // 16-key groups per warp and tile
  static constexpr int BOX = TK * 128;            // one 128-byte x TK-key box
  static constexpr int ES = KVT ? 1 : 2;          // bytes per K/V element
  static constexpr int KCH = DK * ES / 128;       // 128-byte boxes per K row
  static constexpr int VCH = DV * ES / 128;
  static constexpr int STAGE_BYTES = (KCH + VCH) * BOX;
  // Two stages keep a D<=192 CTA near 70 KB of shared memory, so three CTAs
  // share an SM.
  static constexpr int NSTAGE = 2;
  static constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;
  static constexpr int P_BYTES = kDecWarps * kRows * 16 * G * 2;      // per warp: P[row][16 G keys], 16-bit
  static constexpr int MROW = DV + 4;                                 // merge row: O, m, l, pad
  static constexpr int MERGE_BYTES = kDecWarps * kRows * MROW * 4;
  static constexpr int OFF_P = RING_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8 + 16 + 1024;   // + alignment slack
  static_assert(MERGE_BYTES <= RING_BYTES, "merge area reuses the ring");
  static_assert(DK % 16 == 0 && DV % 32 == 0, "MMA shapes");
};

// m16n8k16 MMAs, fp32 accumulate: bf16 or f16 operands (A row-major, B column-major)
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_16816_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp8 codes (the low 16 bits of w; lower byte first) -> f16 pair (exact).
template <int KVT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t w) {
  uint32_t h;
  if constexpr (KVT == 1) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\t}" : "=r"(h) : "r"(w));
  } else {   // E5M2 is the upper byte of an f16
    h = __byte_perm(w, 0u, 0x1404);
  }
  return h;
}

// The same for the high 16 bits of w.
template <int KVT>
__device__ __forceinline__ uint32_t fp8x2_hi_to_f16x2(uint32_t w) {
  uint32_t h;
  if constexpr (KVT == 1) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}" : "=r"(h) : "r"(w));
  } else {
    h = __byte_perm(w, 0u, 0x3424);
  }
  return h;
}

template <int DK, int DV, int KVT>
__global__ void __launch_bounds__(kDecThreads, (DV <= 128) ? 3 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                  const FwdParams p) {
  using C = DecodeCfg<DK, DV, KVT>;
  constexpr int NR = kRows;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the array itself so that every access
  // through it stays a shared-memory access with 32-bit addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint16_t* p_s = reinterpret_cast<uint16_t*>(smem + C::OFF_P);
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

  // visible key interval [lo, hi] (inclusive) of packed row rr inside this
  // split; empty (lo > hi) for padding rows and rows that see nothing here
  auto interval = [&](int rr, int& lo_, int& hi_) {
    const int pr = prow0 + rr;
    lo_ = 1;
    hi_ = 0;
    if (pr < rows) {
      const int i = pr / p.r;
      int l = s_lo, h = s_hi - 1;
      if (p.wl >= 0) l = max(l, i + off - p.wl);
      if (p.wr >= 0) h = min(h, i + off + p.wr);
      l = max(l, 0);
      if (l <= h) {
        lo_ = l;
        hi_ = h;
      }
    }
  };
  int klo = INT32_MAX, khi = -1;
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) {
    int l, h;
    interval(rr, l, h);
    if (l <= h) {
      klo = min(klo, l);
      khi = max(khi, h + 1);
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

  constexpr int TK = C::TK;
  const int key_base = (klo / TK) * TK;
  const int ntiles = (khi - key_base + TK - 1) / TK;

  if (tid == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
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
      // rows per load: a piece inside one page, the same rule as the host's map
      // (the whole tile, else 64 rows, else one page)
      const int ps = p.page_size;
      const int rpl = !paged ? TK : (ps % TK == 0 ? TK : (ps % 64 == 0 ? 64 : ps));
      int t = 0;
      for (; t < ntiles; ++t) {
        const int st = t % C::NSTAGE;
        const int key = key_base + t * TK;
        if (!paged) {
          if (t >= C::NSTAGE && !mbar_wait(&empty[st], ((t / C::NSTAGE) - 1) & 1, guard)) break;
          uint8_t* dst = smem + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
          const int row = k_row0 + key;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(dst + c * C::BOX, &mapK, &full[st], c * INNER, row, g, kb);
#pragma unroll
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(dst + (C::KCH + c) * C::BOX, &mapV, &full[st], c * INNER, row, g, kb);
        } else {
          // the page of the tile's first key, read before the slot wait so
          // that its latency overlaps it (pages of 64+ keys: one per tile)
          const int pi0 = key / p.page_size;
          const int page0 = pi0 < p.max_pages ? p.page_table[int64_t(b) * p.max_pages + pi0] : p.num_pages;
          if (t >= C::NSTAGE && !mbar_wait(&empty[st], ((t / C::NSTAGE) - 1) & 1, guard)) break;
          uint8_t* dst = smem + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
          for (int sub = 0; sub < TK; sub += rpl) {
            const int kk = key + sub;
            const int pi = kk / p.page_size;
            const int page =
                sub == 0 ? page0 : (pi < p.max_pages ? p.page_table[int64_t(b) * p.max_pages + pi] : p.num_pages);
            const int r = kk - pi * p.page_size;
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_4d(dst + c * C::BOX + sub * 128, &mapK, &full[st], c * INNER, r, g, page);
#pragma unroll
            for (int c = 0; c < C::VCH; ++c)
              tma_load_4d(dst + (C::KCH + c) * C::BOX + sub * 128, &mapV, &full[st], c * INNER, r, g, page);
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

  // ---------------- compute warps (tensor cores) ----------------
  // Fragment coordinates of m16n8k16: g8 = lane / 4 picks the row (A) / column
  // (B) group, t4 = lane % 4 the k pair. k indices {2t, 2t+1, 2t+8, 2t+9} of a
  // 16-wide step stand for positions 4t..4t+3 (dims in QK, keys in PV).
  const int g8 = lane >> 2, t4 = lane & 3;
  constexpr int KS = DK / 16;     // QK k steps
  constexpr int MT = DV / 16;     // PV m tiles (16 output columns each)
  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q);

  // q^T as the B operand of S^T = K q^T: row g8 (zero for padding rows), dims
  // 16kk + 4t4 .. +3 (b0 = first two, b1 = last two)
  uint32_t qf[KS][2];
  float sscale = p.scale_log2 * (p.k_descale ? p.k_descale[int64_t(b) * p.hkv + g] : 1.f);
  {
    const bool real = prow0 + g8 < rows;
    const __nv_bfloat16* qrow = qg;
    if (real) {
      int i, h;
      row_out(g8, i, h);
      qrow = qg + (varlen ? 0 : int64_t(b) * p.q_bs) + int64_t(q_row0 + i) * p.q_rs + int64_t(h) * p.q_hs;
    }
    if constexpr (KVT == 0) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint2 w = make_uint2(0u, 0u);
        if (real) w = *reinterpret_cast<const uint2*>(qrow + 16 * kk + 4 * t4);
        qf[kk][0] = w.x;
        qf[kk][1] = w.y;
      }
    } else {
      // f16 operands: q x 2^-e with e >= 0 chosen (per warp; every warp loads
      // the same rows) so that the largest |q| stays below 2^15
      float mx = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint2 w = make_uint2(0u, 0u);
        if (real) w = *reinterpret_cast<const uint2*>(qrow + 16 * kk + 4 * t4);
        qf[kk][0] = w.x;
        qf[kk][1] = w.y;
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16lo_to_f32(w.x)), fabsf(bf16hi_to_f32(w.x))),
                             fmaxf(fabsf(bf16lo_to_f32(w.y)), fabsf(bf16hi_to_f32(w.y)))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const int e = (mx >= 32768.f) ? ilogbf(mx) - 14 : 0;
      sscale = ldexpf(sscale, e);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const __half2 hv = __floats2half2_rn(ldexpf(bf16lo_to_f32(qf[kk][u]), -e),
                                               ldexpf(bf16hi_to_f32(qf[kk][u]), -e));
          qf[kk][u] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      }
    }
  }
  // this thread's two rows (2 t4, 2 t4 + 1) of every S and O fragment
  int lo0, hi0, lo1, hi1;
  interval(2 * t4, lo0, hi0);
  interval(2 * t4 + 1, lo1, hi1);
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // l: this thread's keys only
  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  constexpr int G = C::G;
  constexpr int WK = 16 * G;                      // keys per warp and tile
  uint16_t* pw = p_s + warp * (NR * WK);          // this warp's P[row][WK keys]
  const int key_end = min(sk, s_hi);              // keys at or past this are never used

  // Byte offsets (from stage 0) of this thread's first K and V fragment words.
  // The 128-byte swizzle stores 16-byte granule j of tile row r at granule
  // j ^ (r & 7). The rows one thread reads in a fragment agree in their low
  // three bits with a per-thread value, so a fragment word of k step kk (K) or
  // of column block j and key i (V) sits at (offset ^ (c << 4)) + d, with c
  // and d compile-time constants.
  uint32_t kofs, vofs;
  if constexpr (KVT == 0) {
    kofs = (warp * WK + g8) * 128 + ((((t4 >> 1) ^ g8)) << 4) + 8 * (t4 & 1);
    vofs = C::KCH * C::BOX + (warp * WK + 4 * t4) * 128 + ((((g8 >> 1) ^ (4 * (t4 & 1)))) << 4) + 8 * (g8 & 1);
  } else {
    kofs = (warp * WK + g8) * 128 + (g8 << 4) + 4 * t4;
    vofs = C::KCH * C::BOX + (warp * WK + 4 * t4) * 128 + ((((g8 >> 2) ^ (4 * (t4 & 1)))) << 4) + 4 * (g8 & 3);
  }
  auto lds32 = [&](uint32_t o) { return *reinterpret_cast<const uint32_t*>(smem + o); };
  auto lds64 = [&](uint32_t o) { return *reinterpret_cast<const uint2*>(smem + o); };

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % C::NSTAGE;
    if (!mbar_wait(&full[st], (t / C::NSTAGE) & 1, guard)) {
      ok = false;
      break;
    }
    uint8_t* stage = smem + st * C::STAGE_BYTES;
    const int tkey0 = key_base + t * TK;
    const uint32_t kst = st * C::STAGE_BYTES + kofs, vst = st * C::STAGE_BYTES + vofs;

    // V rows at or past key_end may hold anything (NaN included). The warp
    // whose rows reach them zeroes them in shared memory before its P.V, so
    // that no 0 * NaN reaches O; the fence orders these writes before the
    // next TMA write into the stage.
    const int vlim = key_end - tkey0;
    const bool vtail = vlim < warp * WK + WK;
    if (vtail) {
      const int r0 = max(vlim, warp * WK);
      const int nchunk = (warp * WK + WK - r0) * C::VCH * 8;
      for (int idx = lane; idx < nchunk; idx += 32) {
        const int rr = r0 + idx / (C::VCH * 8), rem = idx % (C::VCH * 8);
        *reinterpret_cast<uint4*>(stage + (C::KCH + rem / 8) * C::BOX + rr * 128 + (rem % 8) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }

    // ---- S^T = K q^T over this warp's WK keys, in 16-key groups ----
    float sv[G][4];
#pragma unroll
    for (int grp = 0; grp < G; ++grp) {
      const int ka = warp * WK + grp * 16 + g8, kb = ka + 8;   // this thread's two keys (tile rows)
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        if constexpr (KVT == 0) {
          // dims 16kk + 4t4 .. +3: 8 bytes in box kk/4, granule 2(kk%4) + t4/2; row kb = ka + 8
          const uint32_t o = (kst ^ ((2 * (kk & 3)) << 4)) + (kk >> 2) * C::BOX + grp * 2048;
          const uint2 x = lds64(o), y = lds64(o + 1024);
          mma_16816_bf16(sacc, x.x, y.x, x.y, y.y, qf[kk][0], qf[kk][1]);
        } else {
          // dims 16kk + 4t4 .. +3: 4 bytes in box kk/8, granule kk%8
          const uint32_t o = (kst ^ ((kk & 7) << 4)) + (kk >> 3) * C::BOX + grp * 2048;
          const uint32_t x = lds32(o), y = lds32(o + 1024);
          mma_16816_f16(sacc, fp8x2_to_f16x2<KVT>(x), fp8x2_to_f16x2<KVT>(y), fp8x2_hi_to_f16x2<KVT>(x),
                        fp8x2_hi_to_f16x2<KVT>(y), qf[kk][0], qf[kk][1]);
        }
      }
      // sacc: (key ka, row 2t4), (ka, 2t4+1), (kb, 2t4), (kb, 2t4+1); base-2 scores
      const int ja = tkey0 + ka, jb = tkey0 + kb;
      sv[grp][0] = (ja >= lo0 && ja <= hi0) ? sacc[0] * sscale : -INFINITY;
      sv[grp][1] = (ja >= lo1 && ja <= hi1) ? sacc[1] * sscale : -INFINITY;
      sv[grp][2] = (jb >= lo0 && jb <= hi0) ? sacc[2] * sscale : -INFINITY;
      sv[grp][3] = (jb >= lo1 && jb <= hi1) ? sacc[3] * sscale : -INFINITY;
    }
    // ---- online softmax over the warp's keys (rows 2t4 and 2t4+1) ----
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int grp = 0; grp < G; ++grp) {
      bm0 = fmax3(bm0, sv[grp][0], sv[grp][2]);
      bm1 = fmax3(bm1, sv[grp][1], sv[grp][3]);
    }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
    }
    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
    float f0 = 1.f, f1 = 1.f;
    float pv[G][4];
#pragma unroll
    for (int grp = 0; grp < G; ++grp) pv[grp][0] = pv[grp][1] = pv[grp][2] = pv[grp][3] = 0.f;
    if (mn0 != -INFINITY) {
      f0 = ex2_approx(m0 - mn0);
#pragma unroll
      for (int grp = 0; grp < G; ++grp) {
        pv[grp][0] = ex2_approx(sv[grp][0] - mn0);
        pv[grp][2] = ex2_approx(sv[grp][2] - mn0);
      }
    }
    if (mn1 != -INFINITY) {
      f1 = ex2_approx(m1 - mn1);
#pragma unroll
      for (int grp = 0; grp < G; ++grp) {
        pv[grp][1] = ex2_approx(sv[grp][1] - mn1);
        pv[grp][3] = ex2_approx(sv[grp][3] - mn1);
      }
    }
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int grp = 0; grp < G; ++grp) {
      ps0 += pv[grp][0] + pv[grp][2];
      ps1 += pv[grp][1] + pv[grp][3];
    }
    l0 = l0 * f0 + ps0;
    l1 = l1 * f1 + ps1;
    if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= f0;
        o[mt][1] *= f1;
        o[mt][2] *= f0;
        o[mt][3] *= f1;
      }
    }
    // P -> shared memory as P[row][key] (16-bit: bf16 with bf16 V, f16 with fp8 V)
    auto p16 = [](float v) -> uint16_t {
      if constexpr (KVT == 0) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
      } else {
        return __half_as_ushort(__float2half_rn(v));
      }
    };
#pragma unroll
    for (int grp = 0; grp < G; ++grp) {
      pw[(2 * t4) * WK + grp * 16 + g8] = p16(pv[grp][0]);
      pw[(2 * t4 + 1) * WK + grp * 16 + g8] = p16(pv[grp][1]);
      pw[(2 * t4) * WK + grp * 16 + g8 + 8] = p16(pv[grp][2]);
      pw[(2 * t4 + 1) * WK + grp * 16 + g8 + 8] = p16(pv[grp][3]);
    }
    __syncwarp();
    // ---- O^T += V^T P^T, one 16-key group at a time ----
#pragma unroll
    for (int grp = 0; grp < G; ++grp) {
      // P^T as the B operand: row g8, keys 16 grp + 4t4 .. +3
      const uint2 pf = *reinterpret_cast<const uint2*>(pw + g8 * WK + grp * 16 + 4 * t4);
      // this thread's V rows (tile keys) are warp * WK + grp * 16 + 4 t4 + i, i < 4
#pragma unroll
      for (int j = 0; j < DV / 32; ++j) {
        // columns 32j + 4g8 .. +3: m tile 2j holds (4g8, 4g8+1), m tile 2j+1 (4g8+2, 4g8+3)
        if constexpr (KVT == 0) {
          // granule 4(j%2) + g8/2 of box j/2
          uint2 r[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            r[i] = lds64((vst ^ ((i ^ (4 * (j & 1))) << 4)) + (j >> 1) * C::BOX + grp * 2048 + i * 128);
          mma_16816_bf16(o[2 * j], __byte_perm(r[0].x, r[1].x, 0x5410), __byte_perm(r[0].x, r[1].x, 0x7632),
                         __byte_perm(r[2].x, r[3].x, 0x5410), __byte_perm(r[2].x, r[3].x, 0x7632), pf.x, pf.y);
          mma_16816_bf16(o[2 * j + 1], __byte_perm(r[0].y, r[1].y, 0x5410), __byte_perm(r[0].y, r[1].y, 0x7632),
                         __byte_perm(r[2].y, r[3].y, 0x5410), __byte_perm(r[2].y, r[3].y, 0x7632), pf.x, pf.y);
        } else {
          // granule 2(j%4) + g8/4 of box j/4
          uint32_t r[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            r[i] = lds32((vst ^ ((i ^ (2 * (j & 3))) << 4)) + (j >> 2) * C::BOX + grp * 2048 + i * 128);
          // byte pairs (key 4t4 + 2c, key 4t4 + 2c + 1) of one column
          const uint32_t c01a = __byte_perm(r[0], r[1], 0x5140), c23a = __byte_perm(r[0], r[1], 0x7362);
          const uint32_t c01b = __byte_perm(r[2], r[3], 0x5140), c23b = __byte_perm(r[2], r[3], 0x7362);
          mma_16816_f16(o[2 * j], fp8x2_to_f16x2<KVT>(c01a), fp8x2_hi_to_f16x2<KVT>(c01a),
                        fp8x2_to_f16x2<KVT>(c01b), fp8x2_hi_to_f16x2<KVT>(c01b), pf.x, pf.y);
          mma_16816_f16(o[2 * j + 1], fp8x2_to_f16x2<KVT>(c23a), fp8x2_hi_to_f16x2<KVT>(c23a),
                        fp8x2_to_f16x2<KVT>(c23b), fp8x2_hi_to_f16x2<KVT>(c23b), pf.x, pf.y);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- merge the four warps' states ----
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");   // ring no longer read
  float* mg = reinterpret_cast<float*>(smem);          // [warp][row][DV + 4]
  {
    float* r0 = mg + (warp * NR + 2 * t4) * C::MROW;
    float* r1 = r0 + C::MROW;
#pragma unroll
    for (int j = 0; j < DV / 32; ++j) {
      const int c = 32 * j + 4 * g8;
      *reinterpret_cast<float4*>(r0 + c) = make_float4(o[2 * j][0], o[2 * j][2], o[2 * j + 1][0], o[2 * j + 1][2]);
      *reinterpret_cast<float4*>(r1 + c) = make_float4(o[2 * j][1], o[2 * j][3], o[2 * j + 1][1], o[2 * j + 1][3]);
    }
    if (g8 == 0) {
      r0[DV] = m0;
      r0[DV + 1] = l0;
      r1[DV] = m1;
      r1[DV + 1] = l1;
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
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mg[(w * NR + rr) * C::MROW + DV]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float* row = mg + (w * NR + rr) * C::MROW;
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

template <int DK, int DV, int KVT = 0>
cudaError_t launch_decode_t(const FwdParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                            cudaStream_t stream) {
  using C = DecodeCfg<DK, DV, KVT>;
  auto kern = decode_kernel<DK, DV, KVT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // packed rows (query rows x heads per KV head) in chunks of kRows over grid.y
  const long long rows = static_cast<long long>(p.max_seqlen_q) * p.r;
  const long long chunks = (rows + kRows - 1) / kRows;
  // grid.y and grid.z are limited to 65535 (long fp8 prefills can exceed it)
  if (p.hkv * chunks > 65535 || p.batch > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(p.num_splits, static_cast<unsigned>(p.hkv * chunks), p.batch);
  kern<<<grid, kDecThreads, C::SMEM, stream>>>(mk, mv, p);
  return cudaGetLastError();
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
    if (dk == 128 && dv == 128) return launch_decode_t<128, 128, 1>(p, mk, mv, stream);
    if (dk == 256 && dv == 256) return launch_decode_t<256, 256, 1>(p, mk, mv, stream);
    return cudaErrorInvalidValue;
  }
  if (p.kv_type == 2) {
    if (dk == 128 && dv == 128) return launch_decode_t<128, 128, 2>(p, mk, mv, stream);
    if (dk == 256 && dv == 256) return launch_decode_t<256, 256, 2>(p, mk, mv, stream);
    return cudaErrorInvalidValue;
  }
  if (dk == 64 && dv == 64) return launch_decode_t<64, 64>(p, mk, mv, stream);
  if (dk == 128 && dv == 128) return launch_decode_t<128, 128>(p, mk, mv, stream);
  if (dk == 192 && dv == 128) return launch_decode_t<192, 128>(p, mk, mv, stream);
  if (dk == 256 && dv == 256) return launch_decode_t<256, 256>(p, mk, mv, stream);
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
