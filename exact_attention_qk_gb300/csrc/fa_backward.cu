// fa_backward.cu - attention backward (dQ, dK, dV) on tcgen05.
//
// The backward of "mslk/attention/flash_attn/flash_bwd_sm100.py": a
// preprocess pass forms D = rowsum(dO * O) from the forward's output; the main
// loop recomputes P = exp(scale * Q K^T - LSE) from the stored LSE, then
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
// The page's kernel accumulates dQ of every key block through global fp32
// atomics; here dQ has a kernel of its own instead, which recomputes S and dP
// per query tile and keeps dQ in tensor memory. That costs two extra GEMMs per
// (query tile, key block) pair but needs no atomics, no fp32 dQ buffer and no
// conversion pass, and the result does not depend on the order blocks finish.
//
//   bwd_preprocess_kernel: lse2 = LSE * log2(e) (+inf for rows without keys
//     and for the padding rows) and D, per (sequence, q head, row).
//   bwd_dq_kernel: one CTA per (128-row query tile, q head, sequence);
//     S = Q K^T and dP = dO V^T for each visible key block, dS in bf16 back
//     into tensor memory, dQ += dS K.
//   bwd_dkdv_kernel: one CTA per (128-key block, KV head, sequence), looping
//     over the q heads of its group and the query tiles that see the block;
//     S^T = K Q^T and dP^T = V dO^T, P^T and dS^T in bf16 back into tensor
//     memory, dV += P^T dO and dK += dS^T Q.
//
// Tensor memory (512 columns, one CTA per SM): S [0,128), dP [128,256),
// accumulators from 256 (dQ; or dV then dK). With the (192, 128) head dims
// dV and dK together (128 + 192 columns) do not fit beside S and dP, so the
// dK/dV kernel runs as two launches: a dV-only pass (S^T, P^T, dV += P^T dO)
// and a dK-only pass (S^T, dP^T, dS^T, dK += dS^T Q). Where two stages of the
// streamed tile pair do not fit in shared memory, its two tiles get rings of
// their own: the 192-column tile (K; Q) two stages, the 128-column one (V; dO)
// one stage, which only the job's first GEMM reads. Two warpgroups share each
// 128 x 128 score block, warpgroup c taking columns [64c, 64c+64) for all 128
// rows, in two phases: P from S (the dK/dV kernel writes P^T back in bf16),
// then dS from dP and the P kept in registers, back in bf16. A bf16 result of
// half c lands in columns [64c, 64c+32) of its own fp32 half, which only that
// warpgroup reads. The MMA thread orders its GEMMs so that each phase of the
// warps overlaps two GEMMs of the tensor pipe (see the issue orders below).
// Every GEMM has the operand forms of the forward kernel: SS with two K-major
// 128B-swizzled tiles, and TS with the bf16 A operand in tensor memory and an
// MN-major B tile.
//
// Warps 0-7 compute (thread t of a warpgroup owns row t of the tile, tensor-
// memory lane t), warp 8 issues the TMA loads, warp 9 the MMAs (one thread).
// Every wait is bounded; on a timeout the CTA raises its abort flag, records
// the failure in the device status word, drains its copies and MMAs, frees
// tensor memory and returns.
#include <cuda_bf16.h>

#include <type_traits>


#include "fa_kernels.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kB = 128;                 // rows of a query tile and of a key block
constexpr int kChunk = 128 * 128;       // bytes of 128 rows x 64 bf16 columns (one 128B-swizzle chunk)

// Passes of the dK/dV kernel: both accumulators (head dims 64 and 128), or
// the dV-only and dK-only passes of the (192, 128) and (256, 256) head dims.
enum : int { kBoth = 0, kDvOnly = 1, kDkOnly = 2 };

template <int DK_, int DV_, int MODE_ = kBoth>
struct BwdCfg {
  static constexpr int DK = DK_, DV = DV_, MODE = MODE_;
  static constexpr int CQ = DK / 64, CV = DV / 64;     // 64-column chunks of a Q or K row, of a dO or V row
  static constexpr int TQ = CQ * kChunk;               // one 128-row tile of Q or K
  static constexpr int TV = CV * kChunk;               // one 128-row tile of dO or V
  static constexpr int PAIR = TQ + TV;
  // resident: Q, dO (dQ) or K, V (dK/dV; K alone in the dV-only pass)
  static constexpr int RES = (MODE == kDvOnly) ? TQ : PAIR;
  // The streamed pair (K, V for dQ; Q, dO and lse2 / D for dK/dV), in the
  // first of these layouts that fits the shared memory:
  //   PAIR2  the pair in two stages;
  //   SPLIT2 rings of their own: the A tile (K; Q with lse2 / D) two stages,
  //          the B tile (V; dO) one, which suffices since only the job's
  //          first GEMM reads it (dP = dO V^T);
  //   PAIR1  the pair in one stage;
  //   BHALF  the A tile one stage, the B tile in two halves (64-column
  //          chunk pairs) through one half-tile slot: dP takes the two
  //          halves of its contraction one after the other.
  static constexpr int LIM = 227 * 1024 - 2048;       // tiles and lse2 / D (barriers aside)
  static constexpr bool PAIR2 = RES + 2 * (PAIR + 1024) <= LIM;
  static constexpr bool SPLIT2 = !PAIR2 && RES + 2 * (TQ + 1024) + TV <= LIM;
  static constexpr bool PAIR1 = !PAIR2 && !SPLIT2 && RES + PAIR + 1024 <= LIM;
  static constexpr bool BHALF = !PAIR2 && !SPLIT2 && !PAIR1;
  static constexpr bool SPLIT = SPLIT2 || BHALF;      // the B tile in a ring of its own
  static constexpr int ST = (PAIR2 || SPLIT2) ? 2 : 1; // stages of the pair, or of the A tile
  static constexpr int A_BYTES = SPLIT ? TQ : PAIR;    // one stage of that ring
  static constexpr int B_PARTS = BHALF ? 2 : 1;        // B loads per job
  static constexpr int B_BYTES = TV / B_PARTS;         // SPLIT: the B slot
  static constexpr int OFF_RES = 0;
  static constexpr int OFF_STR = RES;
  static constexpr int OFF_B = OFF_STR + ST * A_BYTES; // SPLIT: the B slot
  static constexpr int OFF_VEC = OFF_B + (SPLIT ? B_BYTES : 0);   // dK/dV: lse2[128], D[128] per stage
  static constexpr int OFF_BAR = OFF_VEC + ST * 1024;
  static constexpr int NBAR = 18;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  // at least half the SM's shared memory: one CTA (owning all 512 tensor-memory
  // columns) per SM
  static constexpr int SMEM = (SMEM_USED + 1024 < 120 * 1024) ? 120 * 1024 : SMEM_USED + 1024;
  static constexpr int THREADS = 320;
  static constexpr int TMA_WARP = 8, MMA_WARP = 9;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(OFF_STR % 1024 == 0 && PAIR % 1024 == 0 && B_BYTES % 1024 == 0,
                "128B-swizzled tiles start 1024-byte aligned");
  static_assert(!BHALF || (RES + TQ + 1024 + TV / 2 <= LIM && CV % 2 == 0), "a layout that fits");
};

struct BBars {
  uint64_t* res_full;   // resident pair landed
  uint64_t* str_full;   // [ST]
  uint64_t* str_empty;  // [ST]
  uint64_t* s_full;     // S of the current job complete
  uint64_t* dp_full;    // dP of the current job complete
  uint64_t* p_done;     // [2] per column half: S read (and P^T written) by its warpgroup (4 arrivals)
  uint64_t* ds_full;    // [2] per column half: dS written by its warpgroup (4 arrivals)
  uint64_t* acc_full;   // accumulators final
  uint64_t* drain;
  uint64_t* k_fixed;    // dQ kernel, seqused_k: K rows past the used keys cleared
  uint64_t* b_full;     // SPLIT: the B tile's stage landed
  uint64_t* b_empty;    // SPLIT: the B tile's stage read
};

template <class Cfg>
__device__ __forceinline__ BBars carve(uint8_t* smem) {
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  BBars B;
  B.res_full = b; b += 1;
  B.str_full = b; b += Cfg::ST;
  B.str_empty = b; b += Cfg::ST;
  B.s_full = b; b += 1;
  B.dp_full = b; b += 1;
  B.p_done = b; b += 2;
  B.ds_full = b; b += 2;
  B.acc_full = b; b += 1;
  B.drain = b; b += 1;
  B.k_fixed = b; b += 1;
  B.b_full = b; b += 1;
  B.b_empty = b; b += 1;
  return B;
}

template <class Cfg>
__device__ __forceinline__ void init_bars(const BBars& B) {
  mbar_init(B.res_full, 1);
  for (int i = 0; i < Cfg::ST; ++i) {
    mbar_init(&B.str_full[i], 1);
    mbar_init(&B.str_empty[i], 1);
  }
  mbar_init(B.s_full, 1);
  mbar_init(B.dp_full, 1);
  for (int i = 0; i < 2; ++i) {
    mbar_init(&B.p_done[i], 4);
    mbar_init(&B.ds_full[i], 4);
  }
  mbar_init(B.acc_full, 1);
  mbar_init(B.drain, 1);
  mbar_init(B.k_fixed, 1);
  mbar_init(B.b_full, 1);
  mbar_init(B.b_empty, 1);
  fence_barrier_init();
}

// Spin (bounded, ignoring the abort flag) until the given phase completed:
// used to drain copies / MMAs in flight before the CTA exits.
__device__ __forceinline__ void drain_phase(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity) && global_timer_ns() - t0 < timeout_ns) {
  }
}

// D[128 x 128] = A[128 x kdim] B[128 x kdim]^T, both K-major 128B-swizzled
// tiles of 64-column chunks (16 bf16 per instruction).
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, int kdim, uint32_t idesc) {
  const uint64_t ad = sdesc_sw128(a_base, 16, 1024), bd = sdesc_sw128(b_base, 16, 1024);
  for (int kk = 0; kk < kdim / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
    mma_bf16_ss(d_tmem, ad + off, bd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// The 16-deep steps [kk0, kk1) of such a product, accumulating from kk0 > 0 on;
// B's 64-column chunks sit at b_base from chunk b_chunk0 on (a half slot).
__device__ __forceinline__ void issue_ss_part(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, int kk0, int kk1,
                                              int b_chunk0, uint32_t idesc) {
  const uint64_t ad = sdesc_sw128(a_base, 16, 1024), bd = sdesc_sw128(b_base, 16, 1024);
  for (int kk = kk0; kk < kk1; ++kk) {
    const uint32_t aoff = ((kk >> 2) * kChunk + (kk & 3) * 32) >> 4;
    const uint32_t boff = (((kk >> 2) - b_chunk0) * kChunk + (kk & 3) * 32) >> 4;
    mma_bf16_ss(d_tmem, ad + aoff, bd + boff, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[128 x N] (+)= A_h B_h for half h of the 128-deep contraction: A is bf16 in
// tensor memory (columns [64h, 64h+32) of a_tmem, two values per column), B is
// rows [64h, 64h+64) of an MN-major tile (64-column chunks kChunk bytes apart).
__device__ __forceinline__ void issue_ts_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, int h,
                                              uint32_t idesc, bool acc) {
  const uint64_t bd = sdesc_sw128(b_base, kChunk, 1024);
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int kk = h * 4 + k4;
    mma_bf16_ts(d_tmem, a_tmem + h * 64 + k4 * 8, bd + ((kk * 16 * 128) >> 4), idesc, (acc || k4 > 0) ? 1u : 0u);
  }
}

// The same for the first `steps` (0..4) 16-deep slices of half h only.
__device__ __forceinline__ void issue_ts_half_steps(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, int h,
                                                    uint32_t idesc, bool acc, int steps) {
  const uint64_t bd = sdesc_sw128(b_base, kChunk, 1024);
  for (int k4 = 0; k4 < steps; ++k4) {
    const int kk = h * 4 + k4;
    mma_bf16_ts(d_tmem, a_tmem + h * 64 + k4 * 8, bd + ((kk * 16 * 128) >> 4), idesc, (acc || k4 > 0) ? 1u : 0u);
  }
}

// 32 fp32 accumulator columns of one row, times f, to 64 bytes of bf16
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&o)[32], float f) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * f, __uint_as_float(o[2 * e + 1]) * f);
  if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {   // whole 32-byte sectors
    st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
    st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
    return;
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
  d4[2] = make_uint4(w[8], w[9], w[10], w[11]);
  d4[3] = make_uint4(w[12], w[13], w[14], w[15]);
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* dst, int d) {
  for (int c = 0; c < d / 8; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
}

// One sequence of the call: its lengths, its first rows in q's and k's row
// axes (0 when batched), the batch coordinate of the tensor maps and the
// first workspace row of q head h.
// sk: the keys that exist (seqused_k[b] when given); ska: the key rows the
// sequence owns in k's row axis (its capacity), whose rows at or past sk the
// dK/dV kernel sets to 0.
struct BSeq {
  int sq, sk, ska, q_row0, k_row0, bc;
};

__device__ __forceinline__ BSeq bwd_seq(const BwdParams& p, int b) {
  BSeq S;
  if (p.cu_seqlens_q != nullptr) {
    S.q_row0 = p.cu_seqlens_q[b];
    S.sq = p.cu_seqlens_q[b + 1] - S.q_row0;
    S.k_row0 = p.cu_seqlens_k[b];
    S.ska = p.cu_seqlens_k[b + 1] - S.k_row0;
    S.bc = 0;
  } else {
    S.q_row0 = S.k_row0 = 0;
    S.sq = p.seqlen_q;
    S.ska = p.seqlen_k;
    S.bc = b;
  }
  S.sk = p.seqused_k != nullptr ? min(p.seqused_k[b], S.ska) : S.ska;
  return S;
}

__device__ __forceinline__ int64_t ws_row0(const BwdParams& p, int b, int h) {
  return p.cu_seqlens_q != nullptr ? int64_t(h) * p.ws_rows + bwd_ws_row0(p.cu_seqlens_q, b)
                                   : (int64_t(b) * p.hq + h) * p.sq_pad;
}

// ---------------------------------------------------------------------------
// preprocess: one CTA per (sequence, 128-row block, q head), 8 threads per row
__global__ void __launch_bounds__(1024) bwd_preprocess_kernel(const BwdParams p, int dv, int max_mb) {
  const int b = blockIdx.x / max_mb, m = blockIdx.x % max_mb, h = blockIdx.y;
  const BSeq S = bwd_seq(p, b);
  if (m * 128 >= S.sq) return;   // (whole CTA)
  const int sub = threadIdx.x & 7;
  const int i = m * 128 + (threadIdx.x >> 3);
  float acc = 0.f;
  if (i < S.sq) {
    const int64_t o_off = int64_t(S.bc) * p.o_bs + int64_t(S.q_row0 + i) * p.o_rs + int64_t(h) * p.o_hs;
    const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(p.out) + o_off;
    const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(p.dout) + o_off;
    for (int c = sub * 8; c < dv; c += 64) {
      const uint4 a = *reinterpret_cast<const uint4*>(o + c), d = *reinterpret_cast<const uint4*>(g + c);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(bf16lo_to_f32(aw[e]), bf16lo_to_f32(dw[e]), acc);
        acc = fmaf(bf16hi_to_f32(aw[e]), bf16hi_to_f32(dw[e]), acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (sub == 0) {
    float l2 = INFINITY;   // P = exp2(... - inf) = 0 (padding rows, rows without keys)
    if (i < S.sq) {
      const int64_t li = p.cu_seqlens_q != nullptr ? int64_t(h) * p.total_q + S.q_row0 + i
                                                   : (int64_t(b) * p.hq + h) * p.seqlen_q + i;
      const float lse = p.lse[li];
      if (lse != -INFINITY) l2 = lse * 1.4426950408889634f;
    }
    const int64_t w = ws_row0(p, b, h) + i;
    p.lse2[w] = l2;
    p.dsum[w] = acc;
  }
}

// ---------------------------------------------------------------------------
template <int DK, int DV, bool TAIL>
__global__ void __launch_bounds__(BwdCfg<DK, DV>::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                  const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapDO,
                  const BwdParams p) {
  using Cfg = BwdCfg<DK, DV>;
  static_assert(256 + DK <= 512, "tensor memory budget");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the array itself so that accesses
  // through it stay shared-memory accesses with 32-bit addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const BBars B = carve<Cfg>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_BAR + Cfg::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Batched: x = (sequence, q head), y = query tile, longest tiles first. Packed
  // varlen (tiles_fast): x = query tile, so the CTAs of neighbouring tiles of one
  // head, which read the same K/V blocks, run together and share them in L2.
  const int bx = p.tiles_fast ? blockIdx.y : blockIdx.x, by = p.tiles_fast ? blockIdx.x : blockIdx.y;
  const int ny = p.tiles_fast ? static_cast<int>(gridDim.x) : static_cast<int>(gridDim.y);
  const int b = bx / p.hq, h = bx % p.hq, g = h / p.r;
  const int mb = ny - 1 - by;   // longest tiles first
  const BSeq S = bwd_seq(p, b);
  if (mb * kB >= S.sq) return;   // a tile past this sequence's end (whole CTA, before any barrier)
  const int off = S.sk - S.sq;
  const int i0 = mb * kB, ilast = min(i0 + kB - 1, S.sq - 1);
  int klo = 0, khi = S.sk;
  if (p.wl >= 0) klo = max(klo, i0 + off - p.wl);
  if (p.wr >= 0) khi = min(khi, ilast + off + p.wr + 1);
  const int nlo = klo / kB, nhi = (khi > klo) ? (khi + kB - 1) / kB : nlo;
  const bool has = nhi > nlo;

  if (threadIdx.x == 0) {
    init_bars<Cfg>(B);
    *abort_flag = 0;
  }
  if (warp == Cfg::MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitGuard guard{abort_flag, p.status, p.timeout_ns};

  if (warp == Cfg::TMA_WARP) {
    // Lane 0 issues the copies. With seqused_k (TAIL), the whole warp clears
    // the rows of the last, partly used key block from the used length up to
    // the next 16-key step in shared memory: cache rows past seqused_k may
    // hold anything (NaN), and dQ += dS K contracts over them up to that step
    // (dS is 0 there, but 0 * NaN is not).
    if (has) {
      if (lane == 0) {
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapK);
        tma_prefetch_desc(&mapV);
        tma_prefetch_desc(&mapDO);
        uint8_t* res = smem + Cfg::OFF_RES;
        mbar_arrive_expect_tx(B.res_full, Cfg::PAIR);
#pragma unroll
        for (int c = 0; c < (Cfg::CQ > Cfg::CV ? Cfg::CQ : Cfg::CV); ++c) {
          if (c < Cfg::CQ) tma_load_4d(res + c * kChunk, &mapQ, B.res_full, c * 64, S.q_row0 + i0, h, S.bc);
          if (c < Cfg::CV)
            tma_load_4d(res + Cfg::TQ + c * kChunk, &mapDO, B.res_full, c * 64, S.q_row0 + i0, h, S.bc);
        }
      }
      constexpr unsigned wmask = TAIL ? 0xffffffffu : 1u;
      uint32_t u = 0, nka = 0, nbl = 0;   // blocks walked, K (ring) and V (SPLIT) copies issued by lane 0
      if (lane == 0 || TAIL) {
        for (int n = nhi - 1; n >= nlo; --n, ++u) {
          const int st = u % Cfg::ST;
          uint8_t* dst = smem + Cfg::OFF_STR + st * Cfg::A_BYTES;
          bool w = true;
          if (lane == 0) {
            w = u < Cfg::ST || mbar_wait(&B.str_empty[st], ((u - Cfg::ST) / Cfg::ST) & 1, guard);
            if (w) {
              mbar_arrive_expect_tx(&B.str_full[st], Cfg::A_BYTES);
#pragma unroll
              for (int c = 0; c < (Cfg::CQ > Cfg::CV ? Cfg::CQ : Cfg::CV); ++c) {
                if (c < Cfg::CQ)
                  tma_load_4d(dst + c * kChunk, &mapK, &B.str_full[st], c * 64, S.k_row0 + n * kB, g, S.bc);
                if (!Cfg::SPLIT && c < Cfg::CV)
                  tma_load_4d(dst + Cfg::TQ + c * kChunk, &mapV, &B.str_full[st], c * 64, S.k_row0 + n * kB, g,
                              S.bc);
              }
            }
            if (w) ++nka;
            // V(u) into its own slot (in two halves with BHALF), each load once dP
            // has read the previous one
            for (int hp = 0; Cfg::SPLIT && w && hp < Cfg::B_PARTS; ++hp) {
              const uint32_t idx = u * Cfg::B_PARTS + hp;
              w = idx == 0 || mbar_wait(B.b_empty, (idx - 1) & 1, guard);
              if (w) {
                constexpr int CP = Cfg::CV / Cfg::B_PARTS;
                uint8_t* vdst = smem + Cfg::OFF_B;
                mbar_arrive_expect_tx(B.b_full, Cfg::B_BYTES);
#pragma unroll
                for (int c = 0; c < CP; ++c)
                  tma_load_4d(vdst + c * kChunk, &mapV, B.b_full, (hp * CP + c) * 64, S.k_row0 + n * kB, g, S.bc);
                ++nbl;
              }
            }
          }
          if (!__shfl_sync(wmask, w ? 1 : 0, 0)) break;
          const int valid = S.sk - n * kB;
          if (TAIL && valid < kB) {
            if (!__all_sync(wmask, mbar_wait(&B.str_full[st], (u / Cfg::ST) & 1, guard))) break;
            const int pieces = (min(kB, (valid + 15) & ~15) - valid) * Cfg::CQ * 8;   // 16-byte pieces of K
            for (int idx = lane; idx < pieces; idx += 32) {
              const int row = valid + idx / (Cfg::CQ * 8), rem = idx % (Cfg::CQ * 8);
              *reinterpret_cast<uint4*>(dst + (rem >> 3) * kChunk + row * 128 + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp(wmask);
            if (lane == 0) mbar_arrive(B.k_fixed);
          }
        }
      }
      // drain the copies still in flight (only after an abort can any be):
      // nka stages of the ring and nbl B-tile copies were issued
      if (lane == 0) {
        for (uint32_t x = (nka > (uint32_t)Cfg::ST ? nka - Cfg::ST : 0); x < nka; ++x)
          drain_phase(&B.str_full[x % Cfg::ST], (x / Cfg::ST) & 1, p.timeout_ns);
        if (Cfg::SPLIT && nbl > 0) drain_phase(B.b_full, (nbl - 1) & 1, p.timeout_ns);
        drain_phase(B.res_full, 0, p.timeout_ns);
      }
    }
  } else if (warp == Cfg::MMA_WARP) {
    if (lane == 0 && has) {
      // Issue order, block u:  S(0) dP(0) | [S(u) read] S(u+1) [dS(u)] dQ(u) dP(u+1) | ...
      // so that dP(u) runs while the warps form P(u), S(u+1) while they form
      // dS(u), and dQ(u) and dP(u+1) while they form P(u+1). dS(u) lives in
      // dP's columns, which dP(u+1) only overwrites after dQ(u) has read them
      // (the tensor pipe runs one thread's MMAs in order). With SPLIT rings,
      // V(u+1) loads once dP(u) has completed, well before dP(u+1) is issued.
      // With one stage of K, S(u+1) needs K(u+1), which loads only once dQ(u)
      // has released the stage: ... [dS(u)] dQ(u) | S(u+1) dP(u+1).
      constexpr uint32_t IDESC_S = idesc_bf16_f32(kB, kB, false, false);
      constexpr uint32_t IDESC_DQ = idesc_bf16_f32(kB, DK, false, true);
      const uint32_t q_base = smem_u32(smem + Cfg::OFF_RES), do_base = q_base + Cfg::TQ;
      const uint32_t nb = static_cast<uint32_t>(nhi - nlo);
      auto kv = [&](uint32_t u) { return smem_u32(smem + Cfg::OFF_STR + (u % Cfg::ST) * Cfg::A_BYTES); };
      auto vt = [&](uint32_t u) { return Cfg::SPLIT ? smem_u32(smem + Cfg::OFF_B) : kv(u) + Cfg::TQ; };
      // dP(u) = dO V(u)^T; with SPLIT each part of V (both halves of the
      // contraction with BHALF) after its load landed, released by a commit after it
      auto issue_dp = [&](uint32_t u) -> bool {
        constexpr int KP = DV / 16 / Cfg::B_PARTS;   // 16-deep steps per part
        for (int hp = 0; hp < Cfg::B_PARTS; ++hp) {
          if (Cfg::SPLIT) {
            if (!mbar_wait(B.b_full, (u * Cfg::B_PARTS + hp) & 1, guard)) return false;
            tc_fence_after();
          }
          issue_ss_part(tmem + 128, do_base, vt(u), hp * KP, (hp + 1) * KP, hp * (Cfg::CV / Cfg::B_PARTS), IDESC_S);
          if (Cfg::SPLIT) mma_commit(B.b_empty);
        }
        mma_commit(B.dp_full);
        return true;
      };
      bool ok = mbar_wait(B.res_full, 0, guard) && mbar_wait(&B.str_full[0], 0, guard);
      if (ok) {
        issue_ss(tmem, q_base, kv(0), DK, IDESC_S);                         // S  = Q K^T
        mma_commit(B.s_full);
        ok = issue_dp(0);                                                   // dP = dO V^T
      }
      for (uint32_t u = 0; ok && u < nb; ++u) {
        if (!mbar_wait(&B.p_done[0], u & 1, guard) || !mbar_wait(&B.p_done[1], u & 1, guard)) { ok = false; break; }
        if (Cfg::ST > 1 && u + 1 < nb) {
          if (!mbar_wait(&B.str_full[(u + 1) % Cfg::ST], ((u + 1) / Cfg::ST) & 1, guard)) { ok = false; break; }
          tc_fence_after();
          issue_ss(tmem, q_base, kv(u + 1), DK, IDESC_S);
          mma_commit(B.s_full);
        }
        // the last, partly used key block (seqused_k): K cleared up to the next
        // 16-key step, and the contraction stops there
        const int valid = S.sk - (nhi - 1 - static_cast<int>(u)) * kB;
        const bool tail = TAIL && valid < kB;
        if (tail && !mbar_wait(B.k_fixed, 0, guard)) { ok = false; break; }
        const int steps = tail ? (valid + 15) / 16 : 8;
        for (int c = 0; c < 2; ++c) {
          if (!mbar_wait(&B.ds_full[c], u & 1, guard)) { ok = false; break; }
          tc_fence_after();
          if (!tail)
            issue_ts_half(tmem + 256, tmem + 128, kv(u), c, IDESC_DQ, u > 0 || c > 0);   // dQ += dS_c K_c
          else
            issue_ts_half_steps(tmem + 256, tmem + 128, kv(u), c, IDESC_DQ, u > 0 || (c > 0 && steps > 0),
                                min(4, max(0, steps - 4 * c)));
        }
        if (!ok) break;
        mma_commit(&B.str_empty[u % Cfg::ST]);
        if (Cfg::ST == 1 && u + 1 < nb) {
          if (!mbar_wait(&B.str_full[0], (u + 1) & 1, guard)) { ok = false; break; }
          tc_fence_after();
          issue_ss(tmem, q_base, kv(u + 1), DK, IDESC_S);
          mma_commit(B.s_full);
        }
        if (u + 1 < nb && !issue_dp(u + 1)) { ok = false; break; }
      }
      if (ok) mma_commit(B.acc_full);
      mma_commit(B.drain);
      drain_phase(B.drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ====== compute warps: warpgroup c takes key columns [64c, 64c+64) of every
    // block; thread t of a warpgroup owns query row i0 + t (tensor-memory lane t)
    const int c = warp >> 2;
    const int t = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int i = i0 + t;
    const int64_t vrow = ws_row0(p, b, h) + i;   // inside the sequence's 128-row padded region
    __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq) + int64_t(S.bc) * p.q_bs +
                        int64_t(S.q_row0 + i) * p.q_rs + int64_t(h) * p.q_hs + c * (DK / 2);
    if (has) {
      const float nl2 = -p.lse2[vrow], dsum = p.dsum[vrow];
      bool ok = true;
      uint32_t u = 0;
      for (int n = nhi - 1; n >= nlo; --n, ++u) {
        const int jb = n * kB;
        // every (row, key) of the block visible?  (uniform over the CTA)
        const bool full = (jb + kB <= S.sk) && (p.wr < 0 || jb + kB - 1 <= i0 + off + p.wr) &&
                          (p.wl < 0 || jb >= i0 + kB - 1 + off - p.wl);
        // visible columns [c_lo, c_hi] of this row, relative to this warpgroup's first column
        const int c_lo = ((p.wl >= 0) ? i + off - p.wl - jb : INT32_MIN / 2) - 64 * c;
        int c_hi = S.sk - 1 - jb;
        if (p.wr >= 0) c_hi = min(c_hi, i + off + p.wr - jb);
        c_hi -= 64 * c;
        // P = exp2(S scale log2(e) - LSE log2(e)), masked
        if (!mbar_wait(B.s_full, u & 1, guard)) { ok = false; break; }
        tc_fence_after();
        float pf[64];
        // one instance for blocks every key of which this tile sees, one with the
        // mask (column e visible when (unsigned)(e - c_lo) <= (unsigned)(c_hi - c_lo))
        auto p_phase = [&](auto masked) {
          uint32_t sv[64];
          tmem_ld64(tmem + lane_off + 64 * c, sv);
          const int lo_e = (c_hi < c_lo) ? 256 : c_lo;
          const uint32_t width = (c_hi < c_lo) ? 0u : static_cast<uint32_t>(c_hi - c_lo);
          const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nl22 = make_float2(nl2, nl2);
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nl22);
            const float x0 = ex2_approx(x2.x), x1 = ex2_approx(x2.y);
            if constexpr (decltype(masked)::value) {
              pf[e] = (static_cast<uint32_t>(e - lo_e) <= width) ? x0 : 0.f;
              pf[e + 1] = (static_cast<uint32_t>(e + 1 - lo_e) <= width) ? x1 : 0.f;
            } else {
              pf[e] = x0;
              pf[e + 1] = x1;
            }
          }
        };
        if (full)
          p_phase(std::false_type{});
        else
          p_phase(std::true_type{});
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.p_done[c]);
        // dS = P (dP - D), bf16, into the first 32 columns of this half of dP
        if (!mbar_wait(B.dp_full, u & 1, guard)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t dp[64], w[32];
          tmem_ld64(tmem + lane_off + 128 + 64 * c, dp);
#pragma unroll
          const float2 nd2 = make_float2(-dsum, -dsum);
          for (int e = 0; e < 64; e += 2) {
            const float2 d2 = __fmul2_rn(make_float2(pf[e], pf[e + 1]),
                                         __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2));
            float d0 = d2.x, d1 = d2.y;
            if (TAIL) {   // dP of keys past seqused_k may be NaN (their V rows are not data)
              d0 = pf[e] != 0.f ? d0 : 0.f;
              d1 = pf[e + 1] != 0.f ? d1 : 0.f;
            }
            w[e >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st32(tmem + lane_off + 128 + 64 * c, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.ds_full[c]);
      }
      if (ok && mbar_wait(B.acc_full, 0, guard)) {
        tc_fence_after();
        // warpgroup c writes dQ columns [c DK/2, (c+1) DK/2)
#pragma unroll 1
        for (int k = 0; k < DK / 64; ++k) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + 256 + c * (DK / 2) + k * 32, o);
          if (i < S.sq) store_row32(dq + k * 32, o, p.scale);
        }
      }
    } else if (i < S.sq) {
      zero_row(dq, DK / 2);   // no visible key: dQ = 0
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// One CTA of the dK/dV kernel (pass MODE); (xi, yi) is its grid position.
template <int DK, int DV, bool TAIL, int MODE>
__device__ __forceinline__ void dkdv_body(const CUtensorMap& mapQ, const CUtensorMap& mapK, const CUtensorMap& mapV,
                                          const CUtensorMap& mapDO, const BwdParams& p, int xi, int yi) {
  using Cfg = BwdCfg<DK, DV, MODE>;
  static_assert(256 + (MODE == kBoth ? DK + DV : MODE == kDvOnly ? DV : DK) <= 512, "tensor memory budget");
  constexpr bool kDv = MODE != kDkOnly, kDk = MODE != kDvOnly;   // accumulators of this pass
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the array itself so that accesses
  // through it stay shared-memory accesses with 32-bit addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const BBars B = carve<Cfg>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_BAR + Cfg::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Batched: x = (sequence, KV head), y = key block, low key blocks first (under a
  // causal mask they see the most query tiles). Packed varlen (tiles_fast): x =
  // key block, so neighbouring blocks of one KV head, which read the same Q and
  // dO tiles, run together and share them in L2.
  const int bx = p.tiles_fast ? yi : xi;
  const int b = bx / p.hkv, g = bx % p.hkv;
  const int n = p.tiles_fast ? xi : yi;
  const BSeq S = bwd_seq(p, b);
  if (n * kB >= S.sk) {   // a block past this sequence's keys (whole CTA, before any barrier)
    if (TAIL) {   // cache rows past seqused_k: dK = dV = 0 (this pass's accumulators)
      for (int idx = threadIdx.x; idx < 2 * kB; idx += blockDim.x) {
        const int j = n * kB + (idx >> 1);
        const bool is_k = idx & 1;
        if (j >= S.ska || (is_k ? !kDk : !kDv)) continue;
        __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(is_k ? p.dk : p.dv) +
                             int64_t(S.bc) * (is_k ? p.k_bs : p.v_bs) +
                             int64_t(S.k_row0 + j) * (is_k ? p.k_rs : p.v_rs) + int64_t(g) * (is_k ? p.k_hs : p.v_hs);
        zero_row(row, is_k ? DK : DV);
      }
    }
    return;
  }
  const int off = S.sk - S.sq;
  const int j0 = n * kB, jlast = min(j0 + kB - 1, S.sk - 1);
  // query rows that see some key of the block
  int ilo = 0, ihi = S.sq - 1;
  if (p.wr >= 0) ilo = max(ilo, j0 - off - p.wr);
  if (p.wl >= 0) ihi = min(ihi, jlast - off + p.wl);
  const int mlo = ilo / kB, nm = (ihi >= ilo) ? ihi / kB + 1 - mlo : 0;
  const int jobs = nm * p.r;   // (q head of the group, query tile) pairs, head-major

  if (threadIdx.x == 0) {
    init_bars<Cfg>(B);
    *abort_flag = 0;
  }
  if (warp == Cfg::MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitGuard guard{abort_flag, p.status, p.timeout_ns};

  if (warp == Cfg::TMA_WARP) {
    if (lane == 0 && jobs > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapDO);
      uint8_t* res = smem + Cfg::OFF_RES;
      mbar_arrive_expect_tx(B.res_full, Cfg::RES);
#pragma unroll
      for (int c = 0; c < (Cfg::CQ > Cfg::CV ? Cfg::CQ : Cfg::CV); ++c) {
        if (c < Cfg::CQ) tma_load_4d(res + c * kChunk, &mapK, B.res_full, c * 64, S.k_row0 + j0, g, S.bc);
        if (kDk && c < Cfg::CV)   // V feeds dP^T only
          tma_load_4d(res + Cfg::TQ + c * kChunk, &mapV, B.res_full, c * 64, S.k_row0 + j0, g, S.bc);
      }
      uint32_t u = 0, nbl = 0;
      for (; u < static_cast<uint32_t>(jobs); ++u) {
        const int st = u % Cfg::ST;
        const int hh = g * p.r + static_cast<int>(u) / nm, m = mlo + static_cast<int>(u) % nm;
        if (u >= Cfg::ST && !mbar_wait(&B.str_empty[st], ((u - Cfg::ST) / Cfg::ST) & 1, guard)) break;
        uint8_t* dst = smem + Cfg::OFF_STR + st * Cfg::A_BYTES;
        float* vec = reinterpret_cast<float*>(smem + Cfg::OFF_VEC + st * 1024);
        const int64_t vrow = ws_row0(p, b, hh) + m * kB;
        mbar_arrive_expect_tx(&B.str_full[st], Cfg::A_BYTES + 1024);
#pragma unroll
        for (int c = 0; c < (Cfg::CQ > Cfg::CV ? Cfg::CQ : Cfg::CV); ++c) {
          if (c < Cfg::CQ)
            tma_load_4d(dst + c * kChunk, &mapQ, &B.str_full[st], c * 64, S.q_row0 + m * kB, hh, S.bc);
          if (!Cfg::SPLIT && c < Cfg::CV)
            tma_load_4d(dst + Cfg::TQ + c * kChunk, &mapDO, &B.str_full[st], c * 64, S.q_row0 + m * kB, hh, S.bc);
        }
        bulk_load(vec, p.lse2 + vrow, 512, &B.str_full[st]);
        bulk_load(vec + 128, p.dsum + vrow, 512, &B.str_full[st]);
        // dO(u) into its own slot (in two halves with BHALF), each load once
        // dP^T has read the previous one
        bool bw = true;
        for (int hp = 0; Cfg::SPLIT && hp < Cfg::B_PARTS; ++hp) {
          const uint32_t idx = u * Cfg::B_PARTS + hp;
          if (idx > 0 && !mbar_wait(B.b_empty, (idx - 1) & 1, guard)) { bw = false; break; }
          constexpr int CP = Cfg::CV / Cfg::B_PARTS;
          uint8_t* ddst = smem + Cfg::OFF_B;
          mbar_arrive_expect_tx(B.b_full, Cfg::B_BYTES);
#pragma unroll
          for (int c = 0; c < CP; ++c)
            tma_load_4d(ddst + c * kChunk, &mapDO, B.b_full, (hp * CP + c) * 64, S.q_row0 + m * kB, hh, S.bc);
          ++nbl;
        }
        if (!bw) { ++u; break; }
      }
      // drain the copies still in flight (only after an abort can any be): u
      // stages of the ring and nbl B-tile copies were issued
      for (uint32_t x = (u > (uint32_t)Cfg::ST ? u - Cfg::ST : 0); x < u; ++x)
        drain_phase(&B.str_full[x % Cfg::ST], (x / Cfg::ST) & 1, p.timeout_ns);
      if (Cfg::SPLIT && nbl > 0) drain_phase(B.b_full, (nbl - 1) & 1, p.timeout_ns);
      drain_phase(B.res_full, 0, p.timeout_ns);
    }
  } else if (warp == Cfg::MMA_WARP) {
    if (lane == 0 && jobs > 0) {
      // Issue order, job u:  S(0) dP(0) | [P(u)] dV(u) S(u+1) [dS(u)] dK(u) dP(u+1) | ...
      // so that dP(u) runs while the warps form P(u), dV(u) and S(u+1) while
      // they form dS(u), and dK(u) and dP(u+1) while they form P(u+1). P^T(u)
      // and dS^T(u) live in S's and dP's columns, which S(u+1) and dP(u+1) only
      // overwrite after dV(u) and dK(u) have read them (one thread's MMAs run
      // in order). The dV-only pass drops dP and dK, the dK-only pass dV (its
      // S(u+1) then waits only for the warps to have read S(u)). With SPLIT
      // rings, dO(u+1) loads once dP(u) has completed, before dP(u+1) is issued.
      // With one stage, S(u+1) needs Q(u+1), which loads only once the job's
      // last GEMM has released the stage: ... dK(u) | S(u+1) dP(u+1).
      constexpr uint32_t IDESC_S = idesc_bf16_f32(kB, kB, false, false);
      constexpr uint32_t IDESC_DV = idesc_bf16_f32(kB, DV, false, true);
      constexpr uint32_t IDESC_DK = idesc_bf16_f32(kB, DK, false, true);
      constexpr uint32_t DV_COL = 256, DK_COL = (MODE == kBoth) ? 256 + DV : 256;
      const uint32_t k_base = smem_u32(smem + Cfg::OFF_RES), v_base = k_base + Cfg::TQ;
      const uint32_t nj = static_cast<uint32_t>(jobs);
      auto qs = [&](uint32_t u) { return smem_u32(smem + Cfg::OFF_STR + (u % Cfg::ST) * Cfg::A_BYTES); };
      auto dot = [&](uint32_t u) { return Cfg::SPLIT ? smem_u32(smem + Cfg::OFF_B) : qs(u) + Cfg::TQ; };
      // dP^T(u) = V dO(u)^T; with SPLIT each part of dO (both halves of the
      // contraction with BHALF) after its load landed, released by a commit after it
      auto issue_dp = [&](uint32_t u) -> bool {
        constexpr int KP = DV / 16 / Cfg::B_PARTS;   // 16-deep steps per part
        for (int hp = 0; hp < Cfg::B_PARTS; ++hp) {
          if (Cfg::SPLIT) {
            if (!mbar_wait(B.b_full, (u * Cfg::B_PARTS + hp) & 1, guard)) return false;
            tc_fence_after();
          }
          issue_ss_part(tmem + 128, v_base, dot(u), hp * KP, (hp + 1) * KP, hp * (Cfg::CV / Cfg::B_PARTS), IDESC_S);
          if (Cfg::SPLIT) mma_commit(B.b_empty);
        }
        mma_commit(B.dp_full);
        return true;
      };
      bool ok = mbar_wait(B.res_full, 0, guard) && mbar_wait(&B.str_full[0], 0, guard);
      if (ok) {
        issue_ss(tmem, k_base, qs(0), DK, IDESC_S);                          // S^T  = K Q^T
        mma_commit(B.s_full);
        if constexpr (kDk) ok = issue_dp(0);                                 // dP^T = V dO^T
      }
      for (uint32_t u = 0; ok && u < nj; ++u) {
        const uint32_t qb = qs(u), dob = dot(u);
        const bool acc = u > 0;
        for (int c = 0; c < 2; ++c) {
          if (!mbar_wait(&B.p_done[c], u & 1, guard)) { ok = false; break; }
          if constexpr (kDv) {
            tc_fence_after();
            issue_ts_half(tmem + DV_COL, tmem, dob, c, IDESC_DV, acc || c > 0);   // dV += P^T_c dO_c
          }
        }
        if (!ok) break;
        if (Cfg::ST > 1 && u + 1 < nj) {
          if (!mbar_wait(&B.str_full[(u + 1) % Cfg::ST], ((u + 1) / Cfg::ST) & 1, guard)) { ok = false; break; }
          issue_ss(tmem, k_base, qs(u + 1), DK, IDESC_S);
          mma_commit(B.s_full);
        }
        if constexpr (kDk) {
          for (int c = 0; c < 2; ++c) {
            if (!mbar_wait(&B.ds_full[c], u & 1, guard)) { ok = false; break; }
            tc_fence_after();
            issue_ts_half(tmem + DK_COL, tmem + 128, qb, c, IDESC_DK, acc || c > 0);   // dK += dS^T_c Q_c
          }
          if (!ok) break;
        }
        mma_commit(&B.str_empty[u % Cfg::ST]);
        if (Cfg::ST == 1 && u + 1 < nj) {
          if (!mbar_wait(&B.str_full[0], (u + 1) & 1, guard)) { ok = false; break; }
          tc_fence_after();
          issue_ss(tmem, k_base, qs(u + 1), DK, IDESC_S);
          mma_commit(B.s_full);
        }
        if constexpr (kDk) {
          if (u + 1 < nj && !issue_dp(u + 1)) { ok = false; break; }
        }
      }
      if (ok) mma_commit(B.acc_full);
      mma_commit(B.drain);
      drain_phase(B.drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ====== compute warps: warpgroup c takes query columns [64c, 64c+64) of
    // every job; thread t of a warpgroup owns key row j0 + t (tensor-memory lane t)
    const int c = warp >> 2;
    const int t = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int j = j0 + t;
    __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(p.dk) + int64_t(S.bc) * p.k_bs +
                        int64_t(S.k_row0 + j) * p.k_rs + int64_t(g) * p.k_hs;
    __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(p.dv) + int64_t(S.bc) * p.v_bs +
                        int64_t(S.k_row0 + j) * p.v_rs + int64_t(g) * p.v_hs;
    // the accumulator columns this warpgroup writes: with both, warpgroup 0 all
    // of dV and warpgroup 1 all of dK (times the softmax scale); in a one-
    // accumulator pass, warpgroup c its half [c n/2, (c+1) n/2)
    constexpr int kOut = (MODE == kDkOnly) ? DK : DV;
    auto out_cols = [&]() { return (MODE == kBoth) ? (c == 0 ? DV : DK) : kOut / 2; };
    auto out_row = [&]() {
      const bool wdk = (MODE == kBoth) ? c == 1 : MODE == kDkOnly;
      return (wdk ? dk : dv) + ((MODE == kBoth) ? 0 : c * (kOut / 2));
    };
    if (jobs > 0) {
      bool ok = true;
      for (uint32_t u = 0; u < static_cast<uint32_t>(jobs); ++u) {
        const int st = u % Cfg::ST;
        const int m = mlo + static_cast<int>(u) % nm;
        const int ib = m * kB;
        const bool full = (j0 + kB <= S.sk) && (ib + kB <= S.sq) &&
                          (p.wr < 0 || j0 + kB - 1 <= ib + off + p.wr) && (p.wl < 0 || j0 >= ib + kB - 1 + off - p.wl);
        // visible query columns [c_lo, c_hi] of this key row, relative to this warpgroup's first column
        const int c_lo = ((p.wr >= 0) ? j - off - p.wr - ib : INT32_MIN / 2) - 64 * c;
        int c_hi = S.sq - 1 - ib;
        if (p.wl >= 0) c_hi = min(c_hi, j - off + p.wl - ib);
        if (j >= S.sk) c_hi = -1 + 64 * c;
        c_hi -= 64 * c;
        // the stage's lse2 / D landed with its tiles
        if (!mbar_wait(&B.str_full[st], (u / Cfg::ST) & 1, guard)) { ok = false; break; }
        const float* vl = reinterpret_cast<const float*>(smem + Cfg::OFF_VEC + st * 1024) + 64 * c;
        const float* vd = vl + 128;
        // P^T = exp2(S^T scale log2(e) - LSE log2(e)), masked; bf16 into the half's first 32 columns
        if (!mbar_wait(B.s_full, u & 1, guard)) { ok = false; break; }
        tc_fence_after();
        float pf[64];
        // one instance for jobs every (key, query) pair of which is visible, one
        // with the mask (column e visible when (unsigned)(e - c_lo) <= (unsigned)(c_hi - c_lo))
        auto p_phase = [&](auto masked) {
          uint32_t sv[64], pw[32];
          tmem_ld64(tmem + lane_off + 64 * c, sv);
          const int lo_e = (c_hi < c_lo) ? 256 : c_lo;
          const uint32_t width = (c_hi < c_lo) ? 0u : static_cast<uint32_t>(c_hi - c_lo);
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(vl + e);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int q = 0; q < 4; q += 2) {
              const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(sv[e + q]), __uint_as_float(sv[e + q + 1])),
                                           make_float2(p.scale_log2, p.scale_log2), make_float2(-lv[q], -lv[q + 1]));
              const float x0 = ex2_approx(x2.x), x1 = ex2_approx(x2.y);
              if constexpr (decltype(masked)::value) {
                pf[e + q] = (static_cast<uint32_t>(e + q - lo_e) <= width) ? x0 : 0.f;
                pf[e + q + 1] = (static_cast<uint32_t>(e + q + 1 - lo_e) <= width) ? x1 : 0.f;
              } else {
                pf[e + q] = x0;
                pf[e + q + 1] = x1;
              }
            }
            pw[e >> 1] = pack_bf16x2(pf[e], pf[e + 1]);
            pw[(e >> 1) + 1] = pack_bf16x2(pf[e + 2], pf[e + 3]);
          }
          if constexpr (kDv) tmem_st32(tmem + lane_off + 64 * c, pw);   // P^T feeds dV only
        };
        if (full)
          p_phase(std::false_type{});
        else
          p_phase(std::true_type{});
        if constexpr (kDv) tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.p_done[c]);
        if constexpr (!kDk) continue;
        // dS^T = P^T (dP^T - D), bf16 into the first 32 columns of this half of dP^T
        if (!mbar_wait(B.dp_full, u & 1, guard)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t dp[64], dw[32];
          tmem_ld64(tmem + lane_off + 128 + 64 * c, dp);
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(vd + e);
            const float2 a2 = __fmul2_rn(make_float2(pf[e], pf[e + 1]),
                                         __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                                    make_float2(-d4.x, -d4.y)));
            const float2 b2 = __fmul2_rn(make_float2(pf[e + 2], pf[e + 3]),
                                         __fadd2_rn(make_float2(__uint_as_float(dp[e + 2]), __uint_as_float(dp[e + 3])),
                                                    make_float2(-d4.z, -d4.w)));
            dw[e >> 1] = pack_bf16x2(a2.x, a2.y);
            dw[(e >> 1) + 1] = pack_bf16x2(b2.x, b2.y);
          }
          tmem_st32(tmem + lane_off + 128 + 64 * c, dw);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.ds_full[c]);
      }
      if (ok && mbar_wait(B.acc_full, 0, guard)) {
        tc_fence_after();
        const bool wdk = (MODE == kBoth) ? c == 1 : MODE == kDkOnly;
        const int ocols = out_cols();
        const uint32_t ocol = (MODE == kBoth) ? 256 + c * DV : 256 + c * (kOut / 2);
        __nv_bfloat16* dst = out_row();
        const float f = wdk ? p.scale : 1.f;
#pragma unroll 1
        for (int k = 0; k < ocols / 32; ++k) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + ocol + k * 32, o);
          if (j < S.sk) store_row32(dst + k * 32, o, f);
        }
        if (TAIL && j >= S.sk && j < S.ska) zero_row(dst, ocols);   // cache rows past seqused_k
      }
    } else if (j < (TAIL ? S.ska : S.sk)) {
      zero_row(out_row(), out_cols());   // no query sees these keys (or they are past seqused_k)
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DK, int DV, bool TAIL, int MODE>
__global__ void __launch_bounds__(BwdCfg<DK, DV, MODE>::THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                    const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapDO,
                    const BwdParams p) {
  dkdv_body<DK, DV, TAIL, MODE>(mapQ, mapK, mapV, mapDO, p, blockIdx.x, blockIdx.y);
}

// Both passes of the two-pass head dims in one grid: the even CTAs in x run
// the dV pass and the odd ones the dK pass of the same (KV head, key block),
// so that each pass's long causal CTAs share the SMs with the other's instead
// of running after them.
template <int DK, int DV, bool TAIL>
__global__ void __launch_bounds__(BwdCfg<DK, DV, kDkOnly>::THREADS, 1)
    bwd_dkdv2_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                     const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapDO,
                     const BwdParams p) {
  static_assert(BwdCfg<DK, DV, kDvOnly>::THREADS == BwdCfg<DK, DV, kDkOnly>::THREADS, "one block shape");
  const int xi = static_cast<int>(blockIdx.x >> 1), yi = static_cast<int>(blockIdx.y);
  if (blockIdx.x & 1)
    dkdv_body<DK, DV, TAIL, kDkOnly>(mapQ, mapK, mapV, mapDO, p, xi, yi);
  else
    dkdv_body<DK, DV, TAIL, kDvOnly>(mapQ, mapK, mapV, mapDO, p, xi, yi);
}

template <int DK, int DV, bool TAIL>
constexpr int kSmem2 = BwdCfg<DK, DV, kDvOnly>::SMEM > BwdCfg<DK, DV, kDkOnly>::SMEM ? BwdCfg<DK, DV, kDvOnly>::SMEM
                                                                                   : BwdCfg<DK, DV, kDkOnly>::SMEM;

template <int DK, int DV, bool TAIL, int MODE>
cudaError_t launch_dkdv(const BwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mdo, dim3 grid, cudaStream_t stream) {
  using Cfg = BwdCfg<DK, DV, MODE>;
  bwd_dkdv_kernel<DK, DV, TAIL, MODE><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mk, mv, mdo, p);
  return cudaGetLastError();
}

// dK and dV: one launch with both accumulators, or the dV-only and dK-only passes
template <int DK, int DV, bool TAIL>
constexpr bool kOnePass = 256 + DK + DV <= 512;

template <int DK, int DV, bool TAIL>
cudaError_t set_dkdv_smem() {   // (host calls kept ahead of the launches: they delay them otherwise)
  if constexpr (kOnePass<DK, DV, TAIL>) {
    return cudaFuncSetAttribute(bwd_dkdv_kernel<DK, DV, TAIL, kBoth>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                BwdCfg<DK, DV, kBoth>::SMEM);
  } else {
    return cudaFuncSetAttribute(bwd_dkdv2_kernel<DK, DV, TAIL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmem2<DK, DV, TAIL>);
  }
}

template <int DK, int DV, bool TAIL>
cudaError_t launch_dkdv_all(const BwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mdo, dim3 grid, cudaStream_t stream) {
  if constexpr (kOnePass<DK, DV, TAIL>) {
    return launch_dkdv<DK, DV, TAIL, kBoth>(p, mq, mk, mv, mdo, grid, stream);
  } else {   // both passes in one grid, twice as wide in x
    bwd_dkdv2_kernel<DK, DV, TAIL><<<dim3(2 * grid.x, grid.y), BwdCfg<DK, DV, kDkOnly>::THREADS,
                                     kSmem2<DK, DV, TAIL>, stream>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError();
  }
}

template <int DK, int DV, bool TAIL>
cudaError_t launch_bwd_t(const BwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, cudaStream_t stream, const BwdSide& side) {
  using Cfg = BwdCfg<DK, DV>;
  // batched: every sequence's lengths; varlen: the longest (CTAs past a
  // shorter sequence's end return at once)
  const int mblocks = (p.seqlen_q + kB - 1) / kB, nblocks = (p.seqlen_k + kB - 1) / kB;
  if (mblocks > 0 && p.batch > 0) {
    bwd_preprocess_kernel<<<dim3(p.batch * mblocks, p.hq), 1024, 0, stream>>>(p, DV, mblocks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<DK, DV, TAIL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM);
  if (e != cudaSuccess) return e;
  if ((e = set_dkdv_smem<DK, DV, TAIL>()) != cudaSuccess) return e;
  const dim3 gq = p.tiles_fast ? dim3(mblocks, p.batch * p.hq) : dim3(p.batch * p.hq, mblocks);
  const dim3 gk = p.tiles_fast ? dim3(nblocks, p.batch * p.hkv) : dim3(p.batch * p.hkv, nblocks);
  if (mblocks > 0 && nblocks > 0 && side.stream != nullptr) {
    // The two kernels only share read-only inputs. dK/dV (few long CTAs under
    // a causal mask, longest first) goes on the caller's second stream, which
    // the caller gives a higher priority, so that its CTAs are placed first;
    // the many short dQ CTAs fill the SMs it leaves idle. The caller's events
    // fork the second stream from `stream` and join it back.
    if ((e = cudaEventRecord(side.fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(side.stream, side.fork, 0)) != cudaSuccess) return e;
    if ((e = launch_dkdv_all<DK, DV, TAIL>(p, mq, mk, mv, mdo, gk, side.stream)) != cudaSuccess) return e;
    bwd_dq_kernel<DK, DV, TAIL><<<gq, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaEventRecord(side.join, side.stream)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, side.join, 0);
  }
  if (nblocks > 0) {   // one stream: dK/dV, then dQ
    if ((e = launch_dkdv_all<DK, DV, TAIL>(p, mq, mk, mv, mdo, gk, stream)) != cudaSuccess) return e;
  }
  if (mblocks > 0) {
    bwd_dq_kernel<DK, DV, TAIL><<<gq, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

bool bwd_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 192 && dv == 128) || (dk == 256 && dv == 256);
}

cudaError_t launch_bwd(const BwdParams& p, int dk, int dv, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t stream, const BwdSide& side) {
  // the TAIL instances handle key caches with unused rows (seqused_k)
  const bool tail = p.seqused_k != nullptr;
  if (dk == 64 && dv == 64)
    return tail ? launch_bwd_t<64, 64, true>(p, mq, mk, mv, mdo, stream, side)
                : launch_bwd_t<64, 64, false>(p, mq, mk, mv, mdo, stream, side);
  if (dk == 128 && dv == 128)
    return tail ? launch_bwd_t<128, 128, true>(p, mq, mk, mv, mdo, stream, side)
                : launch_bwd_t<128, 128, false>(p, mq, mk, mv, mdo, stream, side);
  if (dk == 192 && dv == 128)
    return tail ? launch_bwd_t<192, 128, true>(p, mq, mk, mv, mdo, stream, side)
                : launch_bwd_t<192, 128, false>(p, mq, mk, mv, mdo, stream, side);
  if (dk == 256 && dv == 256)
    return tail ? launch_bwd_t<256, 256, true>(p, mq, mk, mv, mdo, stream, side)
                : launch_bwd_t<256, 256, false>(p, mq, mk, mv, mdo, stream, side);
  return cudaErrorInvalidValue;
}

}  // namespace fa
