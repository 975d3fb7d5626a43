// fa_prefill.cu - persistent, warp-specialised tcgen05 attention forward.
//
// The FlashAttention forward of "mslk/attention/flash_attn/interface.py"
// (`_flash_attn_fwd`, FlashAttentionForwardSm100: 128x128 tiles, q_stage 2,
// persistent when dense) re-designed here for sm_103a from the Blackwell idioms
// the backward page ("mslk/attention/flash_attn/flash_bwd_sm100.py") shows:
// TMA loads into 128B-swizzled shared memory, mbarrier pipelines, a single
// MMA-issuing thread, tcgen05 accumulators in tensor memory, the P operand of
// P.V read straight from tensor memory, and exp2 with the scale folded in.
//
// One CTA per SM loops over work tiles (m-block, q head, sequence); causal
// tiles come longest first. A tile is NQ x 128 query rows:
//   NQ = 2 (head dims 64, 128, 192/128): two 128-row Q tiles share each K/V
//     tile; softmax warpgroup s owns Q tile s, and the MMA warp ping-pongs
//       PV(n,0) S(n-1,0) PV(n,1) S(n-1,1) ...
//     so each softmax overlaps the other tile's GEMMs.
//     TMEM: S0 [0,128) S1 [128,256) O0 [256,256+DV) O1 [256+DV,256+2DV).
//   NQ = 1 (head dim 256): one Q tile, S double-buffered (slots alternate by
//     block), O in [256,512).
// P (bf16) overwrites the first 64 columns of its S slot. Key blocks run from
// the diagonal downwards so the masked blocks come first. The running max is
// rescaled lazily: O and l are only rescaled when the row max grows by more
// than 4 (base-2 units), the threshold of the FA4 notes on the sm_120 page.
//
// Warps: [0, 4*NSM) softmax (NSM = NQ warpgroups), then one MMA warp, one
// Q+K TMA warp and one V TMA warp. Every mbarrier wait is bounded; on a
// timeout the CTA raises a shared abort flag, records the failure in the
// device status word, drains its copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include <type_traits>

#include "fa_kernels.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;                 // query rows per Q tile
constexpr int kBN = 128;                 // keys per K/V block
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 bf16 (one swizzle-128B column chunk)
constexpr float kRescaleThreshold = 4.f;

template <int DK_, int DV_>
struct PrefillCfg {
  static constexpr int DK = DK_, DV = DV_;
  static constexpr int NQ = (DV <= 128) ? 2 : 1;
  static constexpr int NSM = NQ;                         // softmax warpgroups
  static constexpr int KST = (DK == 64) ? 3 : (DK == 192 || DK == 256) ? (DK == 256 ? 1 : 2) : 2;
  static constexpr int VST = (DK == 64) ? 3 : (DK == 192 || DK == 256) ? 1 : 2;
  static constexpr int KCH = DK / 64, VCH = DV / 64;
  static constexpr int Q_BYTES = KCH * kChunkBytes;
  static constexpr int K_BYTES = KCH * kChunkBytes;
  static constexpr int V_BYTES = VCH * kChunkBytes;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * K_BYTES;
  // O staging for coalesced TMA stores: two 32-column x 32-row buffers per
  // softmax warp (two-tile kernels with D <= 128, where shared memory has room)
  static constexpr bool OSTAGE = (NQ == 2) && (DK <= 128);
  static constexpr int OFF_OST = OFF_V + VST * V_BYTES;
  static constexpr int OST_BYTES = OSTAGE ? 2 * kChunkBytes : 0;
  static constexpr int OFF_BAR = OFF_OST + OST_BYTES;
  static constexpr int NBAR = 2 * 2 + 2 * KST + 3 * VST + 2 + 2 + 2 + 2 + 2 + 2 + 2;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  // at least half the SM's shared memory, so one CTA (the one that owns all
  // 512 TMEM columns) is resident per SM
  static constexpr int SMEM = (SMEM_USED + 1024 < 120 * 1024) ? 120 * 1024 : SMEM_USED + 1024;
  // warpgroups: NSM softmax warpgroups, then one holding the MMA warp, the two
  // TMA warps and one idle warp (whole warpgroups, for setmaxnreg)
  static constexpr int MMA_WARP = 4 * NSM;
  static constexpr int TMA_QK_WARP = MMA_WARP + 1;
  static constexpr int TMA_V_WARP = MMA_WARP + 2;
  static constexpr int PV_WARP = MMA_WARP + 3;   // NQ == 2: issues the P.V GEMMs
  static constexpr int THREADS = 32 * 4 * (NSM + 1);
  // register split (NQ == 2): 256 x 200 + 128 x 104 (or 256 x 192 + 128 x 120) = 384 x 168 at launch
  static constexpr int REG_SOFTMAX = (DK == 192) ? 192 : 200;
  static constexpr int REG_OTHER = (DK == 192) ? 120 : 104;
  static constexpr int ROWS_PER_TILE = NQ * kBM;
  static constexpr int O_COL = 256;
  static_assert(NQ == 2 ? (256 + 2 * DV <= 512) : (256 + DV <= 512), "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Pack-GQA ("interface.py", pack_gqa; the sm_120 PR page, Pack-GQA: the q heads
// sharing a KV head fold into the row axis): in the PACK instances tile row t of a
// sequence is query row t / r of q head g*r + t % r, so one tile reads each
// K/V block once for r heads. Otherwise tile rows are query rows of head h.
struct Tile {
  int b, h, g, mb;      // h: q head (unpacked) or the KV head (packed)
  int split;            // SPLIT instances: the key split this tile covers
  int q_row0, k_row0;   // first row of the sequence in q's / k's row axis
  int sq, sk;
  int rows;             // tile rows of the sequence: sq, or sq * r packed
};

struct Range {
  int r0;       // first tile row of this Q tile inside the sequence
  int i0, i1;   // first and last query row it covers
  bool active;  // the Q tile has rows
  int nlo, nhi; // key blocks [nlo, nhi) hold visible keys; empty when nhi <= nlo
};

// The k-th tile of this CTA in a persistent grid: tiles are sorted longest
// first, and the CTA order reverses every round ("snake"), so a CTA that got a
// long tile in one round gets a short one in the next.
__device__ __forceinline__ int tile_of(int k) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return k * g + ((k & 1) ? g - 1 - c : c);
}

template <int ROWS_PER_TILE, bool PACK, bool SPLIT>
__device__ __forceinline__ bool fetch_tile(const FwdParams& p, int t, Tile& T) {
  // SPLIT instances: consecutive work items are the key splits of one tile
  T.split = 0;
  if constexpr (SPLIT) {
    T.split = t % p.num_splits;
    t /= p.num_splits;
  }
  if (p.cu_seqlens_q == nullptr) {
    if (t >= p.num_tiles) return false;
    const int nh = PACK ? p.hkv : p.hq;
    const int per = nh * p.batch;
    const int mbi = t / per, rem = t - mbi * per;
    T.mb = p.m_blocks - 1 - mbi;   // longest-first for causal; a fixed order otherwise
    T.h = rem % nh;
    T.b = rem / nh;
    T.q_row0 = 0;
    T.k_row0 = 0;
    T.sq = p.seqlen_q;
    T.sk = p.seqused_k ? p.seqused_k[T.b] : p.seqlen_k;
  } else {
    const int total = p.tile_prefix[p.batch];
    if (t >= total) return false;
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.tile_prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    T.b = lo;
    const int local = t - p.tile_prefix[lo];
    const int nh = PACK ? p.hkv : p.hq;
    const int nmb = (p.tile_prefix[lo + 1] - p.tile_prefix[lo]) / nh;
    T.mb = nmb - 1 - local / nh;
    T.h = local % nh;
    T.q_row0 = p.cu_seqlens_q[lo];
    T.sq = p.cu_seqlens_q[lo + 1] - T.q_row0;
    T.k_row0 = p.cu_seqlens_k[lo];
    T.sk = p.seqused_k ? p.seqused_k[lo] : p.cu_seqlens_k[lo + 1] - T.k_row0;
  }
  T.g = PACK ? T.h : T.h / p.r;
  T.rows = PACK ? T.sq * p.r : T.sq;
  return true;
}

template <bool PACK, bool SPLIT>
__device__ __forceinline__ Range stage_range(const FwdParams& p, const Tile& T, int r0) {
  Range R;
  R.r0 = r0;
  R.nlo = R.nhi = 0;
  int ilast;
  if constexpr (PACK) {
    R.active = r0 < T.rows;
    R.i0 = r0 / p.r;
    R.i1 = min(r0 + kBM - 1, T.rows - 1) / p.r;
    ilast = R.i1;
  } else {
    R.active = r0 < T.sq;
    R.i0 = r0;
    R.i1 = r0 + kBM - 1;
    ilast = min(r0 + kBM - 1, T.sq - 1);
  }
  if (!R.active) return R;
  const int off = T.sk - T.sq;
  int klo = 0, khi = T.sk;
  if (p.wl >= 0) klo = max(klo, R.i0 + off - p.wl);
  if (p.wr >= 0) khi = min(khi, ilast + off + p.wr + 1);
  if constexpr (SPLIT) {   // split s covers keys [s L, (s+1) L), L a multiple of kBN
    klo = max(klo, T.split * p.split_len);
    khi = min(khi, (T.split + 1) * p.split_len);
  }
  if (khi > klo) {
    R.nlo = klo / kBN;
    R.nhi = (khi + kBN - 1) / kBN;
  }
  return R;
}

__device__ __forceinline__ bool has_work(const Range& R) { return R.nhi > R.nlo; }
__device__ __forceinline__ bool part(const Range& R, int n) { return R.nhi > R.nlo && n >= R.nlo && n < R.nhi; }

// true when some (row, key) of Q tile R x key block n is not visible
__device__ __forceinline__ bool needs_mask(const FwdParams& p, const Tile& T, const Range& R, int n) {
  const int off = T.sk - T.sq;
  const bool full = ((n + 1) * kBN <= T.sk) && (p.wr < 0 || (n + 1) * kBN - 1 <= R.i0 + off + p.wr) &&
                    (p.wl < 0 || n * kBN >= R.i1 + off - p.wl);
  return !full;
}

// Block n is the last, partly filled key block of a sequence whose KV cache
// has unused slots (seqused_k given, TAIL instances only): its V rows past the
// sequence are cleared in shared memory before P.V, which stops at the next
// 16-key boundary.
template <bool TAIL>
__device__ __forceinline__ bool tail_fix(const Tile& T, int n) {
  return TAIL && T.sk - n * kBN < kBN;
}

template <bool TAIL>
__device__ __forceinline__ int pv_steps(const Tile& T, int n) {
  return tail_fix<TAIL>(T, n) ? (T.sk - n * kBN + 15) / 16 : kBN / 16;
}

struct Bars {
  uint64_t* q_full;    // [2]
  uint64_t* q_empty;   // [2]
  uint64_t* k_full;    // [KST]
  uint64_t* k_empty;
  uint64_t* v_full;    // [VST]
  uint64_t* v_empty;
  uint64_t* v_fixed;   // [VST] tail rows of the V tile cleared (seqused_k)
  uint64_t* s_full;    // [2] per S slot
  uint64_t* p_full;    // [2] per S slot
  uint64_t* p_half;    // [2] per S slot (NQ == 2): P of keys [0, 64) stored
  uint64_t* o_bar;     // [2] per O: one phase per P.V
  uint64_t* o_empty;   // [2] per O: epilogue done reading
  uint64_t* pv_done;   // [2] per S slot (NQ == 2): the P.V reading its P has completed
  uint64_t* drain;     // [2] per issuing thread
};

template <class Cfg>
__device__ __forceinline__ Bars carve_bars(uint8_t* smem) {
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  Bars B;
  B.q_full = b; b += 2;
  B.q_empty = b; b += 2;
  B.k_full = b; b += Cfg::KST;
  B.k_empty = b; b += Cfg::KST;
  B.v_full = b; b += Cfg::VST;
  B.v_empty = b; b += Cfg::VST;
  B.v_fixed = b; b += Cfg::VST;
  B.s_full = b; b += 2;
  B.p_full = b; b += 2;
  B.p_half = b; b += 2;
  B.o_bar = b; b += 2;
  B.o_empty = b; b += 2;
  B.pv_done = b; b += 2;
  B.drain = b; b += 2;
  return B;
}

// Key block n of sequence b from a paged cache ("interface.py",
// `_flash_attn_fwd`: k/v (num_pages, page_size, Hkv, D), page_table
// (batch, max_pages)): key j is row j % page_size of page
// page_table[b, j / page_size]. The block is moved in pieces that each lie
// inside one page (128 rows when page_size is a multiple of 128, else 64, else
// page_size rows); a page index outside the pool reads zeros.
template <int NCH>
__device__ __forceinline__ void load_paged(const FwdParams& p, int b, int n, uint8_t* dst, const CUtensorMap* map,
                                           uint64_t* bar, int g) {
  const int ps = p.page_size;
  const int rpl = (ps % kBN == 0) ? kBN : (ps % 64 == 0 ? 64 : ps);
  for (int sub = 0; sub < kBN; sub += rpl) {
    const int key = n * kBN + sub;
    const int pi = key / ps;
    const int page = pi < p.max_pages ? p.page_table[int64_t(b) * p.max_pages + pi] : p.num_pages;
    const int row = key - pi * ps;
#pragma unroll
    for (int c = 0; c < NCH; ++c) tma_load_4d(dst + c * kChunkBytes + sub * 128, map, bar, c * 64, row, g, page);
  }
}

// Spin (bounded, ignoring the abort flag) until the given phase completed:
// used to drain copies / MMAs in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity) && global_timer_ns() - t0 < timeout_ns) {
  }
}

template <int DK, int DV, bool TAIL, bool PACK, bool SPLIT>
__global__ void __launch_bounds__(PrefillCfg<DK, DV>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                   const FwdParams p) {
  using Cfg = PrefillCfg<DK, DV>;
  constexpr int NQ = Cfg::NQ;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the array itself so that accesses
  // through it stay shared-memory accesses with 32-bit addressing
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars B = carve_bars<Cfg>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_BAR + Cfg::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool varlen = p.cu_seqlens_q != nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.q_full[i], 1);
      mbar_init(&B.q_empty[i], 1);
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.p_full[i], 4);      // one arrival per softmax warp
      mbar_init(&B.p_half[i], 4);
      mbar_init(&B.o_bar[i], 1);
      mbar_init(&B.o_empty[i], 4);
      mbar_init(&B.pv_done[i], 1);
      mbar_init(&B.drain[i], 1);
    }
    for (int i = 0; i < Cfg::KST; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
    }
    for (int i = 0; i < Cfg::VST; ++i) {
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
      mbar_init(&B.v_fixed[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
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
  if (warp >= Cfg::MMA_WARP) {
  // the warpgroup of the MMA, TMA and idle warps gives registers away ...
  if constexpr (NQ == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::REG_OTHER));
  if (warp == Cfg::TMA_QK_WARP || warp == Cfg::TMA_V_WARP) {
    // ================= TMA producers =================
    // Q/K: lane 0 alone. V: lane 0, or the whole warp when a KV cache with
    // unused slots (seqused_k) may need rows cleared.
    constexpr unsigned vmask = TAIL ? 0xffffffffu : 1u;
    if (lane == 0 || (TAIL && warp == Cfg::TMA_V_WARP)) {
      const bool is_k = warp == Cfg::TMA_QK_WARP;
      if (is_k) {
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapK);
      } else if (lane == 0) {
        tma_prefetch_desc(&mapV);
      }
      uint32_t kc = 0, qc[2] = {0, 0};
      bool ok = true;
      // K(j) and V(j) are released separately, each by one commit after the
      // last MMA that reads it (K(j) after S(j, *), V(j) after P.V(j, *)), so
      // the next tile of a ring loads as early as possible.
      auto wait_release = [&](uint32_t j, uint64_t* ring, int depth) -> bool {
        return mbar_wait(&ring[j % depth], (j / depth) & 1, guard);
      };
      for (int k = 0; ok; ++k) {
        Tile T;
        if (!fetch_tile<Cfg::ROWS_PER_TILE, PACK, SPLIT>(p, tile_of(k), T)) break;
        Range R[NQ];
        int nlo = INT32_MAX, nhi = INT32_MIN;
#pragma unroll
        for (int s = 0; s < NQ; ++s) {
          R[s] = stage_range<PACK, SPLIT>(p, T, T.mb * Cfg::ROWS_PER_TILE + s * kBM);
          if (has_work(R[s])) {
            nlo = min(nlo, R[s].nlo);
            nhi = max(nhi, R[s].nhi);
          }
        }
        if (nhi <= nlo) continue;
        const int cb = varlen ? 0 : T.b;
        if (is_k) {
#pragma unroll
          for (int s = 0; s < NQ; ++s) {
            if (!has_work(R[s])) continue;
            if (qc[s] > 0 && !mbar_wait(&B.q_empty[s], (qc[s] - 1) & 1, guard)) { ok = false; break; }
            uint8_t* dst = smem + Cfg::OFF_Q + s * Cfg::Q_BYTES;
            mbar_arrive_expect_tx(&B.q_full[s], Cfg::Q_BYTES);
#pragma unroll
            for (int c = 0; c < Cfg::KCH; ++c) {
              if constexpr (PACK)   // (d, head in group, query row, KV head, batch): r heads x 128/r rows
                tma_load_5d(dst + c * kChunkBytes, &mapQ, &B.q_full[s], c * 64, 0, T.q_row0 + R[s].r0 / p.r, T.g,
                            cb);
              else
                tma_load_4d(dst + c * kChunkBytes, &mapQ, &B.q_full[s], c * 64, T.q_row0 + R[s].r0, T.h, cb);
            }
            ++qc[s];
          }
          for (int n = nhi - 1; ok && n >= nlo; --n) {
            const int st = kc % Cfg::KST;
            if (kc >= Cfg::KST && !wait_release(kc - Cfg::KST, B.k_empty, Cfg::KST)) { ok = false; break; }
            uint8_t* dst = smem + Cfg::OFF_K + st * Cfg::K_BYTES;
            mbar_arrive_expect_tx(&B.k_full[st], Cfg::K_BYTES);
            if (p.page_table == nullptr) {
#pragma unroll
              for (int c = 0; c < Cfg::KCH; ++c)
                tma_load_4d(dst + c * kChunkBytes, &mapK, &B.k_full[st], c * 64, T.k_row0 + n * kBN, T.g, cb);
            } else {
              load_paged<Cfg::KCH>(p, T.b, n, dst, &mapK, &B.k_full[st], T.g);
            }
            ++kc;
          }
        } else {
          for (int n = nhi - 1; ok && n >= nlo; --n) {
            const int st = kc % Cfg::VST;
            uint8_t* dst = smem + Cfg::OFF_V + st * Cfg::V_BYTES;
            bool w = true;
            if (lane == 0) {
              w = kc < Cfg::VST || wait_release(kc - Cfg::VST, B.v_empty, Cfg::VST);
              if (w) {
                mbar_arrive_expect_tx(&B.v_full[st], Cfg::V_BYTES);
                if (p.page_table == nullptr) {
#pragma unroll
                  for (int c = 0; c < Cfg::VCH; ++c)
                    tma_load_4d(dst + c * kChunkBytes, &mapV, &B.v_full[st], c * 64, T.k_row0 + n * kBN, T.g, cb);
                } else {
                  load_paged<Cfg::VCH>(p, T.b, n, dst, &mapV, &B.v_full[st], T.g);
                }
              }
            }
            if (!__shfl_sync(vmask, w ? 1 : 0, 0)) { ok = false; break; }
            if (tail_fix<TAIL>(T, n)) {
              // Cache slots at or past seqused_k may never have been written
              // (NaN); P is 0 there, but 0 * NaN is not. Clear the rows up to
              // the next 16-key step boundary: the P.V of this block stops there.
              const int valid = T.sk - n * kBN;
              const bool f = __all_sync(vmask, mbar_wait(&B.v_full[st], (kc / Cfg::VST) & 1, guard));
              if (!f) { ok = false; break; }
              const int pieces = (min(kBN, (valid + 15) & ~15) - valid) * Cfg::VCH * 8;
              for (int idx = lane; idx < pieces; idx += 32) {
                const int row = valid + idx / (Cfg::VCH * 8), rem = idx % (Cfg::VCH * 8);
                *reinterpret_cast<uint4*>(dst + (rem >> 3) * kChunkBytes + row * 128 + (rem & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp(vmask);
              if (lane == 0) mbar_arrive(&B.v_fixed[st]);
            }
            ++kc;
          }
        }
      }
      // drain the copies still in flight (only after an abort can any be)
      if (is_k) {
        const int nst = Cfg::KST;
        for (uint32_t u = (kc > (uint32_t)nst ? kc - nst : 0); u < kc; ++u)
          drain_wait(&B.k_full[u % nst], (u / nst) & 1, p.timeout_ns);
        for (int s = 0; s < NQ; ++s)
          if (qc[s] > 0) drain_wait(&B.q_full[s], (qc[s] - 1) & 1, p.timeout_ns);
      } else if (lane == 0) {
        const int nst = Cfg::VST;
        for (uint32_t u = (kc > (uint32_t)nst ? kc - nst : 0); u < kc; ++u)
          drain_wait(&B.v_full[u % nst], (u / nst) & 1, p.timeout_ns);
      }
    }
  } else if (warp == Cfg::MMA_WARP || (NQ == 2 && warp == Cfg::PV_WARP)) {
    // ================= MMA issuers =================
    // A tcgen05.mma takes about 50 cycles to issue and the tensor queue holds
    // only a few instructions, while an M=128 N=128 K=16 MMA runs 64 cycles:
    // one thread issuing every GEMM of the two-tile kernels (plus its waits
    // and commits) cannot keep the pipe busy. So with NQ == 2 lane 0 of the
    // MMA warp issues S = Q K^T and lane 0 of the P.V warp (another SM
    // sub-partition) issues O += P V. S(n-1, t) overwrites the TMEM columns
    // P(n, t) occupies, so it waits until the P.V reading them has completed
    // (pv_done[t]). The head-dim-256 kernel keeps one issuing thread.
    if (lane == 0) {
      const bool s_role = warp == Cfg::MMA_WARP;
      constexpr uint32_t IDESC_S = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(kBM, DV, false, true);
      const uint32_t q_base = smem_u32(smem + Cfg::OFF_Q);
      const uint32_t k_base = smem_u32(smem + Cfg::OFF_K);
      const uint32_t v_base = smem_u32(smem + Cfg::OFF_V);

      // S[slot] = Q[qs] K[kst]^T, K-major operands, 16 deep per instruction
      // Descriptors are built once per operand; a K step only moves the start
      // address, which lives in the low bits (no carry: addresses < 256 KB).
      auto issue_s = [&](int qs, int slot, int kst) {
        const uint32_t d = tmem + slot * 128;
        const uint64_t qd = sdesc_sw128(q_base + qs * Cfg::Q_BYTES, 16, 1024);
        const uint64_t kd = sdesc_sw128(k_base + kst * Cfg::K_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          mma_bf16_ss(d, qd + off, kd + off, IDESC_S, kk > 0);
        }
      };
      // O[o] (+)= P[slot] V[vst]; P from TMEM, V MN-major (64-column chunks 16 KB apart)
      auto issue_pv = [&](int o, int slot, int vst, bool acc, int steps) {
        const uint32_t d = tmem + Cfg::O_COL + o * DV;
        const uint64_t vd = sdesc_sw128(v_base + vst * Cfg::V_BYTES, kChunkBytes, 1024);
        const uint32_t pa = tmem + slot * 128;
        if (steps == kBN / 16) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_bf16_ts(d, pa + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, (kk > 0 || acc) ? 1u : 0u);
        } else {
          for (int kk = 0; kk < steps; ++kk)
            mma_bf16_ts(d, pa + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, (kk > 0 || acc) ? 1u : 0u);
        }
      };
      // the 16-key steps [k0, k1) of the same product (P of keys 16 k0 .. 16 k1 - 1)
      auto issue_pv_steps = [&](int o, int slot, int vst, bool acc, int k0, int k1) {
        const uint32_t d = tmem + Cfg::O_COL + o * DV;
        const uint64_t vd = sdesc_sw128(v_base + vst * Cfg::V_BYTES, kChunkBytes, 1024);
        const uint32_t pa = tmem + slot * 128;
        if (k0 == 0 && k1 == 4) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(d, pa + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, (kk > 0 || acc) ? 1u : 0u);
        } else if (k0 == 4 && k1 == 8) {
#pragma unroll
          for (int kk = 4; kk < 8; ++kk)
            mma_bf16_ts(d, pa + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, 1u);
        } else {
          for (int kk = k0; kk < k1; ++kk)
            mma_bf16_ts(d, pa + kk * 8, vd + ((kk * 16 * 128) >> 4), IDESC_PV, (kk > 0 || acc) ? 1u : 0u);
        }
      };
      uint32_t vfix = 0;   // parity bit per V stage of its v_fixed barrier
      auto wait_fix = [&](int n, int vst, const Tile& T) -> bool {
        if (!tail_fix<TAIL>(T, n)) return true;
        const bool r = mbar_wait(&B.v_fixed[vst], (vfix >> vst) & 1u, guard);
        vfix ^= 1u << vst;
        return r;
      };

      uint32_t kc = 0, vc = 0, qw[2] = {0, 0}, pw[2] = {0, 0}, ou[2] = {0, 0};
      uint32_t sc[2] = {0, 0};   // NQ == 2: S GEMMs issued per slot (one pv_done phase each)
      uint32_t jc = 0;   // NQ == 1: jobs so far (S slot = job parity)
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Tile T;
        if (!fetch_tile<Cfg::ROWS_PER_TILE, PACK, SPLIT>(p, tile_of(k), T)) break;
        Range R[NQ];
        int nlo = INT32_MAX, nhi = INT32_MIN;
#pragma unroll
        for (int s = 0; s < NQ; ++s) {
          R[s] = stage_range<PACK, SPLIT>(p, T, T.mb * Cfg::ROWS_PER_TILE + s * kBM);
          if (has_work(R[s])) {
            nlo = min(nlo, R[s].nlo);
            nhi = max(nhi, R[s].nhi);
          }
        }
        if (nhi <= nlo) continue;
        bool first_s[2] = {true, true}, first_pv[2] = {true, true};

        auto wait_q = [&](int s) -> bool {
          if (!first_s[s]) return true;
          first_s[s] = false;
          const bool r = mbar_wait(&B.q_full[s], qw[s] & 1, guard);
          ++qw[s];
          return r;
        };
        auto before_pv = [&](int o) -> bool {   // O[o] free for the tile's first P.V
          if (!first_pv[o]) return true;
          first_pv[o] = false;
          bool r = true;
          if (ou[o] > 0) r = mbar_wait(&B.o_empty[o], (ou[o] - 1) & 1, guard);
          ++ou[o];
          return r;
        };

        if constexpr (NQ == 2) {
          // Q tile t takes part in key block n when lo[t] <= n < hi[t]
          const int lo[2] = {has_work(R[0]) ? R[0].nlo : INT32_MAX, has_work(R[1]) ? R[1].nlo : INT32_MAX};
          const int hi[2] = {has_work(R[0]) ? R[0].nhi : INT32_MIN, has_work(R[1]) ? R[1].nhi : INT32_MIN};
          if (s_role) {
            // ---- S = Q K^T for every block, both Q tiles; K(n) released after S(n, *)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (hi[t] > lo[t]) {
                if (!mbar_wait(&B.q_full[t], qw[t] & 1, guard)) { ok = false; break; }
                ++qw[t];
              }
            }
            if (!ok) break;
            for (int n = nhi - 1; n >= nlo; --n) {
              const int st = kc % Cfg::KST;
              if (!mbar_wait(&B.k_full[st], (kc / Cfg::KST) & 1, guard)) { ok = false; break; }
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (n < lo[t] || n >= hi[t]) continue;
                // the previous P of this slot has been read by its P.V
                if (sc[t] > 0 && !mbar_wait(&B.pv_done[t], (sc[t] - 1) & 1, guard)) { ok = false; break; }
                tc_fence_after();
                issue_s(t, t, st);
                mma_commit(&B.s_full[t]);
                if (n == lo[t]) mma_commit(&B.q_empty[t]);
                ++sc[t];
              }
              if (!ok) break;
              mma_commit(&B.k_empty[st]);
              ++kc;
            }
          } else {
            // ---- O += P V for every block, both Q tiles; V(n) released after P.V(n, *)
            for (int n = nhi - 1; n >= nlo; --n) {
              const int vst = vc % Cfg::VST;
              if (!mbar_wait(&B.v_full[vst], (vc / Cfg::VST) & 1, guard)) { ok = false; break; }
              if (!wait_fix(n, vst, T)) { ok = false; break; }
              const int steps = pv_steps<TAIL>(T, n);
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (n < lo[t] || n >= hi[t]) continue;
                if (n == hi[t] - 1) {   // O[t] free once the previous tile's epilogue read it
                  if (ou[t] > 0 && !mbar_wait(&B.o_empty[t], (ou[t] - 1) & 1, guard)) { ok = false; break; }
                  ++ou[t];
                }
                // keys [0, 64) as soon as their P is stored, then the rest
                if (!mbar_wait(&B.p_half[t], pw[t] & 1, guard)) { ok = false; break; }
                tc_fence_after();
                issue_pv_steps(t, t, vst, n != hi[t] - 1, 0, min(4, steps));
                if (!mbar_wait(&B.p_full[t], pw[t] & 1, guard)) { ok = false; break; }
                ++pw[t];
                tc_fence_after();
                issue_pv_steps(t, t, vst, n != hi[t] - 1, 4, steps);
                mma_commit(&B.pv_done[t]);
                if (n == lo[t]) mma_commit(&B.o_bar[t]);   // O[t] complete for this tile
              }
              if (!ok) break;
              mma_commit(&B.v_empty[vst]);
              ++vc;
            }
          }
        } else {
          // one Q tile, S slots alternate: S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ...
          const int cnt = nhi - nlo;
          auto do_s = [&](int i) -> bool {
            const int st = kc % Cfg::KST;
            if (!mbar_wait(&B.k_full[st], (kc / Cfg::KST) & 1, guard)) return false;
            if (!wait_q(0)) return false;
            const int slot = (jc + i) & 1;
            issue_s(0, slot, st);
            mma_commit(&B.s_full[slot]);
            if (i == cnt - 1) mma_commit(&B.q_empty[0]);
            mma_commit(&B.k_empty[st]);
            ++kc;
            return true;
          };
          for (int i = 0; ok && i < min(2, cnt); ++i) ok = do_s(i);
          for (int i = 0; ok && i < cnt; ++i) {
            const int slot = (jc + i) & 1;
            const int vst = vc % Cfg::VST;
            if (!mbar_wait(&B.v_full[vst], (vc / Cfg::VST) & 1, guard)) { ok = false; break; }
            if (!wait_fix(nhi - 1 - i, vst, T)) { ok = false; break; }
            const uint32_t pwc = slot ? pw[1] : pw[0];
            if (!mbar_wait(&B.p_full[slot], pwc & 1, guard)) { ok = false; break; }
            if (slot) ++pw[1]; else ++pw[0];
            tc_fence_after();
            const bool acc = i > 0;
            if (!before_pv(0)) { ok = false; break; }
            issue_pv(0, slot, vst, acc, pv_steps<TAIL>(T, nhi - 1 - i));
            mma_commit(&B.o_bar[0]);
            mma_commit(&B.v_empty[vst]);
            ++vc;
            if (i + 2 < cnt) ok = do_s(i + 2);
          }
          jc += cnt;
        }
      }
      // wait for every MMA this thread issued before TMEM is released
      uint64_t* drain = &B.drain[s_role ? 0 : 1];
      mma_commit(drain);
      drain_wait(drain, 0, p.timeout_ns);
    }
    __syncwarp();
  }
  } else {
    // ... and the softmax warpgroups take them
    if constexpr (NQ == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REG_SOFTMAX));
    // ================= softmax warpgroups =================
    const int wg = warp >> 2;                 // Q tile (NQ == 2) or 0
    const int row_local = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int o_idx = (NQ == 2) ? wg : 0;
    const uint32_t o_addr = tmem + lane_off + Cfg::O_COL + o_idx * DV;
    uint32_t sw0 = 0, sw1 = 0;  // S waits per slot
    uint32_t ow = 0;           // o_bar phases consumed (one per P.V of this O, in order)
    uint32_t jc = 0;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Tile T;
      if (!fetch_tile<Cfg::ROWS_PER_TILE, PACK, SPLIT>(p, tile_of(k), T)) break;
      const Range R = stage_range<PACK, SPLIT>(p, T, T.mb * Cfg::ROWS_PER_TILE + wg * kBM);
      if (!R.active) continue;
      const int trow = R.r0 + row_local;                       // tile row
      const bool valid = PACK ? trow < T.rows : trow < T.sq;
      const int i = PACK ? trow / p.r : trow;                  // query row
      const int hh = PACK ? T.g * p.r + trow % p.r : T.h;      // q head
      const int64_t orow = (varlen ? 0 : int64_t(T.b) * p.o_bs) + int64_t(T.q_row0 + i) * p.o_rs +
                           int64_t(hh) * p.o_hs;
      const int64_t lrow = varlen ? int64_t(hh) * p.total_q + T.q_row0 + i
                                  : (int64_t(T.b) * p.hq + hh) * p.seqlen_q + i;
      // SPLIT instances write fp32 partials: O_s (normalised by its own row
      // sum) at [split][row][head][d] and LSE_s at [split][head-major row],
      // the layouts the combine reads
      float* opart = nullptr;
      float* lpart = nullptr;
      if constexpr (SPLIT) {
        const int64_t rows_total = varlen ? int64_t(p.total_q) : int64_t(p.batch) * p.seqlen_q;
        const int64_t ri = varlen ? int64_t(T.q_row0 + i) : int64_t(T.b) * p.seqlen_q + i;
        opart = p.out_partial + ((int64_t(T.split) * rows_total + ri) * p.hq + hh) * DV;
        lpart = p.lse_partial + (varlen ? (int64_t(T.split) * p.hq + hh) * p.total_q + T.q_row0 + i
                                        : ((int64_t(T.split) * p.batch + T.b) * p.hq + hh) * p.seqlen_q + i);
      }
      if (!has_work(R)) {
        if (valid) {
          if constexpr (SPLIT) {
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < DV / 4; ++c) reinterpret_cast<float4*>(opart)[c] = z;
            *lpart = -INFINITY;
          } else {
            uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < DV / 8; ++c) *reinterpret_cast<uint4*>(out + orow + c * 8) = z;
            if (p.lse) p.lse[lrow] = -INFINITY;
          }
        }
        continue;
      }
      const int off = T.sk - T.sq;
      float m = -INFINITY, l = 0.f;
      // One instance of the block body for blocks with masked keys and one for
      // blocks without: sharing the code after the mask made every block
      // slower, and the masked instance's per-column test is one unsigned
      // range compare (measured: causal +2 to 3 %, varlen +1 to 3 %)
      auto block = [&](auto masked, int n) -> bool {
        const int slot = (NQ == 2) ? wg : (jc & 1);
        if (!mbar_wait(&B.s_full[slot], (slot ? sw1 : sw0) & 1, guard)) return false;
        if (slot) ++sw1; else ++sw0;
        tc_fence_after();
        uint32_t r[128];
        float* s = reinterpret_cast<float*>(r);
        float bmax = -INFINITY;
        if constexpr (decltype(masked)::value) {
          // ---- a block with masked keys ----
          const int jb = n * kBN;
          const int c_lo = (p.wl >= 0) ? i + off - p.wl - jb : INT32_MIN / 2;
          int c_hi = T.sk - 1 - jb;
          if (p.wr >= 0) c_hi = min(c_hi, i + off + p.wr - jb);
          const bool row_vis = c_hi >= c_lo && c_hi >= 0 && c_lo <= 127;   // the row sees a key here
          // column c is visible when (unsigned)(c - c_lo) <= (unsigned)(c_hi - c_lo); an
          // empty range gets a lower end past every column
          const int lo_e = (c_hi < c_lo) ? 256 : c_lo;
          const uint32_t width = (c_hi < c_lo) ? 0u : static_cast<uint32_t>(c_hi - c_lo);
          auto apply_mask = [&]() {
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = (static_cast<uint32_t>(c - lo_e) <= width) ? s[c] : -INFINITY;
          };
          const bool first = n == R.nhi - 1;
          float m_new = m, lsum = 0.f;
          bool need = false;
          // The load's own row max covers the masked columns too, so it is only an
          // upper bound mc of the visible max (a max over the masked row costs far
          // more here). P is first formed against mc, masked columns exactly 0; the
          // largest P then gives the visible block max, mc + log2(p_max), and P is
          // scaled to the reference the online softmax would have used, so the
          // row's largest P is 1 as with the exact max. A row whose visible keys
          // all sit more than 100 (base 2) under mc is redone below with the
          // visible max (S is still in tensor memory).
          float hw;
          tmem_ld128_max(tmem + lane_off + slot * 128, r, hw);
          apply_mask();
          const float mc = fmaxf(m, row_vis ? hw * p.scale_log2 : -INFINITY);
          const float muc = (mc == -INFINITY) ? 0.f : mc;
          {
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-muc, -muc);
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
              s[c] = ex2_approx(x.x);
              s[c + 1] = ex2_approx(x.y);
            }
          }
          float pm[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) pm[j] = s[j];
#pragma unroll
          for (int c = 8; c + 16 <= 128; c += 16) {
#pragma unroll
            for (int j = 0; j < 8; ++j) pm[j] = fmax3(pm[j], s[c + j], s[c + 8 + j]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) pm[j] = fmaxf(pm[j], s[120 + j]);
          const float p_max = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
          if (!__any_sync(0xffffffffu, row_vis && !(p_max >= 0x1p-100f))) {
            const float mb = (p_max > 0.f) ? muc + __log2f(p_max) : -INFINITY;   // visible block max
            m_new = fmaxf(m, mb);
            need = first || m_new > m + kRescaleThreshold;
            const float mref = need ? m_new : m;
            const float mu = (mref == -INFINITY) ? 0.f : mref;
            const float g = (p_max > 0.f) ? ex2_approx(muc - mu) : 0.f;
            const float2 g2 = make_float2(g, g);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const float2 pv = __fmul2_rn(make_float2(s[2 * c], s[2 * c + 1]), g2);
              acc[c & 3] = __fadd2_rn(acc[c & 3], pv);
              r[c] = pack_bf16x2(pv.x, pv.y);
            }
            const float2 a2 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
            lsum = a2.x + a2.y;
            // P into tensor memory over S's first 64 columns (published below)
            if constexpr (NQ == 2) {
              tmem_st32(tmem + lane_off + slot * 128, reinterpret_cast<uint32_t(&)[32]>(r[0]));
              tmem_st32(tmem + lane_off + slot * 128 + 32, reinterpret_cast<uint32_t(&)[32]>(r[32]));
            } else {
              tmem_st64(tmem + lane_off + slot * 128, reinterpret_cast<uint32_t(&)[64]>(r));
            }
          } else {
            // (rare) the same with the visible max, S read again 32 columns at a
            // time and each chunk's P stored over S columns already read
            float bx = -INFINITY;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t t[32];
              tmem_ld32(tmem + lane_off + slot * 128 + 32 * ch, t);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (static_cast<uint32_t>(32 * ch + e - lo_e) <= width) bx = fmaxf(bx, __uint_as_float(t[e]));
            }
            m_new = fmaxf(m, bx * p.scale_log2);
            need = first || m_new > m + kRescaleThreshold;
            const float mref = need ? m_new : m;
            const float mu = (mref == -INFINITY) ? 0.f : mref;
            float sum = 0.f;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t t[32], w[16];
              tmem_ld32(tmem + lane_off + slot * 128 + 32 * ch, t);
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                float pv[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int e = 2 * k + u;
                  const bool vis = static_cast<uint32_t>(32 * ch + e - lo_e) <= width;
                  pv[u] = vis ? ex2_approx(fmaf(__uint_as_float(t[e]), p.scale_log2, -mu)) : 0.f;
                  sum += pv[u];
                }
                w[k] = pack_bf16x2(pv[0], pv[1]);
              }
              tmem_st16(tmem + lane_off + slot * 128 + 16 * ch, w);
            }
            lsum = sum;
          }
          tmem_st_wait();
          // the O rescale (not on a tile's first block), as for unmasked blocks
          bool pending = (NQ == 1) && !first;
          if (first) {
            m = m_new;
          } else if (__any_sync(0xffffffffu, need)) {
            if (NQ == 1) {
              if (!mbar_wait(&B.o_bar[o_idx], ow & 1, guard)) return false;
              ++ow;
              pending = false;
            }
            tc_fence_after();
            const float f = need ? ex2_approx(m - m_new) : 1.f;
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(o_addr + c * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
              tmem_st32(o_addr + c * 32, o);
            }
            tmem_st_wait();
            if (need) {
              l *= f;
              m = m_new;
            }
          }
          l += lsum;
          if (pending) {
            if (!mbar_wait(&B.o_bar[o_idx], ow & 1, guard)) return false;
            ++ow;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (NQ == 2) mbar_arrive(&B.p_half[slot]);
            mbar_arrive(&B.p_full[slot]);
          }
          ++jc;
          return true;
        } else {
          // every column is visible: the load returns the row max with the row
          float hw;
          tmem_ld128_max(tmem + lane_off + slot * 128, r, hw);
          bmax = hw * p.scale_log2;
        }
        if constexpr (!decltype(masked)::value) {
          const float m_new = fmaxf(m, bmax);
          // The previous P.V of this O (if any in this tile) has a phase on o_bar
          // that is consumed exactly once: before O is rescaled, or else just
          // before this block's P is published (so the next P.V cannot run ahead).
          // NQ == 1 only: with NQ == 2, S(n) completing implies every earlier
          // P.V of this O completed (the S thread issued S(n) only after the
          // P.V of the block before had completed, pv_done).
          bool pending = (NQ == 1) && (n != R.nhi - 1);
          if (n == R.nhi - 1) {
            m = m_new;
          } else {
            const bool need = m_new > m + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
              if (NQ == 1) {
                if (!mbar_wait(&B.o_bar[o_idx], ow & 1, guard)) return false;
                ++ow;
                pending = false;
              }
              tc_fence_after();
              const float f = need ? ex2_approx(m - m_new) : 1.f;
#pragma unroll 1
              for (int c = 0; c < DV / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_addr + c * 32, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                tmem_st32(o_addr + c * 32, o);
              }
              tmem_st_wait();
              if (need) {
                l *= f;
                m = m_new;
              }
            }
          }
          const float mu = (m == -INFINITY) ? 0.f : m;
          const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
          const float2 nm2 = make_float2(-mu, -mu);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
          if constexpr (NQ == 2) {
            // P in two halves: keys [0, 64) are stored and published first, so
            // that the P.V thread starts on them while the rest is computed
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
              s[c] = ex2_approx(x.x);
              s[c + 1] = ex2_approx(x.y);
              acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(s[c], s[c + 1]));
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = pack_bf16x2(s[2 * c], s[2 * c + 1]);
            tmem_st32(tmem + lane_off + slot * 128, reinterpret_cast<uint32_t(&)[32]>(r[0]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.p_half[slot]);
#pragma unroll
            for (int c = 64; c < 128; c += 2) {
              const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
              s[c] = ex2_approx(x.x);
              s[c + 1] = ex2_approx(x.y);
              acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(s[c], s[c + 1]));
            }
#pragma unroll
            for (int c = 32; c < 64; ++c) r[c] = pack_bf16x2(s[2 * c], s[2 * c + 1]);
            tmem_st32(tmem + lane_off + slot * 128 + 32, reinterpret_cast<uint32_t(&)[32]>(r[32]));
            tmem_st_wait();
          } else {
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
              s[c] = ex2_approx(x.x);
              s[c + 1] = ex2_approx(x.y);
              acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(s[c], s[c + 1]));
            }
#pragma unroll
            for (int c = 0; c < 64; ++c) r[c] = pack_bf16x2(s[2 * c], s[2 * c + 1]);
            tmem_st64(tmem + lane_off + slot * 128, reinterpret_cast<uint32_t(&)[64]>(r));
            tmem_st_wait();
          }
          const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
          const float2 a = __fadd2_rn(a01, a23);
          l += a.x + a.y;
          if (pending) {
            if (!mbar_wait(&B.o_bar[o_idx], ow & 1, guard)) return false;
            ++ow;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.p_full[slot]);
          ++jc;
        }
        return true;
      };
      for (int n = R.nhi - 1; n >= R.nlo; --n) {
        const bool go = needs_mask(p, T, R, n) ? block(std::true_type{}, n) : block(std::false_type{}, n);
        if (!go) { ok = false; break; }
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE (natural log) ----
      if (!mbar_wait(&B.o_bar[o_idx], ow & 1, guard)) { ok = false; break; }
      ++ow;
      tc_fence_after();
      const bool empty_row = !(l > 0.f);
      const float inv_l = empty_row ? 0.f : 1.f / l;
      // Each warp's 32 rows go out by TMA, 32 columns at a time, through two
      // 2 KB staging buffers used in turn (rows 64-byte swizzled, so the
      // warp's 16-byte writes take the minimum four wavefronts): a chunk only
      // waits for the store two chunks back to have read its buffer. Rows past
      // the tensor end are clipped by the store, and no wait spans more than
      // the warp. Rows of a varlen tile that would run into the next sequence,
      // and packed groups of more than 32 heads, are written row by row.
      const int wrow0 = R.r0 + (warp & 3) * 32;   // first tile row of this warp
      bool staged = false;
      if constexpr (Cfg::OSTAGE && !SPLIT) staged = (!varlen || wrow0 + 32 <= T.rows) && (!PACK || p.r <= 32);
      if constexpr (SPLIT) {
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
          if (valid) {
            float* dst = opart + c * 32;
            if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {   // whole 32-byte sectors
#pragma unroll
              for (int e = 0; e < 4; ++e)
                st_global_v8(dst + 8 * e, __float_as_uint(__uint_as_float(o[8 * e]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 1]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 2]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 3]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 4]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 5]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 6]) * inv_l),
                             __float_as_uint(__uint_as_float(o[8 * e + 7]) * inv_l));
            } else {
              float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                d4[e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                    __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
            }
          }
        }
        if (valid) *lpart = empty_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
      } else if (staged) {
        uint8_t* stg = smem + Cfg::OFF_OST + wg * kChunkBytes + (warp & 3) * (kChunkBytes / 4);
        const int cb = varlen ? 0 : T.b;
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint8_t* buf = stg + (c & 1) * 2048;
          if (lane == 0) bulk_wait_read_but_one();   // the store two chunks back has read buf
          __syncwarp();
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v4 = make_uint4(
                pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l),
                pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l),
                pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l),
                pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l));
            *reinterpret_cast<uint4*>(buf + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) = v4;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PACK)
              tma_store_5d(&mapO, buf, c * 32, 0, T.q_row0 + wrow0 / p.r, T.g, cb);
            else
              tma_store_4d(&mapO, buf, c * 32, T.q_row0 + wrow0, T.h, cb);
            bulk_commit_group();
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
          if (valid) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
            __nv_bfloat16* dst = out + orow + c * 32;
            if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {   // whole 32-byte sectors
              st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
              d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
              d4[2] = make_uint4(w[8], w[9], w[10], w[11]);
              d4[3] = make_uint4(w[12], w[13], w[14], w[15]);
            }
          }
        }
      }
      if (!SPLIT && valid && p.lse) p.lse[lrow] = empty_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.o_empty[o_idx]);
    }
    // the staging buffers stay in use until every store has completed
    if constexpr (Cfg::OSTAGE) {
      if (lane == 0) bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void varlen_prepare_kernel(const int* cu_seqlens_q, int batch, int rows_per_tile, int hq,
                                      int mult, int* prefix) {
  __shared__ int part[1024];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (batch + nt - 1) / nt;
  const int b0 = min(batch, tid * per), b1 = min(batch, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) {
    const int sq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    sum += ((sq * mult + rows_per_tile - 1) / rows_per_tile) * hq;
  }
  part[tid] = sum;
  __syncthreads();
  for (int o = 1; o < nt; o <<= 1) {
    const int v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = part[tid] - sum;
  for (int b = b0; b < b1; ++b) {
    prefix[b] = run;
    const int sq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    run += ((sq * mult + rows_per_tile - 1) / rows_per_tile) * hq;
  }
  if (tid == nt - 1) prefix[batch] = part[tid];
}

template <int DK, int DV>
cudaError_t launch_prefill_t(const FwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, const CUtensorMap& mo, int num_sms, cudaStream_t stream) {
  using Cfg = PrefillCfg<DK, DV>;
  // the TAIL instances clear cache rows past seqused_k, the PACK ones fold q
  // heads into tile rows; the plain instance has neither
  // (the SPLIT instances, for grids that would leave SMs idle, take the TAIL
  // form whether or not the cache has unused slots)
  auto kern = p.write_partial ? (p.pack ? prefill_kernel<DK, DV, true, true, true> : prefill_kernel<DK, DV, true, false, true>)
            : p.seqused_k != nullptr ? (p.pack ? prefill_kernel<DK, DV, true, true, false> : prefill_kernel<DK, DV, true, false, false>)
                                     : (p.pack ? prefill_kernel<DK, DV, false, true, false> : prefill_kernel<DK, DV, false, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  if (e != cudaSuccess) return e;
  long long tiles;
  if (p.cu_seqlens_q == nullptr) {
    tiles = p.num_tiles;
  } else {
    const long long rows = (long long)p.max_seqlen_q * (p.pack ? p.r : 1);
    tiles = (long long)p.batch * (p.pack ? p.hkv : p.hq) * ((rows + Cfg::ROWS_PER_TILE - 1) / Cfg::ROWS_PER_TILE);
  }
  if (p.write_partial) tiles *= p.num_splits;
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 192 && dv == 128) ||
         (dk == 256 && dv == 256);
}

int prefill_rows_per_tile(int dk, int dv) {
  if (dk == 64 && dv == 64) return PrefillCfg<64, 64>::ROWS_PER_TILE;
  if (dk == 128 && dv == 128) return PrefillCfg<128, 128>::ROWS_PER_TILE;
  if (dk == 192 && dv == 128) return PrefillCfg<192, 128>::ROWS_PER_TILE;
  if (dk == 256 && dv == 256) return PrefillCfg<256, 256>::ROWS_PER_TILE;
  return 0;
}

cudaError_t launch_prefill(const FwdParams& p, int dk, int dv, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mo, int num_sms, cudaStream_t stream) {
  if (dk == 64 && dv == 64) return launch_prefill_t<64, 64>(p, mq, mk, mv, mo, num_sms, stream);
  if (dk == 128 && dv == 128) return launch_prefill_t<128, 128>(p, mq, mk, mv, mo, num_sms, stream);
  if (dk == 192 && dv == 128) return launch_prefill_t<192, 128>(p, mq, mk, mv, mo, num_sms, stream);
  if (dk == 256 && dv == 256) return launch_prefill_t<256, 256>(p, mq, mk, mv, mo, num_sms, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_varlen_prepare(const FwdParams& p, int rows_per_tile, cudaStream_t stream) {
  varlen_prepare_kernel<<<1, 1024, 0, stream>>>(p.cu_seqlens_q, p.batch, rows_per_tile, p.pack ? p.hkv : p.hq,
                                                p.pack ? p.r : 1, p.tile_prefix);
  return cudaGetLastError();
}

}  // namespace fa
