// fa_selftest.cu - test-only library (libfa_selftest.so) that exercises the
// tcgen05 building blocks of the prefill kernel on single tiles, so that a
// descriptor or layout mistake shows up in isolation:
//   fa_selftest_qk:  S[128x128] = Q[128xDK] K[128xDK]^T   (both K-major, SW128)
//   fa_selftest_pv:  O[128xDV]  = P[128x128] V[128xDV]    (P from TMEM, V MN-major)
//   fa_selftest_wait_timeout: the bounded mbarrier wait on a barrier nothing
//                    arrives on gives up, reports and lets the CTA exit cleanly
// Inputs are bf16 device arrays (row-major, contiguous); outputs fp32.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_ptx.cuh"

namespace {

using namespace fa;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool map2d(CUtensorMap* m, const void* base, int cols, int rows) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  auto enc = reinterpret_cast<EncodeTiledFn>(ptr);
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

constexpr uint64_t kTimeout = 2000000000ull;

template <int DK>
__global__ void __launch_bounds__(128) qk_kernel(const __grid_constant__ CUtensorMap mq,
                                                 const __grid_constant__ CUtensorMap mk, float* s_out, int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  constexpr int CH = DK / 64;
  uint8_t* qs = smem;
  uint8_t* ks = smem + CH * 16384;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * CH * 16384);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const WaitGuard g{abort_flag, status, kTimeout};
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], 2 * CH * 16384);
    for (int c = 0; c < CH; ++c) {
      tma_load_2d(qs + c * 16384, &mq, &bars[0], c * 64, 0);
      tma_load_2d(ks + c * 16384, &mk, &bars[0], c * 64, 0);
    }
    if (mbar_wait(&bars[0], 0, g)) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16_ss(tmem, sdesc_sw128(smem_u32(qs) + off, 16, 1024), sdesc_sw128(smem_u32(ks) + off, 16, 1024),
                    idesc, kk > 0);
      }
      mma_commit(&bars[1]);
    }
  }
  __syncwarp();
  if (mbar_wait(&bars[1], 0, g)) {
    tc_fence_after();
    const int row = warp * 32 + lane;
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, r);
      for (int e = 0; e < 32; ++e) s_out[row * 128 + c * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int DV>
__global__ void __launch_bounds__(128) pv_kernel(const __nv_bfloat16* p_in, const __grid_constant__ CUtensorMap mv,
                                                 float* o_out, int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  constexpr int CH = DV / 64;
  uint8_t* vs = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CH * 16384);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NCOL = (DV + 128 <= 256) ? 256 : 512;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 128);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, NCOL);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const WaitGuard g{abort_flag, status, kTimeout};
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  // P row (this thread's) -> TMEM columns [0, 64) packed bf16x2
  {
    const int row = warp * 32 + lane;
    uint32_t r[64];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p_in + row * 128);
    for (int c = 0; c < 64; ++c) r[c] = src[c];
    tmem_st64(tmem + lane_off, r);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars[2]);
  }
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], CH * 16384);
    for (int c = 0; c < CH; ++c) tma_load_2d(vs + c * 16384, &mv, &bars[0], c * 64, 0);
    if (mbar_wait(&bars[0], 0, g) && mbar_wait(&bars[2], 0, g)) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, DV, false, true);
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts(tmem + 128, tmem + kk * 8, sdesc_sw128(smem_u32(vs) + kk * 2048, 16384, 1024), idesc, kk > 0);
      mma_commit(&bars[1]);
    }
  }
  __syncwarp();
  if (mbar_wait(&bars[1], 0, g)) {
    tc_fence_after();
    const int row = warp * 32 + lane;
    for (int c = 0; c < DV / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + 128 + c * 32, r);
      for (int e = 0; e < 32; ++e) o_out[row * DV + c * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, NCOL);
  }
}

// A wait that can never complete (nothing arrives on the barrier): the bounded
// wait must give up after timeout_ns, set the status word, raise the shared
// abort flag so the other waiting warp gives up too, and let the CTA free its
// TMEM and exit. report[0] = 1 if warp 0's wait returned false, report[1] = 1 if
// warp 1 saw the abort (its own wait returned false without timing out first).
__global__ void __launch_bounds__(64, 1) never_kernel(int* status, int* report, unsigned long long timeout_ns) {
  __shared__ uint64_t bar_a, bar_b;
  __shared__ uint32_t slot;
  __shared__ volatile int abort_flag;
  __shared__ int own_status;   // warp 1's status word (it must stay untouched)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar_a, 1);
    mbar_init(&bar_b, 1);
    abort_flag = 0;
    own_status = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (lane == 0) {
    if (warp == 0) {
      const WaitGuard g{&abort_flag, status, timeout_ns};
      report[0] = mbar_wait(&bar_a, 0, g) ? 0 : 1;
    } else {
      // a much longer limit: only the abort raised by warp 0 can end this wait early
      const WaitGuard g{&abort_flag, &own_status, timeout_ns * 1000ull};
      const bool r = mbar_wait(&bar_b, 0, g);
      report[1] = (!r && own_status == 0) ? 1 : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(slot, 32);
  }
}

}  // namespace

extern "C" {

// Runs never_kernel; status and report are device ints (zeroed by the caller).
int fa_selftest_wait_timeout(int* status, int* report, unsigned long long timeout_ns, void* stream) {
  never_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(status, report, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}


// q, k: bf16 [128, dk] row-major; s: fp32 [128, 128]; status: device int (0 on entry)
int fa_selftest_qk(const void* q, const void* k, int dk, float* s, int* status, void* stream) {
  CUtensorMap mq, mk;
  if (!map2d(&mq, q, dk, 128) || !map2d(&mk, k, dk, 128)) return 7;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int smem = 2 * (dk / 64) * 16384 + 1024 + 64;
  cudaError_t e;
  if (dk == 64) {
    cudaFuncSetAttribute(qk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    qk_kernel<64><<<1, 128, smem, st>>>(mq, mk, s, status);
  } else if (dk == 128) {
    cudaFuncSetAttribute(qk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    qk_kernel<128><<<1, 128, smem, st>>>(mq, mk, s, status);
  } else if (dk == 192) {
    cudaFuncSetAttribute(qk_kernel<192>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    qk_kernel<192><<<1, 128, smem, st>>>(mq, mk, s, status);
  } else if (dk == 256) {
    cudaFuncSetAttribute(qk_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    qk_kernel<256><<<1, 128, smem, st>>>(mq, mk, s, status);
  } else {
    return 2;
  }
  e = cudaGetLastError();
  return e == cudaSuccess ? 0 : 5;
}

// p: bf16 [128, 128]; v: bf16 [128, dv]; o: fp32 [128, dv]
int fa_selftest_pv(const void* p, const void* v, int dv, float* o, int* status, void* stream) {
  CUtensorMap mv;
  if (!map2d(&mv, v, dv, 128)) return 7;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int smem = (dv / 64) * 16384 + 1024 + 64;
  const __nv_bfloat16* pp = static_cast<const __nv_bfloat16*>(p);
  if (dv == 64) {
    cudaFuncSetAttribute(pv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    pv_kernel<64><<<1, 128, smem, st>>>(pp, mv, o, status);
  } else if (dv == 128) {
    cudaFuncSetAttribute(pv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    pv_kernel<128><<<1, 128, smem, st>>>(pp, mv, o, status);
  } else if (dv == 256) {
    cudaFuncSetAttribute(pv_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    pv_kernel<256><<<1, 128, smem, st>>>(pp, mv, o, status);
  } else {
    return 2;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

}  // extern "C"
