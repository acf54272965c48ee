// selftest.cu -- libgqa_selftest: single-CTA checks of the sm_103a building
// blocks the prefill kernel is made of, for the GPU test suite only:
//   gqa_selftest_qk  S = A . B^T  (TMA 128B-swizzled loads, K-major smem
//                    descriptors, tcgen05.mma kind::f16, tcgen05.ld; optionally
//                    A copied into TMEM with tcgen05.cp and read from there)
//   gqa_selftest_pv  O = P . V    (P packed to bf16 and stored to TMEM with
//                    tcgen05.st, used as the A operand from TMEM; V MN-major
//                    in 128B-swizzled smem, N = 64 or 128)
// Each runs one CTA on small fixed shapes; shared memory is sized well past
// what the descriptors address.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace {

using namespace gqa;

constexpr uint32_t kHalf = 128u * 128u;   // 128 rows x 128 bytes

// S[128][128] = A[128][64] . B[128][64]^T.  use_cp: A is first copied from
// shared memory into TMEM with tcgen05.cp and read by the MMA from there.
__global__ void __launch_bounds__(128, 1)
    qk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, float* S,
              int use_cp) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sb = smem_raw + (base - raw);
  const uint32_t a_s = base, b_s = base + kHalf;
  const uint32_t bar_ld = base + 4 * kHalf, bar_mma = bar_ld + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sb + 4 * kHalf + 16);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  volatile int no_abort = 0;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar_ld, 2 * kHalf);
    tma_load_4d(a_s, &tmA, bar_ld, 0, 0, 0, 0);
    tma_load_4d(b_s, &tmB, bar_ld, 0, 0, 0, 0);
    mbar_wait(bar_ld, 0, &no_abort, 1000000000ull);
    tc_fence_after();
    const uint32_t idesc = make_idesc_bf16(128, 128, 0, 0);
    if (use_cp) {
      for (int ks = 0; ks < 4; ++ks) tmem_cp_128x256b(tmem + 128 + ks * 8, make_sdesc_sw128(a_s + ks * 32, 16, 1024));
      for (int ks = 0; ks < 4; ++ks)
        umma_ts(tmem, tmem + 128 + ks * 8, make_sdesc_sw128(b_s + ks * 32, 16, 1024), idesc, ks > 0);
    } else {
      for (int ks = 0; ks < 4; ++ks)
        umma_ss(tmem, make_sdesc_sw128(a_s + ks * 32, 16, 1024), make_sdesc_sw128(b_s + ks * 32, 16, 1024), idesc,
                ks > 0);
    }
    umma_commit(bar_mma);
  }
  __syncwarp();
  mbar_wait(bar_mma, 0, &no_abort, 1000000000ull);
  tc_fence_after();
  const int row = threadIdx.x;
  const uint32_t taddr = tmem + (uint32_t(warp * 32) << 16);
  for (int c = 0; c < 128; c += 32) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + c, v);
    tmem_ld_wait_x32(v);
    for (int i = 0; i < 32; ++i) S[row * 128 + c + i] = __uint_as_float(v[i]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// O[128][N] = P[128][128] . V[128][N]; V loaded as N/64 halves [128 keys][64]
template <int N>
__global__ void __launch_bounds__(128, 1)
    pv_kernel(const __grid_constant__ CUtensorMap tmV, const float* P, float* O, uint32_t lbo, uint32_t sbo) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sb = smem_raw + (base - raw);
  const uint32_t v_s = base;
  const uint32_t bar_ld = base + 8 * kHalf, bar_mma = bar_ld + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sb + 8 * kHalf + 16);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const int row = threadIdx.x;
  const uint32_t lane_base = uint32_t(warp * 32) << 16;
  // P row -> packed bf16 pairs in TMEM columns [0, 64)
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
    for (int i = 0; i < 16; ++i) {
      const int k0 = q * 32 + 2 * i;
      pk[i] = pack_bf16x2(P[row * 128 + k0], P[row * 128 + k0 + 1]);
    }
    tmem_st_32x32b_x16(tmem + lane_base + q * 16, pk);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  volatile int no_abort = 0;
  if (threadIdx.x == 0) {
    tc_fence_after();
    mbar_arrive_expect_tx(bar_ld, (N / 64) * kHalf);
    for (int h = 0; h < N / 64; ++h) tma_load_4d(v_s + h * kHalf, &tmV, bar_ld, h * 64, 0, 0, 0);
    mbar_wait(bar_ld, 0, &no_abort, 1000000000ull);
    const uint32_t idesc = make_idesc_bf16(128, N, 0, 1);
    for (int ks = 0; ks < 8; ++ks)
      umma_ts(tmem + 128, tmem + ks * 8, make_sdesc_sw128(v_s + ks * 2048, lbo, sbo), idesc, ks > 0);
    umma_commit(bar_mma);
  }
  __syncwarp();
  mbar_wait(bar_mma, 0, &no_abort, 1000000000ull);
  tc_fence_after();
  for (int c = 0; c < N; c += 32) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tmem + lane_base + 128 + c, v);
    tmem_ld_wait_x32(v);
    for (int i = 0; i < 32; ++i) O[row * N + c + i] = __uint_as_float(v[i]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// [rows][cols] bf16 row-major as a 4-D map (cols, rows, 1, 1), box (64, 128, 1, 1)
bool map_2d(CUtensorMap* m, const void* p, int rows, int cols) {
  void* fnp = nullptr;
  cudaDriverEntryPointQueryResult qr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &qr) !=
          cudaSuccess ||
      qr != cudaDriverEntryPointSuccess)
    return false;
  auto fn = reinterpret_cast<EncodeTiledFn>(fnp);
  const cuuint64_t dims[4] = {cuuint64_t(cols), cuuint64_t(rows), 1, 1};
  const cuuint64_t strides[3] = {cuuint64_t(cols) * 2, cuuint64_t(cols) * rows * 2, cuuint64_t(cols) * rows * 2};
  const cuuint32_t box[4] = {64, 128, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

// A, B: device bf16 [128][64]; S: device fp32 [128][128].  use_cp: A reaches
// the MMA through TMEM (tcgen05.cp) instead of shared memory.  Synchronous.
int gqa_selftest_qk(const void* A, const void* B, float* S, int use_cp) {
  CUtensorMap ma, mb;
  if (!map_2d(&ma, A, 128, 64) || !map_2d(&mb, B, 128, 64)) return 3;
  const int smem = 4 * kHalf + 1024 + 64;
  if (cudaFuncSetAttribute(qk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 3;
  qk_kernel<<<1, 128, smem>>>(ma, mb, S, use_cp ? 1 : 0);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

// P: device fp32 [128][128]; V: device bf16 [128][N]; O: device fp32 [128][N];
// N = 64 or 128.  lbo/sbo: byte offsets of the MN-major V descriptor.  Synchronous.
int gqa_selftest_pv(const float* P, const void* V, float* O, int N, unsigned lbo, unsigned sbo) {
  if (N != 64 && N != 128) return 1;
  if (lbo > 2 * kHalf || sbo > 2 * kHalf) return 1;   // keeps every read inside the 8 * kHalf V area
  CUtensorMap mv;
  if (!map_2d(&mv, V, 128, N)) return 3;
  const int smem = 8 * kHalf + 1024 + 64;
  if (N == 64) {
    if (cudaFuncSetAttribute(pv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return 3;
    pv_kernel<64><<<1, 128, smem>>>(mv, P, O, lbo, sbo);
  } else {
    if (cudaFuncSetAttribute(pv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return 3;
    pv_kernel<128><<<1, 128, smem>>>(mv, P, O, lbo, sbo);
  }
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
