// Dense NVFP4 tensor-core throughput loop: the denominator of the GEMM's
// roofline, measured on the part itself.
//
// "FC2 NVFP4 Scheduling Results", Canonical Operation: the FC2 is a dense
// E2M1 x E2M1 contraction with vector-16 UE4M3 block scales and FP32
// accumulation.  k_fc2_gemm runs it as tcgen05.mma.cta_group::2
// .kind::mxf4nvf4 (M=256, N=256, K=64 per instruction); this kernel issues
// that same instruction back to back, with nothing else in the tensor pipe
// and operands that never leave shared memory, so its rate is the most the
// GEMM's MMAs can reach on this GPU at the clocks it runs at.
//
// Each CTA pair: both CTAs fill two 16 KB operand tiles (128 rows x 128
// bytes, 128-byte swizzle, the GEMM's K-major layout) with fixed
// pseudo-random bytes and store their scale columns (UE4M3 1.0) into tensor
// memory once; one thread of the leader CTA then issues `iters` MMAs,
// cycling through the four K=64 slices of the tile, commits once, and both
// CTAs wait (bounded) for the commit before freeing tensor memory.
#include <cstdio>

#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int PEAK_THREADS = 128;            // four warps: one per TMEM lane quarter
constexpr int TILE_BYTES = 128 * 128;        // 128 rows x 256 E2M1 codes
constexpr uint32_t PEAK_TMEM_COLS = 512;     // accumulator 0..255, scales 256..351
constexpr uint32_t SCALE_COL = 256;          // A scales: 4 columns per K=64 slice
constexpr uint32_t SCALE_W_COL = SCALE_COL + 32;  // W scales: 8 columns per slice
// Far more dynamic shared memory than the two tiles need: two CTAs never
// share an SM, so no two pairs contend for one SM's tensor memory.
constexpr int PEAK_SMEM = 160 * 1024;
static_assert(1024 + 2 * TILE_BYTES <= PEAK_SMEM && 2 * PEAK_SMEM > 233472, "one CTA per SM");
constexpr uint64_t kPeakWaitLimitCycles = 4000000000ull;  // about 2 s at the highest SM clock
constexpr int64_t kMaxIters = int64_t(1) << 22;           // at 128 cycles each, well inside the wait

// kind::mxf4nvf4 instruction descriptor: A and B E2M1 (format 1 at bits 7
// and 10), both K-major, UE4M3 scales, N/8 at bit 17, M/16 at bit 24.
constexpr uint32_t kPeakIdesc = (1u << 7) | (1u << 10) | (uint32_t(256 >> 3) << 17) | (uint32_t(256 >> 4) << 24);

// Shared-memory descriptor of a K-major tile with 128-byte rows and the
// 128-byte swizzle: start address >> 4, leading offset 1 (unused when
// swizzled), 8-row groups 1024 bytes apart, descriptor version 1, SWIZZLE_128B.
__device__ __forceinline__ uint64_t peak_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PEAK_THREADS, 1)
    k_diag_mma_peak(int64_t iters, uint64_t limit_cycles, uint32_t* dev_status, uint64_t* clk) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  // operand bytes: a multiplicative hash of the word index, different per CTA
  for (int i = threadIdx.x; i < 2 * TILE_BYTES / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(tiles)[i] = (uint32_t(i) + 0x9E37u * (rank + 1u)) * 2654435761u;
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's reads
  if (warp == 0) tmem_alloc_pair(&tmem_slot, PEAK_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  {
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0x38383838u;  // four UE4M3 1.0
    const uint32_t quarter = uint32_t(warp * 32) << 16;
#pragma unroll
    for (int c = 0; c < 3; ++c) tmem_st_32x32b_x32(tmem + quarter + SCALE_COL + 32 * c, v);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' tiles and scales are in place
  tc_fence_after();
  if (rank == 0 && threadIdx.x == 0) {
    if (clk != nullptr && blockIdx.x == 0) {
      clk[0] = globaltimer_ns();
      clk[2] = clock64();
    }
    const uint64_t a_desc = peak_desc(smem_u32(tiles)), b_desc = peak_desc(smem_u32(tiles + TILE_BYTES));
    for (int64_t i = 0; i < iters; ++i) {
      const uint32_t j = uint32_t(i & 3);  // K=64 slice: 32 bytes into each 128-byte row
      tc_mma_pair_nvf4(tmem, a_desc + 2 * j, b_desc + 2 * j, kPeakIdesc, tmem + SCALE_COL + 4 * j,
                       tmem + SCALE_W_COL + 8 * j, i != 0);
    }
    tc_commit_pair(&done);
  }
  // each CTA sees the commit before the pair frees its tensor memory
  if (threadIdx.x == 32) {
    if (!mbar_wait_bounded(&done, 0, limit_cycles, nullptr) && dev_status != nullptr)
      atomicExch(dev_status, static_cast<uint32_t>(NVFP4_ETIMEOUT));
    if (clk != nullptr && blockIdx.x == 0) {  // the same SM as the start record
      clk[1] = globaltimer_ns();
      clk[3] = clock64();
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem, PEAK_TMEM_COLS);
}

// SM pairs that run the loop at once: SMs / 2, or fewer if the GPU cannot
// hold that many two-CTA clusters of this kernel together.
nvfp4_status mma_peak_pairs(int* pairs) {
  nvfp4_status st = cuda_check(
      cudaFuncSetAttribute(k_diag_mma_peak, cudaFuncAttributeMaxDynamicSharedMemorySize, PEAK_SMEM),
      "cudaFuncSetAttribute(k_diag_mma_peak)");
  if (st != NVFP4_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count() / 2));
  cfg.blockDim = dim3(PEAK_THREADS);
  cfg.dynamicSmemBytes = PEAK_SMEM;
  int clusters = 0;
  st = cuda_check(cudaOccupancyMaxActiveClusters(&clusters, k_diag_mma_peak, &cfg),
                  "cudaOccupancyMaxActiveClusters(k_diag_mma_peak)");
  if (st != NVFP4_OK) return st;
  *pairs = clusters < sm_count() / 2 ? clusters : sm_count() / 2;
  return *pairs >= 1 ? NVFP4_OK : fail(NVFP4_ECUDA, "nvfp4_diag_mma_peak: no two-CTA cluster fits");
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" int64_t nvfp4_diag_mma_peak_pairs(void) {
  int pairs = 0;
  return mma_peak_pairs(&pairs) == NVFP4_OK ? pairs : -1;
}

extern "C" nvfp4_status nvfp4_diag_mma_peak(int64_t iters, uint32_t* dev_status, uint64_t* clk,
                                            nvfp4_stream_t stream) {
  if (iters < 1 || iters > kMaxIters) return fail(NVFP4_EINVAL, "nvfp4_diag_mma_peak: iters outside 1 .. 2^22");
  if (reinterpret_cast<uintptr_t>(clk) % 8 != 0)
    return fail(NVFP4_EINVAL, "nvfp4_diag_mma_peak: clk must be 8-byte aligned");
  int pairs = 0;
  nvfp4_status st = mma_peak_pairs(&pairs);
  if (st != NVFP4_OK) return st;
  k_diag_mma_peak<<<2 * pairs, PEAK_THREADS, PEAK_SMEM, reinterpret_cast<cudaStream_t>(stream)>>>(
      iters, kPeakWaitLimitCycles, dev_status, clk);
  return cuda_check(cudaGetLastError(), "launch k_diag_mma_peak");
}
