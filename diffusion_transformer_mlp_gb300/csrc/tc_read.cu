// The tensor core's own reading of packed E2M1 bytes.
//
// "FC2 NVFP4 Scheduling Results", Canonical Operation: the FC2 operands are
// packed E2M1 elements (two per byte).  Which element of a byte sits in
// which nibble cannot be seen through an E2M1 x E2M1 GEMM: a swap inside
// every byte is the same permutation of K for both operands, and a dot
// product does not change when both of its vectors are permuted alike.  A
// contraction against an operand with one element per byte can see it.
// This kernel runs one tcgen05.mma.kind::f8f6f4 with A = 128 rows of E2M1
// (32 elements, the QDATA bytes under test) and B = the 32 x 32 identity in
// E4M3 (one byte per element, so its element order is the byte order):
// D[r, n] = the value the tensor core takes for element n of row r.
//
// Operand layout in shared memory (K-major, 128-byte swizzle, as the GEMM
// uses): kind::f8f6f4 places a 4-bit operand in the padded form, 16
// elements to a 16-byte unit whose 8 data bytes carry the 16 packed codes.
// The kernel writes those 8 bytes into both halves of the unit, so the
// result does not depend on which half holds the data.
#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int RD_ROWS = 128;   // MMA M: rows of QDATA read at once
constexpr int RD_ELEMS = 32;   // MMA K: elements per row (16 QDATA bytes)
constexpr int RD_N = 32;       // identity columns, one per element
constexpr int RD_SMEM = 1024 + RD_ROWS * 128 + RD_N * 128;
constexpr uint64_t kReadWaitLimitCycles = 2000000000ull;  // about a second

// Instruction descriptor, kind::f8f6f4: D F32 (1 at bit 4), A E2M1 (5 at
// bit 7), B E4M3 (0 at bit 10), both K-major, N>>3 at bit 17, M>>4 at bit 24.
constexpr uint32_t kReadIdesc =
    (1u << 4) | (5u << 7) | (0u << 10) | (uint32_t(RD_N >> 3) << 17) | (uint32_t(RD_ROWS >> 4) << 24);

__device__ __forceinline__ uint64_t desc_sw128_rd(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// 16-byte unit c of row r of a 128-byte-row tile under the 128-byte swizzle.
__device__ __forceinline__ uint4* unit_sw128(uint8_t* tile, int r, int c) {
  return reinterpret_cast<uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(128, 1)
    k_diag_tc_e2m1_read(const uint8_t* __restrict__ qdata, float* __restrict__ out, uint32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* a_tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* b_tile = a_tile + RD_ROWS * 128;
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < (RD_ROWS + RD_N) * 8; i += blockDim.x) reinterpret_cast<uint4*>(a_tile)[i] = zero;
  __syncthreads();
  {
    // row r = threadIdx.x: units 0 and 1 hold elements 0..15 and 16..31
    const int r = threadIdx.x;
    const uint2* src = reinterpret_cast<const uint2*>(qdata + r * (RD_ELEMS / 2));
    const uint2 lo = src[0], hi = src[1];
    *unit_sw128(a_tile, r, 0) = make_uint4(lo.x, lo.y, lo.x, lo.y);
    *unit_sw128(a_tile, r, 1) = make_uint4(hi.x, hi.y, hi.x, hi.y);
    if (r < RD_N) b_tile[r * 128 + (((r >> 4) ^ (r & 7)) << 4) + (r & 15)] = 0x38;  // E4M3 1.0 at element r
  }
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  fence_proxy_async_smem();  // generic-proxy stores -> the tensor core's reads
  if (warp == 0) tmem_alloc(&tmem_slot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {
    // D = A x B^T, no accumulation into what tensor memory held
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(desc_sw128_rd(smem_u32(a_tile))), "l"(desc_sw128_rd(smem_u32(b_tile))), "r"(kReadIdesc), "r"(0)
        : "memory");
    tc_commit(&done);
  }
  __shared__ int ok_s;
  if (threadIdx.x == 0) {
    ok_s = mbar_wait_bounded(&done, 0, kReadWaitLimitCycles, nullptr) ? 1 : 0;
    if (!ok_s && dev_status != nullptr) atomicExch(dev_status, static_cast<uint32_t>(NVFP4_ETIMEOUT));
  }
  __syncthreads();
  tc_fence_after();
  if (ok_s) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tmem + (uint32_t(warp * 32) << 16), v);
    tc_wait_ld();
    tmem_ld_fence_regs<32>(v);
    float* row = out + (warp * 32 + lane) * RD_N;
#pragma unroll
    for (int j = 0; j < RD_N; ++j) row[j] = __uint_as_float(v[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 32);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_diag_tc_e2m1_read(const uint8_t* qdata, float* out, uint32_t* dev_status,
                                                nvfp4_stream_t stream) {
  if (!qdata || !out || !aligned16(qdata) || !aligned16(out))
    return fail(NVFP4_EINVAL, "nvfp4_diag_tc_e2m1_read: pointers must be non-null and 16-byte aligned");
  nvfp4_status st = cuda_check(
      cudaFuncSetAttribute(k_diag_tc_e2m1_read, cudaFuncAttributeMaxDynamicSharedMemorySize, RD_SMEM),
      "cudaFuncSetAttribute(k_diag_tc_e2m1_read)");
  if (st != NVFP4_OK) return st;
  k_diag_tc_e2m1_read<<<1, RD_ROWS, RD_SMEM, reinterpret_cast<cudaStream_t>(stream)>>>(qdata, out, dev_status);
  return cuda_check(cudaGetLastError(), "launch k_diag_tc_e2m1_read");
}
