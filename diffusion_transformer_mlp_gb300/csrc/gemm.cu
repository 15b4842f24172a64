// Persistent block-scaled NVFP4 GEMM for sm_103a (tcgen05 + TMA + TMEM).
//
// "FC2 NVFP4 Scheduling Results": Canonical Operation (M=37,810 -> padded,
// N=5,376, K=14,336; E2M1 operands with vector-16 UE4M3 scales; FP32
// accumulation; BF16 output), Decision (split-K 1, zero workspace),
// Traffic Attribution (the weight is re-read once per 128-row M tile, 296x,
// and the activation about 42x; the winning schedule keeps those re-reads
// in L2; no global atomics, no reduction traffic, one output write).
// The pages' kernel is a GB10 warp-MMA library kernel; this one is written
// for the datacenter Blackwell tensor core instead:
//
//   warp 0      TMA producer: per k-tile (256 K elements) one 128x128-byte
//               A tile and one W tile (128B swizzle) plus the two 2 KB
//               block-scale chunks (already in the tiled layout the tensor
//               core reads), into a STAGES-deep shared-memory ring.
//   warp 1      MMA issuer: tcgen05.cp of the scale chunks into tensor
//               memory, four tcgen05.mma kind::mxf4nvf4 (K=64 each) per
//               k-tile into a 128x128 FP32 accumulator in tensor memory;
//               two accumulators so the epilogue of tile i overlaps the
//               main loop of tile i+1.
//   warps 2-5   epilogue: tcgen05.ld, multiply by alpha = gA*gW, round to
//               BF16, stage through 128B-swizzled shared memory, TMA store
//               (clipped at row M).
//
// Tiles are walked M-panel-major (all N tiles of one 128-row panel, then
// the next), so the CTAs running at any moment share a few activation
// panels and the whole 43 MB weight through L2.  K is reduced in increasing
// order inside one CTA: no split-K, no workspace, no atomics, and an output
// row does not depend on M.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK_BYTES = 128;  // 256 E2M1 elements
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BK_BYTES;
constexpr int B_BYTES = BN * BK_BYTES;
constexpr int SF_BYTES = 2048;  // 128 rows x 16 scales (four 512-byte 128x4 tiles)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * SF_BYTES;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BYTES = EPI_WARPS * 32 * BN * 2;  // per warp: 32 rows x 128 BF16
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;    // two 128-column FP32 accumulators
constexpr uint32_t SF_COL = 256;   // per stage: 16 columns of A scales, 16 of W scales
static_assert(SF_COL + STAGES * 32 <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0, "stage alignment for 128B swizzle");

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1), both
// K-major, UE4M3 scales (scale format 0), scale-factor ids 0, N>>3 at bit
// 17, M>>4 at bit 24.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes with the 128-byte swizzle: 8-row atoms 1024 bytes apart (SBO),
// descriptor version 1, layout SWIZZLE_128B (2).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// Descriptor for tcgen05.cp of a 32-row x 16-byte block: rows 16 bytes
// apart, 8-row core matrices 128 bytes apart, no swizzle.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(128 >> 4) << 32) | (uint64_t(1) << 46);
}

struct Smem {
  uint8_t* stage;  // STAGES x [A | B | SFA | SFB]
  uint8_t* epi;    // EPI_WARPS x 8 KB
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* mma_done;
  uint32_t* tmem_slot;
  int* abort_flag;
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stage = base;
  s.epi = base + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.epi + EPI_BYTES);
  s.full = bars;
  s.empty = bars + STAGES;
  s.tfull = bars + 2 * STAGES;
  s.tempty = bars + 2 * STAGES + 2;
  s.mma_done = bars + 2 * STAGES + 4;
  s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  return s;
}

struct Params {
  const uint8_t* a_s;
  const uint8_t* w_s;
  const nvfp4_scale_rec* a_rec;
  const nvfp4_scale_rec* w_rec;
  int num_m_tiles, num_n_tiles, num_k_tiles;
  int64_t sf_panel_bytes;  // bytes of scales per 128-row panel: (C4/4) * 512
  uint32_t* dev_status;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void report_timeout(const Params& p, int* abort_flag) {
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  if (p.dev_status != nullptr) atomicExch(p.dev_status, static_cast<uint32_t>(NVFP4_ETIMEOUT));
}

__global__ void __launch_bounds__(THREADS, 1)
    k_fc2_gemm(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
               const __grid_constant__ CUtensorMap tmap_out, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const volatile int* abort_flag = sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], 1);
      mbar_init(&sm.tempty[b], EPI_WARPS);
    }
    mbar_init(sm.mma_done, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_out);
  }
  if (warp == 1) tmem_alloc(sm.tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();
      const uint64_t pol_a = l2_policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // last issued phase per stage
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        const int mb = t / p.num_n_tiles, nb = t - (t / p.num_n_tiles) * p.num_n_tiles;
        const uint8_t* sfa = p.a_s + mb * p.sf_panel_bytes;
        const uint8_t* sfw = p.w_s + nb * p.sf_panel_bytes;
        for (int kt = 0; kt < p.num_k_tiles; ++kt) {
          if (!mbar_wait_bounded(&sm.empty[stage], phase ^ 1u, p.wait_limit_ns, abort_flag)) {
            report_timeout(p, sm.abort_flag);
            ok = false;
            break;
          }
          uint8_t* st = sm.stage + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&sm.full[stage], STAGE_BYTES);
          tma_load_2d(st, &tmap_a, &sm.full[stage], kt * BK_BYTES, mb * BM, pol_a);
          tma_load_2d(st + A_BYTES, &tmap_w, &sm.full[stage], kt * BK_BYTES, nb * BN, pol_w);
          bulk_load(st + A_BYTES + B_BYTES, sfa + kt * SF_BYTES, SF_BYTES, &sm.full[stage], pol_a);
          bulk_load(st + A_BYTES + B_BYTES + SF_BYTES, sfw + kt * SF_BYTES, SF_BYTES, &sm.full[stage], pol_w);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy this thread issued must have landed before the CTA exits
      // (they have, on the normal path: the MMA warp consumed them).
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s))
          if (!mbar_wait_bounded(&sm.full[s], (issued_parity >> s) & 1u, p.wait_limit_ns, nullptr))
            report_timeout(p, sm.abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
        const uint32_t acc = local & 1;
        if (!mbar_wait_bounded(&sm.tempty[acc], ((local >> 1) & 1) ^ 1u, p.wait_limit_ns, abort_flag)) {
          report_timeout(p, sm.abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + ACC_COL + acc * BN;
        for (int kt = 0; kt < p.num_k_tiles; ++kt) {
          if (!mbar_wait_bounded(&sm.full[stage], phase, p.wait_limit_ns, abort_flag)) {
            report_timeout(p, sm.abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = sm.stage + stage * STAGE_BYTES;
          const uint32_t a_addr = smem_u32(st), b_addr = smem_u32(st + A_BYTES);
          const uint32_t sfa_addr = smem_u32(st + A_BYTES + B_BYTES);
          const uint32_t sfb_addr = sfa_addr + SF_BYTES;
          const uint32_t sf_tmem = tmem + SF_COL + stage * 32;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_cp_32x128b_warpx4(sf_tmem + 4 * j, desc_sf(sfa_addr + 512 * j));
            tc_cp_32x128b_warpx4(sf_tmem + 16 + 4 * j, desc_sf(sfb_addr + 512 * j));
          }
          const uint64_t a_desc = desc_sw128(a_addr), b_desc = desc_sw128(b_addr);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // K step j: 64 elements = 32 bytes further along the swizzled row
            tc_mma_nvf4(d_tmem, a_desc + 2 * j, b_desc + 2 * j, kIdesc, sf_tmem + 4 * j, sf_tmem + 16 + 4 * j,
                        (kt | j) != 0);
          }
          tc_commit(&sm.empty[stage]);  // frees the stage once these MMAs complete
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&sm.tfull[acc]);  // accumulator ready once all MMAs complete
      }
      // Nothing may still be reading shared memory or writing tensor memory
      // when the CTA tears down.
      tc_commit(sm.mma_done);
      if (!mbar_wait_bounded(sm.mma_done, 0, p.wait_limit_ns, nullptr)) report_timeout(p, sm.abort_flag);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const float alpha = __fmul_rn(p.a_rec->global_scale, p.w_rec->global_scale);
    uint8_t* stg = sm.epi + q * (32 * BN * 2);
    int local = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
      const int mb = t / p.num_n_tiles, nb = t - (t / p.num_n_tiles) * p.num_n_tiles;
      const uint32_t acc = local & 1;
      // one lane waits, the warp follows its verdict (tcgen05.ld is warp-wide)
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&sm.tfull[acc], (local >> 1) & 1, p.wait_limit_ns, abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) report_timeout(p, sm.abort_flag);
        break;
      }
      tc_fence_after();
      // the previous TMA store must have finished reading the staging buffer
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      const uint32_t row_tmem = tmem + (uint32_t(q * 32) << 16) + ACC_COL + acc * BN;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
              "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
              "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(row_tmem + c * 32));
        tc_wait_ld();
        // row `lane` of this quarter, columns 32c..32c+31 -> 4 chunks of 16 B
        uint8_t* half = stg + (c >> 1) * (32 * 128) + lane * 128;
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __fmul_rn(__uint_as_float(r[t4 * 8 + 2 * i]), alpha);
            const float hi = __fmul_rn(__uint_as_float(r[t4 * 8 + 2 * i + 1]), alpha);
            const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
            w[i] = *reinterpret_cast<const uint32_t*>(&v);
          }
          const int chunk = ((c & 1) * 4 + t4) ^ (lane & 7);
          *reinterpret_cast<uint4*>(half + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // accumulator drained: hand it back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tempty[acc]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int y = mb * BM + q * 32;
        tma_store_2d(&tmap_out, stg, nb * BN, y);
        tma_store_2d(&tmap_out, stg + 32 * 128, nb * BN + 64, y);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host: tensor maps ------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
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

nvfp4_status make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(NVFP4_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, int(r));
    return fail(NVFP4_ECUDA, buf);
  }
  return NVFP4_OK;
}

}  // namespace

// Default bounded-wait limit: far above any legitimate wait (a whole
// canonical GEMM takes about a millisecond) yet short enough that a broken
// pipeline returns control instead of holding the GPU.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;

nvfp4_status fc2_gemm_launch(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec, const void* w_q,
                             const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m, int64_t n, int64_t k,
                             void* out, int64_t ldo, uint32_t* dev_status, cudaStream_t stream,
                             uint64_t wait_limit_ns) {
  if (!a_q || !a_s || !a_rec || !w_q || !w_s || !w_rec || !out)
    return fail(NVFP4_EINVAL, "nvfp4_fc2_gemm: null pointer");
  if (m < 1) return fail(NVFP4_EINVAL, "nvfp4_fc2_gemm: m must be >= 1");
  if (n < BN || n % BN != 0) return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_gemm: n must be a positive multiple of 128");
  if (k < 256 || k % 256 != 0) return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_gemm: k must be a positive multiple of 256");
  if (ldo < n) return fail(NVFP4_EINVAL, "nvfp4_fc2_gemm: ldo < n");
  if (ldo % 8 != 0 || !aligned16(a_q) || !aligned16(a_s) || !aligned16(w_q) || !aligned16(w_s) || !aligned16(out) ||
      !aligned16(a_rec) || !aligned16(w_rec))
    return fail(NVFP4_EALIGN, "nvfp4_fc2_gemm: pointers must be 16-byte aligned and ldo a multiple of 8");
  const int64_t m_pad = nvfp4_padded_rows(m);
  if (m_pad / BM > (int64_t(1) << 24) || n > (int64_t(1) << 24) || k > (int64_t(1) << 24))
    return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_gemm: problem too large");

  CUtensorMap ta, tw, to;
  nvfp4_status st;
  if ((st = make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_q, k / 2, m_pad, k / 2, BK_BYTES, BM, "A")) != NVFP4_OK)
    return st;
  if ((st = make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_q, k / 2, n, k / 2, BK_BYTES, BN, "W")) != NVFP4_OK)
    return st;
  if ((st = make_map_2d(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, n, m, ldo * 2, 64, 32, "out")) != NVFP4_OK)
    return st;

  Params prm;
  prm.a_s = static_cast<const uint8_t*>(a_s);
  prm.w_s = static_cast<const uint8_t*>(w_s);
  prm.a_rec = a_rec;
  prm.w_rec = w_rec;
  prm.num_m_tiles = static_cast<int>(m_pad / BM);
  prm.num_n_tiles = static_cast<int>(n / BN);
  prm.num_k_tiles = static_cast<int>(k / 256);
  prm.sf_panel_bytes = (k / 16 / 4) * 512;
  prm.dev_status = dev_status;
  prm.wait_limit_ns = wait_limit_ns;

  st = cuda_check(cudaFuncSetAttribute(k_fc2_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES),
                  "cudaFuncSetAttribute(k_fc2_gemm)");
  if (st != NVFP4_OK) return st;
  const int tiles = prm.num_m_tiles * prm.num_n_tiles;
  const int grid = tiles < sm_count() ? tiles : sm_count();
  k_fc2_gemm<<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tw, to, prm);
  return cuda_check(cudaGetLastError(), "launch k_fc2_gemm");
}

// ---- diagnostics: the bounded wait on a barrier nothing arrives at ---------

namespace {
__global__ void k_diag_wait_timeout(uint64_t limit_ns, uint32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0, limit_ns, &abort_flag)) *dev_status = NVFP4_ETIMEOUT;
    else *dev_status = NVFP4_OK;
    mbar_arrive(&bar);  // complete the phase so the barrier is left idle
  }
}
}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_fc2_gemm(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                                       const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m,
                                       int64_t n, int64_t k, void* out_bf16, int64_t ldo, uint32_t* dev_status,
                                       nvfp4_stream_t stream) {
  return fc2_gemm_launch(a_q, a_s, a_rec, w_q, w_s, w_rec, m, n, k, out_bf16, ldo, dev_status,
                         reinterpret_cast<cudaStream_t>(stream), kDefaultWaitLimitNs);
}

extern "C" nvfp4_status nvfp4_diag_wait_timeout(uint64_t limit_ns, uint32_t* dev_status, nvfp4_stream_t stream) {
  if (!dev_status || limit_ns < 1 || limit_ns > 1000000000ull)
    return fail(NVFP4_EINVAL, "nvfp4_diag_wait_timeout: bad arguments");
  k_diag_wait_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, dev_status);
  return cuda_check(cudaGetLastError(), "launch k_diag_wait_timeout");
}
