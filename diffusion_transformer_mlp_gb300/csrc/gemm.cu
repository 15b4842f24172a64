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

// Tile of one CTA pair: 256 rows of A x 256 rows of W (256 x 256 outputs);
// each CTA holds 128 rows of A and 128 rows of W per stage and 128 x 256
// FP32 accumulators in its tensor memory.
constexpr int PAIR_M = 256;
constexpr int PAIR_N = 256;
constexpr int HALF = 128;
constexpr int BK_BYTES = 128;  // 256 E2M1 elements per k-tile
constexpr int KT = 2;          // k-tiles per pipeline stage (one TMA box per operand per stage)
constexpr int STAGES = 2;
constexpr int KTILE_BYTES = HALF * BK_BYTES;   // 16 KB: 128 rows x one k-tile
constexpr int A_BYTES = KT * KTILE_BYTES;      // this CTA's 128 A rows x KT k-tiles
constexpr int B_BYTES = KT * KTILE_BYTES;      // this CTA's 128 W rows x KT k-tiles
constexpr int SFA_BYTES = KT * 2048;           // this CTA's 128 rows x 16 scales per k-tile
constexpr int SFB_PANEL = KT * 2048;           // one 128-row W panel
constexpr int SFB_BYTES = 2 * SFB_PANEL;       // all 256 W rows of the tile
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // 76 KB
constexpr int EPI_WARPS = 4;
constexpr int EPI_BYTES = HALF * PAIR_N * 2;   // 128 rows x 256 BF16
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;     // 256 FP32 columns
constexpr uint32_t SF_COL = 256;    // per stage and k-tile: 16 columns of A scales, 32 of W scales
constexpr uint32_t SF_STAGE_COLS = 48 * KT;
static_assert(SF_COL + STAGES * SF_STAGE_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0, "stage alignment for 128B swizzle");

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1), both
// K-major, UE4M3 scales (scale format 0), scale-factor ids 0, N>>3 at bit
// 17, M>>4 at bit 24; M = 256 across the CTA pair.
constexpr uint32_t kIdesc =
    (1u << 7) | (1u << 10) | (uint32_t(PAIR_N >> 3) << 17) | (uint32_t(PAIR_M >> 4) << 24);

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
  uint8_t* epi;    // EPI_WARPS x 32 rows x 256 BF16
  uint64_t* full;  // used in the leader CTA only
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;  // used in the leader CTA only
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
  s.tempty = bars + 2 * STAGES + 1;
  s.mma_done = bars + 2 * STAGES + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 3);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  return s;
}

struct Params {
  const nvfp4_scale_rec* a_rec;
  const nvfp4_scale_rec* w_rec;
  int a_rows;       // padded rows of the activation (multiple of 128)
  int n;            // weight rows (multiple of 128)
  int num_m_tiles;  // ceil(a_rows / 256)
  int num_n_tiles;  // ceil(n / 256)
  int num_stages_k; // ceil(k / 256 / KT)
  int sf_panel_rows;  // rows of 256 B per 128-row scale panel: k / 32
  uint32_t* dev_status;
  uint64_t wait_limit_cycles;
};

__device__ __forceinline__ void report_timeout(const Params& p, int* abort_flag) {
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  if (p.dev_status != nullptr) atomicExch(p.dev_status, static_cast<uint32_t>(NVFP4_ETIMEOUT));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k_fc2_gemm(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
               const __grid_constant__ CUtensorMap tmap_sa, const __grid_constant__ CUtensorMap tmap_sw,
               const __grid_constant__ CUtensorMap tmap_out, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  const volatile int* abort_flag = sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(sm.tfull, 1);
    mbar_init(sm.tempty, 2 * EPI_WARPS);
    mbar_init(sm.mma_done, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_sa);
    prefetch_tmap(&tmap_sw);
    prefetch_tmap(&tmap_out);
  }
  if (warp == 1) tmem_alloc_pair(sm.tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated in both
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();
      const uint64_t pol_a = l2_policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs) {
        const int mt = t / p.num_n_tiles, nt = t - (t / p.num_n_tiles) * p.num_n_tiles;
        // Boxes beyond the operands (the last M or N half) are zero-filled by
        // the TMA and still count their full bytes, so every stage carries
        // 2 x STAGE_BYTES for the leader's barrier.
        const int a_row = mt * PAIR_M + int(rank) * HALF;
        const int b_row = nt * PAIR_N + int(rank) * HALF;
        const int sfa_row0 = (a_row / HALF) * p.sf_panel_rows;
        for (int ks = 0; ks < p.num_stages_k; ++ks) {
          if (!mbar_wait_bounded(&sm.empty[stage], phase ^ 1u, p.wait_limit_cycles, abort_flag)) {
            report_timeout(p, sm.abort_flag);
            ok = false;
            break;
          }
          uint8_t* st = sm.stage + stage * STAGE_BYTES;
          const uint32_t full_leader = mapa_shared(smem_u32(&sm.full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2 * STAGE_BYTES);
          tma_load_3d_pair(st, &tmap_a, full_leader, 0, a_row, ks * KT, pol_a);
          tma_load_3d_pair(st + A_BYTES, &tmap_w, full_leader, 0, b_row, ks * KT, pol_w);
          tma_load_2d_pair(st + A_BYTES + B_BYTES, &tmap_sa, full_leader, 0, sfa_row0 + ks * KT * 8, pol_a);
          tma_load_3d_pair(st + A_BYTES + B_BYTES + SFA_BYTES, &tmap_sw, full_leader, 0, ks * KT * 8, nt * 2, pol_w);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs, ++local) {
        if (!mbar_wait_bounded(sm.tempty, (local & 1) ^ 1u, p.wait_limit_cycles, abort_flag)) {
          report_timeout(p, sm.abort_flag);
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < p.num_stages_k; ++ks) {
          if (!mbar_wait_bounded(&sm.full[stage], phase, p.wait_limit_cycles, abort_flag)) {
            report_timeout(p, sm.abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = sm.stage + stage * STAGE_BYTES;
          const uint32_t a_addr = smem_u32(st), b_addr = smem_u32(st + A_BYTES);
          const uint32_t sfa_addr = smem_u32(st + A_BYTES + B_BYTES);
          const uint32_t sfb_addr = sfa_addr + SFA_BYTES;
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            const uint32_t sfa_tmem = tmem + SF_COL + stage * SF_STAGE_COLS + kk * 48;
            const uint32_t sfb_tmem = sfa_tmem + 16;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tc_cp_pair_32x128b_warpx4(sfa_tmem + 4 * j, desc_sf(sfa_addr + kk * 2048 + 512 * j));
              tc_cp_pair_32x128b_warpx4(sfb_tmem + 8 * j, desc_sf(sfb_addr + kk * 2048 + 512 * j));
              tc_cp_pair_32x128b_warpx4(sfb_tmem + 8 * j + 4, desc_sf(sfb_addr + SFB_PANEL + kk * 2048 + 512 * j));
            }
            const uint64_t a_desc = desc_sw128(a_addr + kk * KTILE_BYTES), b_desc = desc_sw128(b_addr + kk * KTILE_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // K step j: 64 elements = 32 bytes further along the swizzled row
              tc_mma_pair_nvf4(tmem + ACC_COL, a_desc + 2 * j, b_desc + 2 * j, kIdesc, sfa_tmem + 4 * j,
                               sfb_tmem + 8 * j, (ks | kk | j) != 0);
            }
          }
          tc_commit_pair(&sm.empty[stage]);  // frees the stage in both CTAs once these MMAs complete
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(sm.tfull);  // accumulators of both CTAs ready
      }
      // Nothing may still be reading shared memory or writing tensor memory
      // in either CTA when the pair tears down.
      tc_commit_pair(sm.mma_done);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const float alpha = __fmul_rn(p.a_rec->global_scale, p.w_rec->global_scale);
    uint8_t* stg = sm.epi + q * (32 * PAIR_N * 2);
    const uint32_t tempty_leader = mapa_shared(smem_u32(sm.tempty), 0);
    int local = 0;
    for (int t = pair; t < num_tiles; t += num_pairs, ++local) {
      const int mt = t / p.num_n_tiles, nt = t - (t / p.num_n_tiles) * p.num_n_tiles;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(sm.tfull, local & 1, p.wait_limit_cycles, abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) report_timeout(p, sm.abort_flag);
        break;
      }
      tc_fence_after();
      if (lane == 0) bulk_wait_read_all();  // previous stores have read the staging buffer
      __syncwarp();
      const uint32_t row_tmem = tmem + (uint32_t(q * 32) << 16) + ACC_COL;
#pragma unroll 1
      for (int c = 0; c < PAIR_N / 32; ++c) {
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
        uint8_t* sub = stg + (c >> 1) * (32 * 128) + lane * 128;
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __fmul_rn(__uint_as_float(r[t4 * 8 + 2 * i]), alpha);
            const float hi = __fmul_rn(__uint_as_float(r[t4 * 8 + 2 * i + 1]), alpha);
            w[i] = bf16x2_rn(lo, hi);
          }
          const int chunk = ((c & 1) * 4 + t4) ^ (lane & 7);
          *reinterpret_cast<uint4*>(sub + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // accumulator drained: hand it back to the MMA issuer of the pair
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int y = mt * PAIR_M + int(rank) * HALF + q * 32;
        if (y < p.a_rows) {
#pragma unroll
          for (int h = 0; h < PAIR_N / 64; ++h) {
            const int x = nt * PAIR_N + h * 64;
            if (x < p.n) tma_store_2d(&tmap_out, stg + h * (32 * 128), x, y);
          }
        }
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  // teardown: every MMA of the pair has completed before tensor memory is freed
  if (warp == 1 && lane == 0) {
    if (!mbar_wait_bounded(sm.mma_done, 0, p.wait_limit_cycles, nullptr)) report_timeout(p, sm.abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem, TMEM_COLS);
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

nvfp4_status make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(NVFP4_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, dt, cuuint32_t(rank), const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, int(r));
    return fail(NVFP4_ECUDA, buf);
  }
  return NVFP4_OK;
}

}  // namespace

// Default bounded-wait limit in SM cycles (about two seconds at the highest
// clock): far above any legitimate wait (a whole canonical GEMM takes about a
// millisecond) yet short enough that a broken pipeline returns control
// instead of holding the GPU.
constexpr uint64_t kDefaultWaitLimitCycles = 4000000000ull;

nvfp4_status fc2_gemm_launch(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec, const void* w_q,
                             const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m, int64_t n, int64_t k,
                             void* out, int64_t ldo, uint32_t* dev_status, cudaStream_t stream,
                             uint64_t wait_limit_cycles) {
  if (!a_q || !a_s || !a_rec || !w_q || !w_s || !w_rec || !out)
    return fail(NVFP4_EINVAL, "nvfp4_fc2_gemm: null pointer");
  if (m < 1) return fail(NVFP4_EINVAL, "nvfp4_fc2_gemm: m must be >= 1");
  if (n < HALF || n % HALF != 0) return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_gemm: n must be a positive multiple of 128");
  if (k < 256 || k % 256 != 0) return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_gemm: k must be a positive multiple of 256");
  if (ldo < n) return fail(NVFP4_EINVAL, "nvfp4_fc2_gemm: ldo < n");
  if (ldo % 8 != 0 || !aligned16(a_q) || !aligned16(a_s) || !aligned16(w_q) || !aligned16(w_s) || !aligned16(out) ||
      !aligned16(a_rec) || !aligned16(w_rec))
    return fail(NVFP4_EALIGN, "nvfp4_fc2_gemm: pointers must be 16-byte aligned and ldo a multiple of 8");
  const int64_t m_pad = nvfp4_padded_rows(m);
  if (m_pad > (int64_t(1) << 30) || n > (int64_t(1) << 24) || k > (int64_t(1) << 24))
    return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_gemm: problem too large");

  // A and W: 3-D views [k-tile][row][128 B] so one box carries KT k-tiles of
  // 128 rows (each a 128B-swizzled 16 KB tile).  Scales: [bytes / 256, 256]
  // byte rows (one 128-row panel x one k-tile is 8 rows = 2 KB); the W scales
  // as [panel][row][256] so one box carries both panels of a 256-row tile.
  const int64_t sa_rows = nvfp4_scale_bytes(m, k) / 256;
  CUtensorMap ta, tw, tsa, tsw, to;
  nvfp4_status st;
  {
    const cuuint64_t dims[3] = {128, cuuint64_t(m_pad), cuuint64_t(k / 256)};
    const cuuint64_t strides[2] = {cuuint64_t(k / 2), 128};
    const cuuint32_t box[3] = {BK_BYTES, HALF, KT};
    if ((st = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                       "A")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[3] = {128, cuuint64_t(n), cuuint64_t(k / 256)};
    const cuuint64_t strides[2] = {cuuint64_t(k / 2), 128};
    const cuuint32_t box[3] = {BK_BYTES, HALF, KT};
    if ((st = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                       "W")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[2] = {256, cuuint64_t(sa_rows)};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {256, 8 * KT};
    if ((st = make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_s, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                       "A scales")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[3] = {256, cuuint64_t(k / 32), cuuint64_t(n / 128)};
    const cuuint64_t strides[2] = {256, cuuint64_t(k / 32) * 256};
    const cuuint32_t box[3] = {256, 8 * KT, 2};
    if ((st = make_map(&tsw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_s, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                       "W scales")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[2] = {cuuint64_t(n), cuuint64_t(m)};
    const cuuint64_t strides[1] = {cuuint64_t(ldo) * 2};
    const cuuint32_t box[2] = {64, 32};
    if ((st = make_map(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                       "out")) != NVFP4_OK)
      return st;
  }

  Params prm;
  prm.a_rec = a_rec;
  prm.w_rec = w_rec;
  prm.a_rows = static_cast<int>(m_pad);
  prm.n = static_cast<int>(n);
  prm.num_m_tiles = static_cast<int>((m_pad + PAIR_M - 1) / PAIR_M);
  prm.num_n_tiles = static_cast<int>((n + PAIR_N - 1) / PAIR_N);
  // an odd k-tile count ends with a box whose second k-tile lies beyond K:
  // the TMA fills it with zeros, which add nothing to the sums
  prm.num_stages_k = static_cast<int>((k / 256 + KT - 1) / KT);
  prm.sf_panel_rows = static_cast<int>(k / 32);
  prm.dev_status = dev_status;
  prm.wait_limit_cycles = wait_limit_cycles;

  st = cuda_check(cudaFuncSetAttribute(k_fc2_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES),
                  "cudaFuncSetAttribute(k_fc2_gemm)");
  if (st != NVFP4_OK) return st;
  const int tiles = prm.num_m_tiles * prm.num_n_tiles;
  const int pairs = tiles < sm_count() / 2 ? tiles : sm_count() / 2;
  k_fc2_gemm<<<2 * pairs, THREADS, SMEM_BYTES, stream>>>(ta, tw, tsa, tsw, to, prm);
  return cuda_check(cudaGetLastError(), "launch k_fc2_gemm");
}

// ---- diagnostics: the bounded wait on a barrier nothing arrives at ---------

namespace {
__global__ void k_diag_wait_timeout(uint64_t limit_cycles, uint32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(&bar, 0, limit_cycles, &abort_flag)) *dev_status = NVFP4_ETIMEOUT;
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
                         reinterpret_cast<cudaStream_t>(stream), kDefaultWaitLimitCycles);
}

extern "C" nvfp4_status nvfp4_diag_wait_timeout(uint64_t limit_ns, uint32_t* dev_status, nvfp4_stream_t stream) {
  if (!dev_status || limit_ns < 1 || limit_ns > 1000000000ull)
    return fail(NVFP4_EINVAL, "nvfp4_diag_wait_timeout: bad arguments");
  // cycles at the highest SM clock (2.07 GHz) give at least limit_ns of wall time
  k_diag_wait_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns * 21 / 10, dev_status);
  return cuda_check(cudaGetLastError(), "launch k_diag_wait_timeout");
}
