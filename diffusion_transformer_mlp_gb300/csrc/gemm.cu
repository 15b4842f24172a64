// Persistent block-scaled NVFP4 GEMM for sm_103a (tcgen05 + TMA + TMEM).
//
// "FC2 NVFP4 Scheduling Results": Canonical Operation (M=37,810 -> padded,
// N=5,376, K=14,336; E2M1 operands with vector-16 UE4M3 scales; FP32
// accumulation; BF16 output), Decision (split-K 1, zero workspace),
// Traffic Attribution (the weight is re-read once per 128-row M tile, 296x,
// and the activation about 42x; the winning schedule keeps those re-reads
// in L2; no global atomics, no reduction traffic, one output write).
// The pages' kernel is a GB10 warp-MMA library kernel; this one is written
// for the datacenter Blackwell tensor core instead.  A CTA pair computes a
// 256 x 256 output tile with tcgen05.mma.cta_group::2 (M=256, N=256, K=64
// per instruction); each CTA holds 128 rows of A and 128 rows of W per
// k-tile and a 128 x 256 FP32 accumulator in its tensor memory.
//
//   warp 0      operand TMA producer (both CTAs): per stage KT k-tiles (256
//               K elements each) of this CTA's 128 A rows and 128 W rows
//               (128B swizzle, one box per operand and k-tile) into a
//               STAGES-deep shared-memory ring; the leader's barriers count
//               both CTAs' bytes, one barrier per k-tile.  A 64 KB stage
//               takes ~1,800 cycles to land against ~1,050 cycles of MMAs,
//               so three stages are in flight.
//   warp 14     scale TMA producer (both CTAs): per stage this CTA's A
//               scale blocks and the W scale blocks of both 128-row panels
//               of the tile (tiled layout, 12 KB) into an SF_RING-deep ring
//               that runs ahead of the operands.
//   warps 10-13 scale writers (both CTAs), one per TMEM lane quarter: read a
//               stage's UE4M3 words from the ring (ld.shared), store them
//               with tcgen05.st into one of two tensor-memory slots (free
//               once the MMAs of the stage two back have completed) in the
//               layout the MMA reads, and arrive on the leader's stage
//               barrier next to the TMA bytes.  A tcgen05.cp of the scales
//               would sit in the tensor pipe between the MMAs (a 32x128b
//               warpx4 copy costs about half an MMA there); tcgen05.st from
//               other warps does not.
//   warp 1      MMA issuer (leader CTA): per stage and k-tile one wait and
//               four MMAs reading the operands from the stage and the block
//               scales from the stage's tensor-memory slot; one commit per
//               stage.
//   warps 2-9   epilogue (both CTAs), two warps per TMEM lane quarter, 128
//               columns each: tcgen05.ld 32 accumulator columns at a time,
//               multiply by alpha = gA*gW and round to BF16 into registers;
//               after the last load the accumulator goes back to the MMA
//               issuer, and the warp writes its 32 rows x 128 columns
//               through a 1 KB shared-memory slot, 32 rows x 16 columns at
//               a time, with TMA stores (which clip rows >= M and columns
//               >= N).  The issuer waits for the loads at every tile
//               boundary, hence eight warps; the stores overlap the next
//               tile's MMAs and leave the load/store unit to the scale
//               writers.  The SwiGLU epilogue (below) stores h from
//               registers: its silu slice takes the shared memory.
//
// Tiles are walked in groups of N tiles: the whole weight when it fits 48 MB
// (FC2: all 21 N tiles), else 16 MB of it (21 of FC1's 112); each group is walked
// M-panel-major (all N tiles of the group for one 256-row panel, then the
// next), so the CTAs running at any moment share a few activation panels
// and one group's weight rows, which stay in L2 across every panel (one
// M-panel-major sweep over all 112 FC1 N tiles read its weight ~19 times
// from DRAM).  K is reduced in increasing
// order inside one CTA: no split-K, no workspace, no atomics, and an output
// row does not depend on M.
//
// k_fc2_gemm<true> is FC1 with the SwiGLU producer's first pass in the
// epilogue (nvfp4_fc1_swiglu).  W holds the gate rows then the up rows; a
// pair tile takes 128 gate rows from CTA 0 and the matching 128 up rows
// from CTA 1, so every CTA's accumulator holds g in columns 0..127 and u in
// 128..255 for its rows.  The epilogue rounds both to BF16 exactly as the
// plain epilogue would store them, hands the accumulator back, forms
// h = bf16(silu_bf16(g) u) (silu from a 6.5 KB shared-memory slice of the
// producer's table) and stores it, and keeps max |h| for one atomic per
// warp on the activation record.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int PAIR_M = 256;
constexpr int PAIR_N = 256;
constexpr int HALF = 128;
constexpr int BK_BYTES = 128;  // 256 E2M1 elements per k-tile
constexpr int KT = 2;          // k-tiles per pipeline stage (one TMA box per operand per stage)
constexpr int STAGES = 3;
constexpr int KTILE_BYTES = HALF * BK_BYTES;   // 16 KB: 128 rows x one k-tile
constexpr int A_BYTES = KT * KTILE_BYTES;      // this CTA's 128 A rows x KT k-tiles
constexpr int B_BYTES = KT * KTILE_BYTES;      // this CTA's 128 W rows x KT k-tiles
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int KSTEPS = 4 * KT;                 // K=64 MMA steps per stage
// Scale ring: per stage 4*KT blocks of 512 bytes for this CTA's A panel,
// then the same for W panel 0 and W panel 1 of the tile.
constexpr int SF_RING = 2;
constexpr int SFA_BYTES = KSTEPS * 512;
constexpr int SFW_PANEL_BYTES = KSTEPS * 512;
constexpr int SF_STAGE_BYTES = SFA_BYTES + 2 * SFW_PANEL_BYTES;  // 12 KB
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, 128 columns each
constexpr int SF_WARPS = 4;
constexpr int WARP_EPI0 = 2;
constexpr int WARP_SF0 = WARP_EPI0 + EPI_WARPS;
constexpr int WARP_SFP = WARP_SF0 + SF_WARPS;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + SF_RING * SF_STAGE_BYTES + BAR_BYTES;
constexpr int THREADS = (WARP_SFP + 1) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;  // 256 FP32 columns
// Block scales in tensor memory, two slots used by alternate stages
// (KSTEPS K=64 steps j each):
//   A: step j at columns slot + 4j .. + 3; the scales of accumulator row i
//      are read from lane i, column slot + 4j + i/32, and only that column
//      is written.
//   W: step j at column slot + SFW_COL + 8j; accumulator rows of lane
//      quarter g read the scales of W row n from lane 32g + n % 32, column
//      slot + SFW_COL + 8j + n/32, so every quarter holds a copy.
constexpr uint32_t SF_COL = 256;
constexpr uint32_t SFW_COL = 4 * KSTEPS;
constexpr uint32_t SF_SLOT_COLS = 12 * KSTEPS;
constexpr int SF_SLOTS = 2;
static_assert(SF_COL + SF_SLOTS * SF_SLOT_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(STAGES > SF_SLOTS, "a stage's scale slot is free once the stage SF_SLOTS back has completed");
static_assert(KSTEPS == 8, "scale stores are written 32 columns at a time");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0 && SF_STAGE_BYTES % 1024 == 0, "stage alignment");

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

// BF16 silu of a gate for the SwiGLU epilogue: the correctly rounded value
// the producer's table holds ("GB10 component-2 nsys summary": silu in BF16
// ahead of the multiply by up).  The whole table (128 KB) cannot sit in
// shared memory next to the operand ring, but the gates FC1 produces are
// almost all in 2^-10 <= |g| < 8: 13 binades x 128 BF16 mantissas x 2 signs
// = 3,328 entries (6.5 KB), copied into shared memory at kernel start.  The
// rest: g >= 8 gives g (the table's closed form, +inf included); |g| < 2^-10,
// g <= -8, -inf and NaN read the global table.  nvfp4_diag_silu_epilogue
// runs this for all 65,536 gates against the table.
__device__ const uint16_t k_silu_tab_epi[65536] = {
#include "silu_table_full.inc"
};

constexpr int kSiluExpLo = 117;                       // biased exponent of 2^-10
constexpr int kSiluExps = 13;                         // 2^-10 .. 2^3 (exclusive)
constexpr int kSiluHalf = kSiluExps * 128;            // entries per sign
constexpr int kSiluSmemBytes = 2 * kSiluHalf * 2;     // 6,656 bytes

__device__ __forceinline__ void fill_silu_smem(uint16_t* tab_s) {
  for (int i = threadIdx.x; i < 2 * kSiluHalf; i += blockDim.x) {
    const int sign = i / kSiluHalf, r = i - sign * kSiluHalf;
    const uint32_t gb = (uint32_t(sign) << 15) | (uint32_t(kSiluExpLo + r / 128) << 7) | uint32_t(r % 128);
    tab_s[i] = k_silu_tab_epi[gb];
  }
}

__device__ __forceinline__ uint32_t silu_bf16_epi(uint32_t gb, const uint16_t* tab_s) {
  const uint32_t e = (gb >> 7) & 0xFFu;
  if (e - uint32_t(kSiluExpLo) < uint32_t(kSiluExps))
    return tab_s[((gb >> 15) ? kSiluHalf : 0) + (e - kSiluExpLo) * 128 + (gb & 0x7Fu)];
  if (gb < 0x8000u && e >= uint32_t(kSiluExpLo + kSiluExps) && gb <= 0x7F80u) return gb;  // 8 <= g <= +inf
  return k_silu_tab_epi[gb];
}

// h = bf16(silu_bf16(g) * u) for two BF16 (g, u) pairs, as the producer's
// SwiGLU forms it (mul.rn.bf16x2: the exact product rounded once).
__device__ __forceinline__ uint32_t swiglu_pair_epi(uint32_t gw, uint32_t uw, const uint16_t* tab_s) {
  const uint32_t sw = silu_bf16_epi(gw & 0xFFFFu, tab_s) | (silu_bf16_epi(gw >> 16, tab_s) << 16);
  const __nv_bfloat162 h = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&sw),
                                   *reinterpret_cast<const __nv_bfloat162*>(&uw));
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct Smem {
  uint8_t* stage;       // STAGES x [A | B]
  uint8_t* sf;          // SF_RING x [A scales | W scales panel 0 | panel 1]
  uint64_t* full;       // leader: the first k-tile's operand bytes of both CTAs have
                        // landed and the stage's scales are in both CTAs' tensor memory
  uint64_t* full_kt1;   // leader: the second k-tile's operand bytes of both CTAs have landed
  uint64_t* empty;      // each CTA: the stage's MMAs are complete (operands and its scale slot free)
  uint64_t* sf_full;    // each CTA: a scale-ring slot has landed
  uint64_t* sf_empty;   // each CTA: the scale writers have read a ring slot
  uint64_t* tfull;      // each CTA: accumulators complete
  uint64_t* tempty;     // leader: accumulators of both CTAs drained
  uint64_t* mma_done;
  uint32_t* tmem_slot;
  int* abort_flag;
  uint16_t* silu;       // the SwiGLU epilogue's silu entries (k_fc2_gemm<true> only)
  uint8_t* out_stage;   // the plain epilogue's output slots (k_fc2_gemm<false> only; the same bytes)
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stage = base;
  s.sf = base + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.sf + SF_RING * SF_STAGE_BYTES);
  s.full = bars;
  s.full_kt1 = s.full + STAGES;
  s.empty = s.full_kt1 + STAGES;
  s.sf_full = s.empty + STAGES;
  s.sf_empty = s.sf_full + SF_RING;
  s.tfull = s.sf_empty + SF_RING;
  s.tempty = s.tfull + 1;
  s.mma_done = s.tempty + 1;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.mma_done + 1);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.silu = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(bars) + BAR_BYTES);
  s.out_stage = reinterpret_cast<uint8_t*>(bars) + BAR_BYTES;
  return s;
}
static_assert((3 * STAGES + 2 * SF_RING + 3) * 8 + 8 <= BAR_BYTES, "barrier area");
static_assert(SMEM_BYTES + kSiluSmemBytes <= 232448, "shared memory budget of the SwiGLU epilogue");
// the plain epilogue's output slots: one per warp, 32 rows x 16 BF16 columns
constexpr int kOutSlotBytes = 32 * 16 * 2;
static_assert(SMEM_BYTES + EPI_WARPS * kOutSlotBytes <= 232448, "shared memory budget of the plain epilogue");
static_assert((SMEM_BYTES - 1024 - BAR_BYTES) % 1024 == 0 && BAR_BYTES % 128 == 0, "output slots 128-byte aligned");

struct Params {
  const nvfp4_scale_rec* a_rec;
  const nvfp4_scale_rec* w_rec;
  __nv_bfloat16* out;  // [m, ldo] row-major
  int64_t ldo;
  int store32;       // out is 32-byte aligned and ldo a multiple of 16: 32-byte stores
  int m;             // output rows
  int n;             // weight rows (multiple of 128)
  int num_m_tiles;   // ceil(padded rows of the activation / 256)
  int num_n_tiles;   // ceil(n / 256)
  int group_n;       // N tiles per group of the tile order (see tile_coords)
  int num_k_tiles;   // k / 256
  int sf_rows;       // 256-byte rows of one 128-row scale panel: k / 32
  uint32_t* dev_status;
  uint64_t wait_limit_cycles;
  // SwiGLU epilogue (FC1 with the producer's first pass): W rows [0, f) are
  // the gate and [f, 2f) the up projection; a tile's gate panel comes from
  // CTA 0 and the matching up panel from CTA 1, so each CTA's accumulator
  // holds both; h = bf16(silu(g) u) goes to out and max |h| to h_rec.
  int f;
  nvfp4_scale_rec* h_rec;
  // Diagnostic launches only (else null): block 0 writes {start ns, end ns,
  // start cycle, end cycle} of its run, globaltimer and its SM's clock64.
  uint64_t* clk;
};

// Tile order: the N tiles are cut into groups of group_n; a group is walked
// M-panel-major (every N tile of the group for one 256-row panel, then the
// next panel) before the next group starts.  The pairs running at any
// moment then share a few activation panels and one group's weight rows,
// which stay in L2 across all panels; with group_n = num_n_tiles this is
// the plain M-panel-major order.
__device__ __forceinline__ void tile_coords(int t, const Params& p, int& mt, int& nt) {
  const int span = p.group_n * p.num_m_tiles;
  const int g = t / span;
  const int g0 = g * p.group_n;
  const int gs = min(p.group_n, p.num_n_tiles - g0);
  const int r = t - g * span;
  mt = r / gs;
  nt = g0 + (r - mt * gs);
}

__device__ __forceinline__ void report_timeout(const Params& p, int* abort_flag) {
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
  if (p.dev_status != nullptr) atomicExch(p.dev_status, static_cast<uint32_t>(NVFP4_ETIMEOUT));
}

// One lane of a warp waits; the warp follows its result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Params& p,
                                          const volatile int* abort_flag, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, p.wait_limit_cycles, abort_flag);
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Position in a ring of `slots` buffers: the slot and the parity of its
// current use.
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int slots) {
    if (++slot == slots) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// The scale words one writer lane stores for one stage (K=64 steps
// j = 0..KSTEPS-1): lane l of quarter q holds A row 32q + l of this CTA's
// half (one 32-bit word = four scales per step) and W rows 32c + l of the
// pair's tile, c = 0..7 (one 16-byte line of the tiled layout per 128-row
// panel and step).  In a ring slot (tiled layout, one 512-byte block per
// step and panel): the A word at j*512 + 16l + 4q, the W line of panel h at
// SFA_BYTES + h*SFW_PANEL_BYTES + j*512 + 16l.
struct ScaleWords {
  uint32_t a[KSTEPS];
  uint4 w[2 * KSTEPS];  // [2j + panel]
};

__device__ __forceinline__ void read_scales(ScaleWords& v, const uint8_t* slot, int q, int lane) {
#pragma unroll
  for (int j = 0; j < KSTEPS; ++j) {
    v.a[j] = *reinterpret_cast<const uint32_t*>(slot + j * 512 + lane * 16 + q * 4);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      v.w[2 * j + h] = *reinterpret_cast<const uint4*>(slot + SFA_BYTES + h * SFW_PANEL_BYTES + j * 512 + lane * 16);
  }
}

// A: a lane of quarter q reads only column 4j + q of step j, so the writer
// of quarter q stores its word there alone (one column per step).
__device__ __forceinline__ void store_scales(uint32_t taddr, const ScaleWords& v, int q) {
#pragma unroll
  for (int j = 0; j < KSTEPS; ++j)
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr + 4 * j + q), "r"(v.a[j]) : "memory");
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint4* x = v.w + 8 * half;
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr + SFW_COL + 32 * half),
        "r"(x[0].x), "r"(x[0].y), "r"(x[0].z), "r"(x[0].w), "r"(x[1].x), "r"(x[1].y), "r"(x[1].z), "r"(x[1].w),
        "r"(x[2].x), "r"(x[2].y), "r"(x[2].z), "r"(x[2].w), "r"(x[3].x), "r"(x[3].y), "r"(x[3].z), "r"(x[3].w),
        "r"(x[4].x), "r"(x[4].y), "r"(x[4].z), "r"(x[4].w), "r"(x[5].x), "r"(x[5].y), "r"(x[5].z), "r"(x[5].w),
        "r"(x[6].x), "r"(x[6].y), "r"(x[6].z), "r"(x[6].w), "r"(x[7].x), "r"(x[7].y), "r"(x[7].z), "r"(x[7].w)
        : "memory");
  }
}

// Walk of one CTA pair over its (tile, stage) sequence.
struct StageWalk {
  int t, ks;
  __device__ __forceinline__ void next(int stages_per_tile, int num_pairs) {
    if (++ks == stages_per_tile) {
      ks = 0;
      t += num_pairs;
    }
  }
};

template <bool kGated>
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
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  const int nk = p.num_k_tiles;
  const int stages_per_tile = (nk + KT - 1) / KT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the producer's expect_tx arrival plus one per scale writer of either CTA
      mbar_init(&sm.full[s], 1 + 2 * SF_WARPS);
      mbar_init(&sm.full_kt1[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < SF_RING; ++s) {
      mbar_init(&sm.sf_full[s], 1);
      mbar_init(&sm.sf_empty[s], SF_WARPS);
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
    if constexpr (!kGated) prefetch_tmap(&tmap_out);
  }
  if constexpr (kGated) fill_silu_smem(sm.silu);
  if (warp == 1) tmem_alloc_pair(sm.tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated in both
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  if (p.clk != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    p.clk[0] = globaltimer_ns();
    p.clk[2] = clock64();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ operand producer (both CTAs)
    if (lane == 0) {
      // the weight and the activation panels in flight are both re-read (the
      // weight by every M panel, a panel by every N tile of its group): keep
      // both ahead of the output stores in L2
      const uint64_t pol_w = l2_policy_evict_last();
      const uint64_t pol_a = l2_policy_evict_last();
      Ring r;
      bool ok = true;
      int mt = 0, nt = 0, cur_t = -1;
      for (StageWalk w{pair, 0}; w.t < num_tiles && ok; w.next(stages_per_tile, num_pairs), r.next(STAGES)) {
        if (w.t != cur_t) {  // a new tile: its coordinates, once
          tile_coords(w.t, p, mt, nt);
          cur_t = w.t;
        }
        // One box per operand and k-tile: the first k-tile of both operands
        // completes on the stage's barrier, the second on its own, so the
        // first four MMAs can start while the second k-tile lands.  Boxes
        // beyond the operands (the last M or N half, a k-tile past K) are
        // zero-filled by the TMA and still count their full bytes, so each
        // barrier receives STAGE_BYTES (half a stage from each CTA).
        const int a_row = mt * PAIR_M + int(rank) * HALF;
        const int b_row = kGated ? (rank == 0 ? nt * HALF : p.f + nt * HALF) : nt * PAIR_N + int(rank) * HALF;
        if (!mbar_wait_bounded(&sm.empty[r.slot], r.phase ^ 1u, p.wait_limit_cycles, abort_flag)) {
          report_timeout(p, sm.abort_flag);
          ok = false;
          break;
        }
        uint8_t* st = sm.stage + r.slot * STAGE_BYTES;
        const uint32_t full_leader = mapa_shared(smem_u32(&sm.full[r.slot]), 0);
        const uint32_t kt1_leader = mapa_shared(smem_u32(&sm.full_kt1[r.slot]), 0);
        if (leader) {
          mbar_arrive_expect_tx(&sm.full[r.slot], STAGE_BYTES);
          mbar_arrive_expect_tx(&sm.full_kt1[r.slot], STAGE_BYTES);
        }
        tma_load_3d_pair(st, &tmap_a, full_leader, 0, a_row, w.ks * KT, pol_a);
        tma_load_3d_pair(st + A_BYTES, &tmap_w, full_leader, 0, b_row, w.ks * KT, pol_w);
        tma_load_3d_pair(st + KTILE_BYTES, &tmap_a, kt1_leader, 0, a_row, w.ks * KT + 1, pol_a);
        tma_load_3d_pair(st + A_BYTES + KTILE_BYTES, &tmap_w, kt1_leader, 0, b_row, w.ks * KT + 1, pol_w);
      }
    }
  } else if (warp == WARP_SFP) {
    // ------------------------------------------------------------ scale producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();
      const uint64_t pol_a = l2_policy_evict_last();
      Ring r;
      bool ok = true;
      int mt = 0, nt = 0, cur_t = -1;
      for (StageWalk w{pair, 0}; w.t < num_tiles && ok; w.next(stages_per_tile, num_pairs), r.next(SF_RING)) {
        if (w.t != cur_t) {  // a new tile: its coordinates, once
          tile_coords(w.t, p, mt, nt);
          cur_t = w.t;
        }
        if (!mbar_wait_bounded(&sm.sf_empty[r.slot], r.phase ^ 1u, p.wait_limit_cycles, abort_flag)) {
          report_timeout(p, sm.abort_flag);
          ok = false;
          break;
        }
        // A scales: 256-byte rows of the whole scale buffer (this CTA's
        // panel starts at panel * sf_rows); W scales: [panel][row][256].
        // Rows past K (an odd k-tile count) or past the operand are read
        // as whatever the box holds or zero fill and never multiplied or
        // stored.
        uint8_t* sl = sm.sf + r.slot * SF_STAGE_BYTES;
        const int row0 = w.ks * KSTEPS * 2;  // two 256-byte rows per 512-byte block
        mbar_arrive_expect_tx(&sm.sf_full[r.slot], SF_STAGE_BYTES);
        tma_load_2d(sl, &tmap_sa, &sm.sf_full[r.slot], 0, (mt * 2 + int(rank)) * p.sf_rows + row0, pol_a);
        if constexpr (kGated) {
          // the gate and the up panel of the tile, one box each
          tma_load_3d(sl + SFA_BYTES, &tmap_sw, &sm.sf_full[r.slot], 0, row0, nt, pol_w);
          tma_load_3d(sl + SFA_BYTES + SFW_PANEL_BYTES, &tmap_sw, &sm.sf_full[r.slot], 0, row0, p.f / HALF + nt, pol_w);
        } else {
          tma_load_3d(sl + SFA_BYTES, &tmap_sw, &sm.sf_full[r.slot], 0, row0, nt * 2, pol_w);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (lane == 0 && leader) {
      Ring ab;
      int sf_slot = 0;
      int local = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs, ++local) {
        if (!mbar_wait_bounded(sm.tempty, (local & 1) ^ 1u, p.wait_limit_cycles, abort_flag)) {
          report_timeout(p, sm.abort_flag);
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < stages_per_tile; ++ks, ab.next(STAGES), sf_slot ^= 1) {
          if (!mbar_wait_bounded(&sm.full[ab.slot], ab.phase, p.wait_limit_cycles, abort_flag)) {
            report_timeout(p, sm.abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(sm.stage + ab.slot * STAGE_BYTES);
          const uint32_t sf_tmem = tmem + SF_COL + uint32_t(sf_slot) * SF_SLOT_COLS;
          const int kk_end = (ks * KT + KT <= nk) ? KT : nk - ks * KT;
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            if (kk == 1) {  // the second k-tile's operands (zeros past K) have landed
              if (!mbar_wait_bounded(&sm.full_kt1[ab.slot], ab.phase, p.wait_limit_cycles, abort_flag)) {
                report_timeout(p, sm.abort_flag);
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (kk >= kk_end) break;  // the second k-tile of a last stage past K
            const uint64_t a_desc = desc_sw128(st + kk * KTILE_BYTES);
            const uint64_t b_desc = desc_sw128(st + A_BYTES + kk * KTILE_BYTES);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // K step j: 64 elements = 32 bytes further along the swizzled row
              tc_mma_pair_nvf4(tmem + ACC_COL, a_desc + 2 * j, b_desc + 2 * j, kIdesc, sf_tmem + 4 * (4 * kk + j),
                               sf_tmem + SFW_COL + 8 * (4 * kk + j), (ks | kk | j) != 0);
            }
          }
          if (!ok) break;
          tc_commit_pair(&sm.empty[ab.slot]);  // stage and its scale slot reusable in both CTAs
        }
        if (!ok) break;
        tc_commit_pair(sm.tfull);  // accumulators of both CTAs ready
      }
      // Nothing may still be reading shared memory or writing tensor memory
      // in either CTA when the pair tears down.
      tc_commit_pair(sm.mma_done);
    }
  } else if (warp < WARP_SF0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int col0 = ((warp - WARP_EPI0) / 4) * (PAIR_N / 2);  // this warp's half of the columns
    uint8_t* out_slot = sm.out_stage + (warp - WARP_EPI0) * kOutSlotBytes;  // plain epilogue only
    const float alpha = __fmul_rn(p.a_rec->global_scale, p.w_rec->global_scale);
    const uint32_t tempty_leader = mapa_shared(smem_u32(sm.tempty), 0);
    // the output is written once and never read back here: evict it first,
    // so that it does not push the activation panels and the weight out of L2
    uint64_t pol_out;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_out));
    if constexpr (kGated) {
      // SwiGLU: this warp takes gate columns 64*wh .. +63 and the matching
      // up columns 128 + 64*wh .. +63 of its 32 rows, 32 of each per load
      // round; g and u are the BF16 FC1 outputs (accumulator x alpha rounded
      // as the plain epilogue rounds them) and h goes to columns
      // nt*128 + 64*wh of the [m, f] output.  The lane keeps max |h| (bit
      // patterns, as the producer's first pass does) over its stored rows.
      const int wh = (warp - WARP_EPI0) / 4;
      uint32_t amax = 0;
      int local = 0;
      for (int t = pair; t < num_tiles; t += num_pairs, ++local) {
        int mt, nt;
        tile_coords(t, p, mt, nt);
        if (!warp_wait(sm.tfull, local & 1, p, abort_flag, lane)) {
          if (lane == 0) report_timeout(p, sm.abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t lane_tmem = tmem + (uint32_t(q * 32) << 16) + ACC_COL + 64 * wh;
        const int row = mt * PAIR_M + int(rank) * HALF + q * 32 + lane;
        const bool row_ok = row < p.m;
        __nv_bfloat16* hrow = p.out + int64_t(row_ok ? row : 0) * p.ldo + nt * HALF + 64 * wh;
        // both 32-column rounds are loaded and rounded to BF16 (g and u as
        // the plain epilogue would store them) before the accumulator goes
        // back; silu, the product and the stores follow
        uint32_t gw[2][16], uw[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64];
          tmem_ld_32x32b_x32(lane_tmem + 32 * c, r);             // gate
          tmem_ld_32x32b_x32(lane_tmem + HALF + 32 * c, r + 32);  // up
          tc_wait_ld();
          tmem_ld_fence_regs<64>(r);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            gw[c][i] = bf16x2_rn(__fmul_rn(__uint_as_float(r[2 * i]), alpha),
                                 __fmul_rn(__uint_as_float(r[2 * i + 1]), alpha));
            uw[c][i] = bf16x2_rn(__fmul_rn(__uint_as_float(r[32 + 2 * i]), alpha),
                                 __fmul_rn(__uint_as_float(r[32 + 2 * i + 1]), alpha));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = swiglu_pair_epi(gw[c][i], uw[c][i], sm.silu);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = max(amax, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
            __nv_bfloat16* dst = hrow + 32 * c;
            if (p.store32) {
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2)
                asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 16 * k2), "r"(w[8 * k2]),
                             "r"(w[8 * k2 + 1]), "r"(w[8 * k2 + 2]), "r"(w[8 * k2 + 3]), "r"(w[8 * k2 + 4]),
                             "r"(w[8 * k2 + 5]), "r"(w[8 * k2 + 6]), "r"(w[8 * k2 + 7])
                             : "memory");
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
          }
        }
      }
      // the producer's first pass: one atomic per warp on the record
      amax = __reduce_max_sync(0xFFFFFFFFu, amax);
      if (lane == 0 && amax != 0) atomicMax(&p.h_rec->amax_bits, amax);
    } else {
    int local = 0;
    for (int t = pair; t < num_tiles; t += num_pairs, ++local) {
      int mt, nt;
      tile_coords(t, p, mt, nt);
      if (!warp_wait(sm.tfull, local & 1, p, abort_flag, lane)) {
        if (lane == 0) report_timeout(p, sm.abort_flag);
        break;
      }
      tc_fence_after();
      // The warp's 32 rows x 128 columns into registers as BF16 pairs, the
      // accumulator back to the issuer, then the output through the warp's
      // shared-memory slot and TMA stores.  Row-per-lane global stores
      // (32 rows per instruction) held the load/store unit that the scale
      // writers' ld.shared need: this form took FC2 from 1.496 to 1.447 M
      // SM cycles and the FC1 shape from 3.601 to 3.284 M.
      const uint32_t row_tmem = tmem + (uint32_t(q * 32) << 16) + ACC_COL + col0;
      uint32_t wb[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(row_tmem + c * 32, r);
        tc_wait_ld();
        tmem_ld_fence_regs<32>(r);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wb[c][i] = bf16x2_rn(__fmul_rn(__uint_as_float(r[2 * i]), alpha), __fmul_rn(__uint_as_float(r[2 * i + 1]), alpha));
      }
      // accumulator drained: hand it back to the MMA issuer of the pair (the
      // loads are complete: wait::ld, fence::before_thread_sync)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
      // 32 rows x 16 columns per store: lane l writes row l's 32 bytes of
      // the slot (row-major, as the box lays it out); the next fill waits
      // until the previous store has read the slot
      const int y = mt * PAIR_M + int(rank) * HALF + q * 32;
      const int x0 = nt * PAIR_N + col0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          uint4* d = reinterpret_cast<uint4*>(out_slot + lane * 32);
          d[0] = make_uint4(wb[c][8 * hh], wb[c][8 * hh + 1], wb[c][8 * hh + 2], wb[c][8 * hh + 3]);
          d[1] = make_uint4(wb[c][8 * hh + 4], wb[c][8 * hh + 5], wb[c][8 * hh + 6], wb[c][8 * hh + 7]);
          fence_proxy_async_smem();  // the generic-proxy writes, then the TMA's reads
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmap_out, out_slot, x0 + c * 32 + hh * 16, y, pol_out);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // the stores are complete before the CTA exits
    }
  } else {
    // ------------------------------------------------------------ scale writers (both CTAs)
    const int q = warp & 3;  // lane quarter: A rows 32q..32q+31 and this quarter's copy of the W scales
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const uint32_t full_leader = mapa_shared(smem_u32(sm.full), 0);
    Ring r;     // operand stage (its full barrier)
    Ring back;  // the stage SF_SLOTS back, whose MMAs free this stage's tensor-memory scale slot
    Ring sr;    // scale ring slot
    int g = 0;  // stages handled by this pair so far
    int sf_slot = 0;
    for (StageWalk w{pair, 0}; w.t < num_tiles;
         w.next(stages_per_tile, num_pairs), r.next(STAGES), sr.next(SF_RING), sf_slot ^= 1, ++g) {
      if (!warp_wait(&sm.sf_full[sr.slot], sr.phase, p, abort_flag, lane)) {
        if (lane == 0) report_timeout(p, sm.abort_flag);
        break;
      }
      // Read the ring slot into registers and release it, then wait for
      // the tensor-memory slot (the first SF_SLOTS stages find it free).
      // The next TMA into the slot writes through the async proxy: the
      // proxy fence orders these generic-proxy reads before it (without it
      // the refill was seen to race the reads).
      ScaleWords v;
      read_scales(v, sm.sf + sr.slot * SF_STAGE_BYTES, q, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sf_empty[sr.slot]);
      if (g >= SF_SLOTS) {
        if (!warp_wait(&sm.empty[back.slot], back.phase, p, abort_flag, lane)) {
          if (lane == 0) report_timeout(p, sm.abort_flag);
          break;
        }
        back.next(STAGES);
      }
      tc_fence_after();
      store_scales(tmem + lane_base + SF_COL + uint32_t(sf_slot) * SF_SLOT_COLS, v, q);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      // the stores are complete (wait::st, fence::before_thread_sync)
      if (lane == 0) mbar_arrive_cluster_relaxed(full_leader + 8u * uint32_t(r.slot));
    }
  }

  // teardown: every MMA of the pair has completed before tensor memory is freed
  if (warp == 1 && lane == 0) {
    if (!mbar_wait_bounded(sm.mma_done, 0, p.wait_limit_cycles, nullptr)) report_timeout(p, sm.abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (p.clk != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    p.clk[1] = globaltimer_ns();
    p.clk[3] = clock64();
  }
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

// CTA pairs of k_fc2_gemm<gated> that are resident at once on the current
// device (two-CTA clusters at `smem` bytes each: SMs / 2 on a GB300, fewer
// where the GPCs cannot all hold pairs), cached per device and variant.
// The persistent grid is sized to this so that no pair waits for a second
// wave.
nvfp4_status resident_pairs(bool gated, int smem, int* pairs) {
  static std::mutex mu;
  static int cache[64][2] = {};
  int dev = 0;
  nvfp4_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != NVFP4_OK) return st;
  if (dev < 0 || dev >= 64) return fail(NVFP4_EUNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][gated ? 1 : 0];
  if (c == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    int clusters = 0;
    st = cuda_check(cudaOccupancyMaxActiveClusters(&clusters, gated ? k_fc2_gemm<true> : k_fc2_gemm<false>, &cfg),
                    "cudaOccupancyMaxActiveClusters(k_fc2_gemm)");
    if (st != NVFP4_OK) return st;
    if (clusters < 1) return fail(NVFP4_ECUDA, "k_fc2_gemm: no two-CTA cluster fits on this device");
    c = clusters < sm_count() / 2 ? clusters : sm_count() / 2;
  }
  *pairs = c;
  return NVFP4_OK;
}

}  // namespace

// Default bounded-wait limit in SM cycles (about two seconds at the highest
// clock): far above any legitimate wait (a whole canonical GEMM takes about a
// millisecond) yet short enough that a broken pipeline returns control
// instead of holding the GPU.
constexpr uint64_t kDefaultWaitLimitCycles = 4000000000ull;

// The plain GEMM (f = 0: out [m, n]) and the SwiGLU-epilogue GEMM (f > 0:
// W has n = 2f rows, gate then up; out is h [m, f] and h_rec receives max
// |h|).  `name` prefixes the error messages.
nvfp4_status gemm_launch(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec, const void* w_q,
                         const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m, int64_t n, int64_t k, void* out,
                         int64_t ldo, int64_t f, nvfp4_scale_rec* h_rec, uint32_t* dev_status, cudaStream_t stream,
                         uint64_t wait_limit_cycles, const char* name, uint64_t* clk = nullptr) {
  const std::string nm(name);
  const bool gated = f > 0;
  if (!a_q || !a_s || !a_rec || !w_q || !w_s || !w_rec || !out || (gated && !h_rec))
    return fail(NVFP4_EINVAL, nm + ": null pointer");
  if (m < 1 || f < 0) return fail(NVFP4_EINVAL, nm + ": m must be >= 1");
  if (gated && (f % HALF != 0 || n != 2 * f))
    return fail(NVFP4_EUNSUPPORTED, nm + ": f must be a positive multiple of 128 and W must have 2f rows");
  if (n < HALF || n % HALF != 0) return fail(NVFP4_EUNSUPPORTED, nm + ": n must be a positive multiple of 128");
  if (k < 256 || k % 256 != 0) return fail(NVFP4_EUNSUPPORTED, nm + ": k must be a positive multiple of 256");
  const int64_t out_cols = gated ? f : n;
  if (ldo < out_cols) return fail(NVFP4_EINVAL, nm + ": output leading dimension too small");
  if (ldo % 8 != 0 || !aligned16(a_q) || !aligned16(a_s) || !aligned16(w_q) || !aligned16(w_s) || !aligned16(out) ||
      !aligned16(a_rec) || !aligned16(w_rec) || (gated && !aligned16(h_rec)))
    return fail(NVFP4_EALIGN, nm + ": pointers must be 16-byte aligned and the leading dimension a multiple of 8");
  const int64_t m_pad = nvfp4_padded_rows(m);
  if (m_pad > (int64_t(1) << 30) || n > (int64_t(1) << 24) || k > (int64_t(1) << 24))
    return fail(NVFP4_EUNSUPPORTED, nm + ": problem too large");

  // A and W: 3-D views [k-tile][row][128 B]; one box is one k-tile of 128
  // rows (a 128B-swizzled 16 KB tile).  Scales: the A scales as
  // [bytes / 256][256] (one 128-row panel x one k-tile is 8 rows = 2 KB),
  // the W scales as [panel][k / 32][256] so one box carries a stage of both
  // panels of a 256-row tile.
  const int64_t sa_rows = nvfp4_scale_bytes(m, k) / 256;
  CUtensorMap ta, tw, tsa, tsw, tout;
  nvfp4_status st;
  {
    const cuuint64_t dims[3] = {128, cuuint64_t(m_pad), cuuint64_t(k / 256)};
    const cuuint64_t strides[2] = {cuuint64_t(k / 2), 128};
    const cuuint32_t box[3] = {BK_BYTES, HALF, 1};
    if ((st = make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                       "A")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[3] = {128, cuuint64_t(n), cuuint64_t(k / 256)};
    const cuuint64_t strides[2] = {cuuint64_t(k / 2), 128};
    const cuuint32_t box[3] = {BK_BYTES, HALF, 1};
    if ((st = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                       "W")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[2] = {256, cuuint64_t(sa_rows)};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {256, 2 * KSTEPS};
    if ((st = make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_s, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                       "A scales")) != NVFP4_OK)
      return st;
  }
  {
    const cuuint64_t dims[3] = {256, cuuint64_t(k / 32), cuuint64_t(n / 128)};
    const cuuint64_t strides[2] = {256, cuuint64_t(k / 32) * 256};
    const cuuint32_t box[3] = {256, 2 * KSTEPS, gated ? 1u : 2u};
    if ((st = make_map(&tsw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_s, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                       "W scales")) != NVFP4_OK)
      return st;
  }
  {
    // the output [m, out_cols] BF16, rows ldo apart: one 32-row x 16-column
    // box per store of the plain epilogue (rows >= m, columns >= out_cols
    // are clipped by the TMA)
    const cuuint64_t dims[2] = {cuuint64_t(out_cols), cuuint64_t(m)};
    const cuuint64_t strides[1] = {cuuint64_t(ldo) * 2};
    const cuuint32_t box[2] = {16, 32};
    if ((st = make_map(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                       "output")) != NVFP4_OK)
      return st;
  }
  Params prm;
  prm.a_rec = a_rec;
  prm.w_rec = w_rec;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.ldo = ldo;
  prm.store32 = (reinterpret_cast<uintptr_t>(out) % 32 == 0 && ldo % 16 == 0) ? 1 : 0;
  prm.m = static_cast<int>(m);
  prm.n = static_cast<int>(n);
  prm.num_m_tiles = static_cast<int>((m_pad + PAIR_M - 1) / PAIR_M);
  prm.num_n_tiles = static_cast<int>(gated ? f / HALF : (n + PAIR_N - 1) / PAIR_N);
  {
    // Weight bytes of one N tile (256 rows: E2M1 codes and UE4M3 scales).
    // A weight that fits 48 MB stays in L2 whole: one group (FC2's 43 MB;
    // splitting it made every group re-read the activation: 0.92 against
    // 0.89 ms).  A larger one goes in groups of 16 MB (FC1, qkv: 16 MB
    // measured best against 8, 24, 32, 48 MB and one group).
    const int64_t tile_bytes = int64_t(PAIR_N) * (k / 2 + k / 16);
    const int64_t g = tile_bytes * prm.num_n_tiles <= (int64_t(48) << 20) ? prm.num_n_tiles
                                                                           : (int64_t(16) << 20) / tile_bytes;
    prm.group_n = static_cast<int>(g < 1 ? 1 : (g > prm.num_n_tiles ? prm.num_n_tiles : g));
  }
  // an odd k-tile count ends with a stage whose second k-tile lies beyond
  // K: the TMA fills it with zeros and no MMA reads it
  prm.num_k_tiles = static_cast<int>(k / 256);
  prm.sf_rows = static_cast<int>(k / 32);
  prm.dev_status = dev_status;
  prm.wait_limit_cycles = wait_limit_cycles;
  prm.f = static_cast<int>(f);
  prm.h_rec = h_rec;
  prm.clk = clk;
  if (gated) {
    st = cuda_check(cudaMemsetAsync(h_rec, 0, sizeof(nvfp4_scale_rec), stream), "memset h_rec");
    if (st != NVFP4_OK) return st;
  }

  auto kernel = gated ? k_fc2_gemm<true> : k_fc2_gemm<false>;
  const int smem = gated ? SMEM_BYTES + kSiluSmemBytes : SMEM_BYTES + EPI_WARPS * kOutSlotBytes;
  st = cuda_check(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                  "cudaFuncSetAttribute(k_fc2_gemm)");
  if (st != NVFP4_OK) return st;
  const int tiles = prm.num_m_tiles * prm.num_n_tiles;
  int max_pairs = 0;
  st = resident_pairs(gated, smem, &max_pairs);
  if (st != NVFP4_OK) return st;
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  kernel<<<2 * pairs, THREADS, smem, stream>>>(ta, tw, tsa, tsw, tout, prm);
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
__global__ void k_diag_silu_epilogue(uint16_t* out) {
  __shared__ uint16_t tab_s[2 * kSiluHalf];
  fill_silu_smem(tab_s);
  __syncthreads();
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < 65536u; g += gridDim.x * blockDim.x)
    out[g] = static_cast<uint16_t>(silu_bf16_epi(g, tab_s));
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_fc2_gemm(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                                       const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m,
                                       int64_t n, int64_t k, void* out_bf16, int64_t ldo, uint32_t* dev_status,
                                       nvfp4_stream_t stream) {
  return gemm_launch(a_q, a_s, a_rec, w_q, w_s, w_rec, m, n, k, out_bf16, ldo, 0, nullptr, dev_status,
                     reinterpret_cast<cudaStream_t>(stream), kDefaultWaitLimitCycles, "nvfp4_fc2_gemm");
}

extern "C" nvfp4_status nvfp4_fc1_swiglu(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                                         const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m,
                                         int64_t f, int64_t k, void* h_bf16, int64_t ldh, nvfp4_scale_rec* h_rec,
                                         uint32_t* dev_status, nvfp4_stream_t stream) {
  if (f < 1) return fail(NVFP4_EINVAL, "nvfp4_fc1_swiglu: f must be >= 1");
  return gemm_launch(a_q, a_s, a_rec, w_q, w_s, w_rec, m, 2 * f, k, h_bf16, ldh, f, h_rec, dev_status,
                     reinterpret_cast<cudaStream_t>(stream), kDefaultWaitLimitCycles, "nvfp4_fc1_swiglu");
}

extern "C" nvfp4_status nvfp4_diag_fc2_gemm_clock(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                                                  const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec,
                                                  int64_t m, int64_t n, int64_t k, void* out_bf16, int64_t ldo,
                                                  uint32_t* dev_status, uint64_t* clk, nvfp4_stream_t stream) {
  if (!clk || reinterpret_cast<uintptr_t>(clk) % 8 != 0)
    return fail(NVFP4_EINVAL, "nvfp4_diag_fc2_gemm_clock: clk must be an 8-byte aligned device pointer");
  return gemm_launch(a_q, a_s, a_rec, w_q, w_s, w_rec, m, n, k, out_bf16, ldo, 0, nullptr, dev_status,
                     reinterpret_cast<cudaStream_t>(stream), kDefaultWaitLimitCycles, "nvfp4_diag_fc2_gemm_clock", clk);
}

extern "C" nvfp4_status nvfp4_diag_wait_timeout(uint64_t limit_ns, uint32_t* dev_status, nvfp4_stream_t stream) {
  if (!dev_status || limit_ns < 1 || limit_ns > 1000000000ull)
    return fail(NVFP4_EINVAL, "nvfp4_diag_wait_timeout: bad arguments");
  // cycles at the highest SM clock (2.07 GHz) give at least limit_ns of wall time
  k_diag_wait_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns * 21 / 10, dev_status);
  return cuda_check(cudaGetLastError(), "launch k_diag_wait_timeout");
}

extern "C" nvfp4_status nvfp4_diag_silu_epilogue(uint16_t* out, nvfp4_stream_t stream) {
  if (!out) return fail(NVFP4_EINVAL, "nvfp4_diag_silu_epilogue: null pointer");
  k_diag_silu_epilogue<<<64, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out);
  return cuda_check(cudaGetLastError(), "launch k_diag_silu_epilogue");
}
