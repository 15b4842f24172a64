// Two-pass NVFP4 producers: the fused SwiGLU activation quantiser and the
// weight quantiser.
//
// "GB10 component-2 nsys summary", nvfp4: the unfused path runs absmax
// partials, a scale finalize, a block-scale zeroing and an activation pack
// as separate launches, and notes that the global scale must be known
// before any element is quantised.  "FC2 NVFP4 Scheduling Results",
// Canonical Operation: the accepted producer fuses SwiGLU into the NVFP4
// quantisation and pads M.  Here that is two streaming kernels:
//   pass 1  k_amax  : read gate|up (or W), form h, max |h| -> rec (one
//                     atomicMax per CTA on the bit pattern of a non-negative
//                     float, so the result is order independent)
//   pass 2  k_quant : re-read, form h again, per-16 block scale, E2M1 codes,
//                     two codes per byte, scales at the 128x4 tiled offset,
//                     pad rows and pad scale columns written as zero
// h is never stored.  The scale finalize is folded into pass 2's prologue,
// the zeroing into its stores.
//
// Work unit: one warp handles 512 consecutive elements of one row; lane l
// owns the 16-element block 16l..16l+15 (two 16-byte loads of gate, two of
// up), four lanes one 4-column group of scales.  SwiGLU kernels keep the
// 65,536-entry BF16 silu table (128 KB) in shared memory, one CTA per SM.
#include <cuda_bf16.h>

#include <cstdio>

#include "common.cuh"

namespace nvfp4 {
namespace {

// SwiGLU kernels run one CTA per SM with the whole silu table (128 KB) in
// shared memory: 1024 threads for pass 1, 768 for pass 2 (which keeps the
// next unit's loads in registers while it computes, 80 registers a thread);
// weight kernels need no table.
constexpr int kThreadsAmaxSwiglu = 1024;
constexpr int kThreadsQuantSwiglu = 768;
constexpr int kThreadsWeight = 256;
constexpr int kSegElems = 512;  // elements of one row handled by one warp per unit (16 per lane)
constexpr int kTableBytes = 65536 * 2;

// Correctly rounded BF16 silu of every BF16 gate, indexed by its bit pattern;
// generated at build time by gen_silu_table.py.  Closed forms behind it:
// |g| < 2^-10 gives g/2 (a lost bit rounds toward +inf: silu(g) > g/2),
// g >= 8 gives g, g <= -128 gives -0, +inf gives +inf, -inf and NaN give NaN.
__device__ const uint16_t k_silu_tab[65536] = {
#include "silu_table_full.inc"
};

__device__ __forceinline__ float bf16_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// silu of both BF16 gates in a word, as a BF16 pair.
__device__ __forceinline__ uint32_t silu_pair(uint32_t gw, const uint16_t* tab) {
  return uint32_t(tab[gw & 0xFFFFu]) | (uint32_t(tab[gw >> 16]) << 16);
}

// Two SwiGLU outputs h = RNE_bf16(silu_bf16(g) * u): the BF16 product of two
// BF16 values is their exact binary32 product rounded once (mul.rn.bf16x2).
__device__ __forceinline__ uint32_t swiglu_pair(uint32_t gw, uint32_t uw, const uint16_t* tab) {
  const uint32_t sw = silu_pair(gw, tab);
  const __nv_bfloat162 h = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&sw),
                                   *reinterpret_cast<const __nv_bfloat162*>(&uw));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Elementwise max of two BF16 pairs (NaN propagates).
__device__ __forceinline__ uint32_t max_pair(uint32_t a, uint32_t b) {
  const __nv_bfloat162 m = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                       *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}

template <bool kSwiglu>
__device__ __forceinline__ void load_table(uint16_t* tab) {
  if constexpr (kSwiglu) {
    const uint4* src = reinterpret_cast<const uint4*>(k_silu_tab);
    uint4* dst = reinterpret_cast<uint4*>(tab);
    for (int i = threadIdx.x; i < kTableBytes / 16; i += blockDim.x) dst[i] = src[i];
    __syncthreads();
  }
}

// Raw 16-element slice of one lane: 2 x 16 B of gate (or W) and, with
// SwiGLU, 2 x 16 B of up.
struct Slice {
  uint32_t g[8];
  uint32_t u[8];
};

template <bool kSwiglu, bool kStream>
__device__ __forceinline__ void load_slice(const uint16_t* row, uint32_t cols, uint32_t c0, Slice& s) {
  const uint4* pg = reinterpret_cast<const uint4*>(row + c0);
  uint4 a, b;
  if constexpr (kStream) {
    a = __ldcs(pg);
    b = __ldcs(pg + 1);
  } else {
    a = __ldg(pg);
    b = __ldg(pg + 1);
  }
  s.g[0] = a.x, s.g[1] = a.y, s.g[2] = a.z, s.g[3] = a.w, s.g[4] = b.x, s.g[5] = b.y, s.g[6] = b.z, s.g[7] = b.w;
  if constexpr (kSwiglu) {
    const uint4* pu = reinterpret_cast<const uint4*>(row + cols + c0);
    if constexpr (kStream) {
      a = __ldcs(pu);
      b = __ldcs(pu + 1);
    } else {
      a = __ldg(pu);
      b = __ldg(pu + 1);
    }
    s.u[0] = a.x, s.u[1] = a.y, s.u[2] = a.z, s.u[3] = a.w, s.u[4] = b.x, s.u[5] = b.y, s.u[6] = b.z, s.u[7] = b.w;
  }
}

// max |h| of a slice as a binary32 bit pattern (integer max keeps NaN: its bit
// patterns sort above +inf).
template <bool kSwiglu>
__device__ __forceinline__ uint32_t slice_absmax_bits(const Slice& s, const uint16_t* tab) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t hw = kSwiglu ? swiglu_pair(s.g[i], s.u[i], tab) : s.g[i];
    m = max(m, max((hw << 16) & 0x7FFFFFFFu, hw & 0x7FFF0000u));
  }
  return m;
}

// An upper bound of max |h| over a SwiGLU slice, exact to apply: |silu(g)|
// is at most max(g, 0.2785) for every g, hence at most max(|g|, 0.28125),
// so |h| = RNE(|silu_bf16(g) u|) <= RNE(max(|g|, 0.28125) |u|), which is
// what mul.rn.bf16x2 returns.  NaN and Inf inputs give a NaN or Inf bound.
__device__ __forceinline__ float slice_bound(const Slice& s) {
  const uint32_t c = 0x3E903E90u;  // 0.28125 in both halves
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t ga = max_pair(s.g[i] & 0x7FFF7FFFu, c);
    const uint32_t ua = s.u[i] & 0x7FFF7FFFu;
    const __nv_bfloat162 b = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&ga),
                                     *reinterpret_cast<const __nv_bfloat162*>(&ua));
    m = max_pair(m, *reinterpret_cast<const uint32_t*>(&b));
  }
  // the larger half, by bit pattern so that a NaN half wins
  return __uint_as_float(max((m << 16) & 0x7FFFFFFFu, m & 0x7FFF0000u));
}

// Walks the units (row, segment) of a [rows, cols] grid, grid-strided over
// warps, without a division in the loop.  Indices are 32-bit: the host
// refuses tensors with 2^31 or more units or padded rows (integer index
// arithmetic was half of pass 2's instructions in 64 bits).
struct UnitWalker {
  uint32_t row, seg;
  uint32_t step_rows, step_segs, segs;
  __device__ UnitWalker(uint32_t first, uint32_t stride, uint32_t segs_) : segs(segs_) {
    row = first / segs;
    seg = first - row * segs;
    step_rows = stride / segs;
    step_segs = stride - step_rows * segs;
  }
  __device__ __forceinline__ void next() {
    row += step_rows;
    seg += step_segs;
    if (seg >= segs) {
      seg -= segs;
      ++row;
    }
  }
};

// Pass 1: rec->amax_bits = max over the tensor of the bit pattern of |h|.
// Each lane keeps the exact max of what it has evaluated; a SwiGLU slice whose
// bound does not exceed that max cannot change it and is skipped.  Two units
// in flight per warp; loads keep the default L2 policy so the tail of the
// tensor is still in L2 when pass 2 (which walks backwards) starts.
template <bool kSwiglu>
__global__ void __launch_bounds__(kSwiglu ? kThreadsAmaxSwiglu : kThreadsWeight)
    k_amax(const uint16_t* __restrict__ x, uint32_t rows, uint32_t cols, uint32_t ld, nvfp4_scale_rec* rec) {
  extern __shared__ __align__(16) uint16_t tab[];
  __shared__ uint32_t wmax[32];
  load_table<kSwiglu>(tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint32_t segs = (cols + kSegElems - 1) / kSegElems;
  const uint32_t first = blockIdx.x * uint32_t(nwarps) + uint32_t(warp);
  const uint32_t stride = gridDim.x * uint32_t(nwarps);
  uint32_t amax = 0;  // bit pattern of the exact max |h| this lane has evaluated
  UnitWalker w(first, stride, segs);
  while (w.row < rows) {
    const uint32_t r0 = w.row, c0 = w.seg * kSegElems + lane * 16;
    w.next();
    const uint32_t r1 = w.row, c1 = w.seg * kSegElems + lane * 16;
    w.next();
    Slice s0, s1;
    const bool v0 = c0 < cols, v1 = r1 < rows && c1 < cols;
    if (v0) load_slice<kSwiglu, false>(x + uint64_t(r0) * ld, cols, c0, s0);
    if (v1) load_slice<kSwiglu, false>(x + uint64_t(r1) * ld, cols, c1, s1);
    if constexpr (kSwiglu) {
      // exact evaluation only where the bound could beat the running max
      if (v0 && !(slice_bound(s0) <= __uint_as_float(amax))) amax = max(amax, slice_absmax_bits<true>(s0, tab));
      if (v1 && !(slice_bound(s1) <= __uint_as_float(amax))) amax = max(amax, slice_absmax_bits<true>(s1, tab));
    } else {
      if (v0) amax = max(amax, slice_absmax_bits<false>(s0, tab));
      if (v1) amax = max(amax, slice_absmax_bits<false>(s1, tab));
    }
  }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int i = 0; i < nwarps; ++i) m = max(m, wmax[i]);
    if (m != 0) atomicMax(&rec->amax_bits, m);
  }
}

// True when q is within 3 units in the last place of a binary32 number with
// at most `sig` significant bits (every rounding boundary of a format with
// sig-1 fraction bits is such a number).  Used to send the rare quotients
// whose rounding a multiply-by-reciprocal could get wrong to a true division.
template <int kSig>
__device__ __forceinline__ bool near_boundary(float q) {
  constexpr uint32_t mask = (1u << (24 - kSig)) - 1u;
  return ((__float_as_uint(q) + 3u) & mask) <= 6u;
}

// Two binary32 products RN(a*s), RN(b*s) in one packed multiply.
__device__ __forceinline__ void mul2_rn(float a, float b, float s, float& x, float& y) {
  asm("{\n\t.reg .b64 t, u, v;\n\t"
      "mov.b64 t, {%2, %3};\n\t"
      "mov.b64 u, {%4, %4};\n\t"
      "mul.rn.f32x2 v, t, u;\n\t"
      "mov.b64 {%0, %1}, v;\n\t}"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "f"(s));
}

// Two binary32 fused multiply-adds RN(a*b + c) in one packed instruction.
__device__ __forceinline__ void fma2_rn(float a0, float a1, float b0, float b1, float c0, float c1, float& x,
                                        float& y) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(x), "=f"(y)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Eight E2M1 codes (RNE, satfinite) packed two per byte, q[0] in bits 0..3.
__device__ __forceinline__ uint32_t e2m1x8_pack(const float* q) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return w;
}

// The 16 E2M1 codes of one block, packed two per byte (element 0 in bits
// 0..3 of .x): E2M1(RN(h / sc)) for the 16 BF16 values in hw (two per word),
// sc > 0 the block's decoded scale and rs = RN(1 / sc).
// n = RN(h * -rs) = -RN(h * rs) is corrected once, Markstein's step (IBM J.
// Res. Dev. 34, 1990): the residual r = h + n*sc is exact as one fma, and
// RN(n + r*(-rs)) = -RN(q + r*rs) then rounds like -h / sc wherever an E2M1
// code can change.  Working on -q keeps the sign of a zero h (+0 and -0 give
// codes 0 and 8); the sign bits of the packed codes are flipped at the end.
// Blocks with a scale below 2^-100 (a global max below ~1e-27) keep the
// plain product and divide the quotients within 3 ulps of a
// 3-significant-bit number, which also catches an infinite reciprocal.
// Over every BF16 h, block-scale code and BF16 global max the codes equal
// those of the correctly rounded quotient (nvfp4_diag_quotient_codes).
__device__ __forceinline__ uint2 block_codes(const uint32_t* hw, float sc, float rs) {
  const float nrs = -rs;
  float n[16];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    mul2_rn(bf16_to_f32(hw[i] & 0xFFFFu), __uint_as_float(hw[i] & 0xFFFF0000u), nrs, n[2 * i], n[2 * i + 1]);
  if (sc >= 0x1p-100f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float r0, r1;
      fma2_rn(n[2 * i], n[2 * i + 1], sc, sc, bf16_to_f32(hw[i] & 0xFFFFu), __uint_as_float(hw[i] & 0xFFFF0000u),
              r0, r1);
      fma2_rn(r0, r1, nrs, nrs, n[2 * i], n[2 * i + 1], n[2 * i], n[2 * i + 1]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (near_boundary<3>(n[j]))
        n[j] = __fdiv_rn((j & 1) ? __uint_as_float(hw[j >> 1] & 0xFFFF0000u) : bf16_to_f32(hw[j >> 1] & 0xFFFFu), -sc);
  }
  return make_uint2(e2m1x8_pack(n) ^ 0x88888888u, e2m1x8_pack(n + 8) ^ 0x88888888u);
}

// Block scale code of a block with max |h| = bmax: E4M3(RN(bmax / d)).
__device__ __forceinline__ uint32_t block_scale_code(float bmax, float d, float rd) {
  if (d == 0.0f) return 0u;
  float r = __fmul_rn(bmax, rd);
  if (near_boundary<5>(r)) r = __fdiv_rn(bmax, d);
  return e4m3_code(r);
}

// One lane's 16-element block of pass 2 at row r, columns cb .. cb+15:
// `loaded` when the slice holds it (r < rows, inside the columns, finite
// global max), `valid` when the block lies inside the columns (else nothing
// is stored).  Writes the packed codes and, from the first lane of each four
// (one 64-element scale group), the group's scale word.  Every lane of the
// warp calls it together (the scale word is gathered with shuffles).
template <bool kSwiglu>
__device__ __forceinline__ void quant_block(const Slice& sl, bool loaded, bool valid, uint32_t r, uint32_t cb,
                                            uint32_t cols, uint32_t cpad4, float g, float d, float rd, bool finite,
                                            const uint16_t* tab, uint8_t* __restrict__ qdata,
                                            uint8_t* __restrict__ scales, int lane) {
  uint32_t hw[8];  // 16 BF16 values of h, two per word
  if (loaded) {
#pragma unroll
    for (int i = 0; i < 8; ++i) hw[i] = kSwiglu ? swiglu_pair(sl.g[i], sl.u[i], tab) : sl.g[i];
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) hw[i] = 0u;
  }
  // |h| max per half; no NaN reaches here (a NaN or Inf anywhere makes the
  // global max non-finite, and then no element is read)
  __nv_bfloat162 mh = __floats2bfloat162_rn(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < 8; ++i) mh = __hmax2(mh, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&hw[i])));
  const uint32_t m2 = *reinterpret_cast<const uint32_t*>(&mh);
  const float bmax = __uint_as_float(max((m2 << 16) & 0x7FFFFFFFu, m2 & 0x7FFF0000u));
  const uint32_t bs = finite ? block_scale_code(bmax, d, rd) : 0u;
  const float sc = __fmul_rn(e4m3_value(bs), g);
  uint2 packed = make_uint2(0u, 0u);
  if (sc != 0.0f && finite) packed = block_codes(hw, sc, __frcp_rn(sc));
  if (valid) *reinterpret_cast<uint2*>(qdata + uint64_t(r) * (cols / 2) + cb / 2) = packed;

  // scales: lanes 4j..4j+3 hold the four blocks of scale group j
  const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, bs, 1);
  const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, bs, 2);
  const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, bs, 3);
  const uint32_t grp = cb / 64;
  if ((lane & 3) == 0 && grp < cpad4) {
    const uint32_t off = ((r >> 7) * cpad4 + grp) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
    *reinterpret_cast<uint32_t*>(scales + off) = bs | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
}

// The global scale from pass 1's record (the bit pattern of max |h|); block
// 0 writes it and the status back to the record.
struct GlobalScale {
  bool finite;
  float g, d, rd;
};

__device__ __forceinline__ GlobalScale global_scale(nvfp4_scale_rec* rec) {
  const uint32_t amax_bits = *reinterpret_cast<volatile uint32_t*>(&rec->amax_bits);
  GlobalScale gs;
  gs.finite = amax_bits < 0x7F800000u;
  gs.g = gs.finite ? __fdiv_rn(__uint_as_float(amax_bits), 2688.0f) : __uint_as_float(0x7FC00000u);
  gs.d = __fmul_rn(6.0f, gs.g);
  gs.rd = (gs.d == 0.0f || !gs.finite) ? 0.0f : __frcp_rn(gs.d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    rec->global_scale = gs.g;
    rec->status = gs.finite ? NVFP4_OK : NVFP4_ENONFINITE;
  }
  return gs;
}

// Pass 2: quantise.  One lane = one 16-element block of each 512-element
// segment of its unit.  Units cover rows
// [0, rows_pad), walked from the end so that the first reads hit what pass 1
// left in L2; rows >= rows are zeros.
template <bool kSwiglu, int kB>
__global__ void __launch_bounds__(kSwiglu ? kThreadsQuantSwiglu : kThreadsWeight, kSwiglu ? 1 : (kB == 2 ? 3 : 4))
    k_quant(const uint16_t* __restrict__ x, uint32_t rows, uint32_t cols, uint32_t ld, uint32_t rows_pad,
            uint8_t* __restrict__ qdata, uint8_t* __restrict__ scales, nvfp4_scale_rec* rec) {
  extern __shared__ __align__(16) uint16_t tab[];
  load_table<kSwiglu>(tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const GlobalScale gs = global_scale(rec);
  const bool finite = gs.finite;

  // A unit is kB consecutive 512-element segments of one row; lane l owns
  // the 16-element block 16l of each.  The plain quantiser takes two blocks
  // a lane on rows that are whole 1024-element units, which halves the
  // per-unit bookkeeping per element (4-6% faster at 7168 and 14336 columns;
  // on a row with a partial last unit the idle half cost more than that).
  static_assert(kB == 1 || (kB == 2 && !kSwiglu), "two blocks a lane for the plain quantiser only");
  constexpr uint32_t kUnit = kSegElems * kB;
  const uint32_t segs = (cols + kUnit - 1) / kUnit;
  const uint32_t cpad4 = (cols / 16 + 3) / 4;  // 4-column scale groups per row
  const uint32_t first = blockIdx.x * uint32_t(nwarps) + uint32_t(warp);
  const uint32_t stride = gridDim.x * uint32_t(nwarps);
  // Software pipeline: the loads of the next unit are issued before the
  // current one is computed, so a warp keeps its loads in flight while it
  // works (pass 2 is otherwise latency bound on them).
  UnitWalker w(first, stride, segs);
  uint32_t r_n = rows_pad - 1 - w.row, seg_n = segs - 1 - w.seg;
  bool more = w.row < rows_pad;
  Slice s_n[kB];
  {
    const uint32_t c0 = seg_n * kUnit + lane * 16;
#pragma unroll
    for (int b = 0; b < kB; ++b)
      if (more && c0 + b * kSegElems < cols && finite && r_n < rows)
        load_slice<kSwiglu, true>(x + uint64_t(r_n) * ld, cols, c0 + b * kSegElems, s_n[b]);
  }
  while (more) {
    const uint32_t r = r_n, seg = seg_n;
    const uint32_t c0 = seg * kUnit + lane * 16;
    Slice s[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) s[b] = s_n[b];
    w.next();
    more = w.row < rows_pad;
    r_n = rows_pad - 1 - w.row;
    seg_n = segs - 1 - w.seg;
    {
      const uint32_t c0n = seg_n * kUnit + lane * 16;
#pragma unroll
      for (int b = 0; b < kB; ++b)
        if (more && c0n + b * kSegElems < cols && finite && r_n < rows)
          load_slice<kSwiglu, true>(x + uint64_t(r_n) * ld, cols, c0n + b * kSegElems, s_n[b]);
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const uint32_t cb = c0 + b * kSegElems;
      const bool valid = cb < cols;
      quant_block<kSwiglu>(s[b], valid && finite && r < rows, valid, r, cb, cols, cpad4, gs.g, gs.d, gs.rd, finite,
                           tab, qdata, scales, lane);
    }
  }
}

// Pass 2 of the plain quantiser over the padded [rows_pad, cols] grid read
// as one sequence of 1024-element units (row-major, so a unit may end in
// one row and go on in the next).  For cols a multiple of 64 and at least
// 1024 that are not whole 1024-element units (5376 = 5.25 x 1024): every
// lane then takes two blocks, where the row walk leaves half a unit of idle
// lanes at each row end and one block a lane.  A 64-element scale group
// never straddles two rows (cols % 64 == 0), a unit at most two (cols >=
// 1024).  Units are walked from the end, as in k_quant.
__global__ void __launch_bounds__(kThreadsWeight, 3)
    k_quant_flat(const uint16_t* __restrict__ x, uint32_t rows, uint32_t cols, uint32_t ld, uint32_t rows_pad,
                 uint8_t* __restrict__ qdata, uint8_t* __restrict__ scales, nvfp4_scale_rec* rec) {
  constexpr uint32_t kUnit = 2 * kSegElems;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const GlobalScale gs = global_scale(rec);
  const bool finite = gs.finite;
  const uint32_t cpad4 = cols / 64;
  const uint32_t units = uint32_t((uint64_t(rows_pad) * cols) / kUnit);  // exact: rows_pad % 128, cols % 64
  const uint32_t first = blockIdx.x * uint32_t(nwarps) + uint32_t(warp);
  const uint32_t stride = gridDim.x * uint32_t(nwarps);
  // (r, c): the first element of the current unit; stepping back `stride`
  // units moves it back by dq rows and dr columns (with a borrow).
  const uint32_t step = stride * kUnit;
  const uint32_t dq = step / cols, dr = step - dq * cols;
  uint32_t f = first;
  uint32_t r = 0, c = 0;
  if (f < units) {
    const uint64_t e0 = uint64_t(units - 1 - f) * kUnit;
    r = uint32_t(e0 / cols);
    c = uint32_t(e0 - uint64_t(r) * cols);
  }
  // this lane's block b of the unit at (r, c): row and column
  auto block_at = [&](uint32_t ur, uint32_t uc, int b, uint32_t& br, uint32_t& bc) {
    bc = uc + uint32_t(b) * kSegElems + uint32_t(lane) * 16;
    br = ur;
    if (bc >= cols) {
      bc -= cols;
      ++br;
    }
  };
  Slice s_n[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    uint32_t br, bc;
    block_at(r, c, b, br, bc);
    if (f < units && finite && br < rows) load_slice<false, true>(x + uint64_t(br) * ld, cols, bc, s_n[b]);
  }
  while (f < units) {
    const uint32_t ur = r, uc = c;
    Slice s[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) s[b] = s_n[b];
    f += stride;
    if (c < dr) {
      c = c + cols - dr;
      r -= dq + 1;
    } else {
      c -= dr;
      r -= dq;
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      uint32_t br, bc;
      block_at(r, c, b, br, bc);
      if (f < units && finite && br < rows) load_slice<false, true>(x + uint64_t(br) * ld, cols, bc, s_n[b]);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      uint32_t br, bc;
      block_at(ur, uc, b, br, bc);
      quant_block<false>(s[b], finite && br < rows, true, br, bc, cols, cpad4, gs.g, gs.d, gs.rd, finite, nullptr,
                         qdata, scales, lane);
    }
  }
}

template <typename K>
nvfp4_status launch_stream_kernel(K kernel, bool swiglu, int threads, cudaStream_t stream, const char* name,
                                  auto... args) {
  const int smem = swiglu ? kTableBytes : 0;
  nvfp4_status st = cuda_check(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem), name);
  if (st != NVFP4_OK) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  kernel<<<sm_count() * per_sm, threads, smem, stream>>>(args...);
  return cuda_check(cudaGetLastError(), name);
}

// given_amax: rec->amax_bits already holds max |x| (from the SwiGLU epilogue
// of FC1), so only pass 2 runs; the plain quantiser is then applied to x.
nvfp4_status quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, bool swiglu, void* qdata,
                      void* scales, nvfp4_scale_rec* rec, cudaStream_t stream, const char* name,
                      bool given_amax = false) {
  if (!x || !qdata || !scales || !rec) return fail(NVFP4_EINVAL, std::string(name) + ": null pointer");
  if (rows < 1 || cols < 16) return fail(NVFP4_EINVAL, std::string(name) + ": rows must be >= 1 and cols >= 16");
  if (cols % 16 != 0) return fail(NVFP4_EUNSUPPORTED, std::string(name) + ": cols must be a multiple of 16");
  const int64_t need = swiglu ? 2 * cols : cols;
  if (ld < need) return fail(NVFP4_EINVAL, std::string(name) + ": ld too small");
  if (ld % 8 != 0 || !aligned16(x) || !aligned16(qdata) || !aligned16(scales) || !aligned16(rec))
    return fail(NVFP4_EALIGN, std::string(name) + ": pointers must be 16-byte aligned and ld a multiple of 8");
  const int64_t rows_pad = nvfp4_padded_rows(rows);
  // the kernels index units, rows, columns and scale bytes in 32 bits
  const int64_t limit = int64_t(1) << 31;
  if (cols > (int64_t(1) << 30) || ld >= limit || rows_pad >= limit ||
      rows_pad * ((cols + kSegElems - 1) / kSegElems) >= limit || nvfp4_scale_bytes(rows, cols) >= limit)
    return fail(NVFP4_EUNSUPPORTED, std::string(name) + ": tensor too large");
  const uint32_t rows32 = static_cast<uint32_t>(rows), cols32 = static_cast<uint32_t>(cols);
  const uint32_t ld32 = static_cast<uint32_t>(ld), rows_pad32 = static_cast<uint32_t>(rows_pad);
  const uint16_t* xin = static_cast<const uint16_t*>(x);
  uint8_t* q = static_cast<uint8_t*>(qdata);
  uint8_t* s = static_cast<uint8_t*>(scales);

  // The plain pass 2 takes two blocks a lane: along each row when it is whole
  // 1024-element units, else over the grid read as one sequence of units
  // when cols allows (a multiple of 64, at least 1024), else one block a lane.
  auto quant_plain = (cols % (2 * kSegElems) == 0)            ? k_quant<false, 2>
                     : (cols % 64 == 0 && cols >= 2 * kSegElems) ? k_quant_flat
                                                                 : k_quant<false, 1>;
  nvfp4_status st;
  if (given_amax)
    return launch_stream_kernel(quant_plain, false, kThreadsWeight, stream, "launch k_quant", xin, rows32, cols32, ld32,
                                rows_pad32, q, s, rec);
  st = cuda_check(cudaMemsetAsync(rec, 0, sizeof(nvfp4_scale_rec), stream), "memset rec");
  if (st != NVFP4_OK) return st;
  if (swiglu) {
    if ((st = launch_stream_kernel(k_amax<true>, true, kThreadsAmaxSwiglu, stream, "launch k_amax", xin, rows32, cols32, ld32, rec)) != NVFP4_OK)
      return st;
    return launch_stream_kernel(k_quant<true, 1>, true, kThreadsQuantSwiglu, stream, "launch k_quant", xin, rows32, cols32, ld32, rows_pad32, q, s, rec);
  }
  if ((st = launch_stream_kernel(k_amax<false>, false, kThreadsWeight, stream, "launch k_amax", xin, rows32, cols32, ld32, rec)) != NVFP4_OK)
    return st;
  return launch_stream_kernel(quant_plain, false, kThreadsWeight, stream, "launch k_quant", xin, rows32, cols32, ld32, rows_pad32, q, s, rec);
}

// ---- diagnostics: the same device functions on test-chosen inputs ----------

__global__ void k_diag_silu_all(uint16_t* out) {
  extern __shared__ __align__(16) uint16_t tab[];
  load_table<true>(tab);
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < 65536u; g += gridDim.x * blockDim.x)
    out[g] = static_cast<uint16_t>(silu_pair(g, tab) & 0xFFFFu);
}

// SwiGLU through the producer's pass-2 path (swiglu_pair, both halves of the
// word), checked against pass 1's path (exact product, rounded once at the
// end) and pass 1's bound; a disagreement is reported as the NaN pattern
// 0x7FFF, which never equals the oracle.
__global__ void k_diag_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t n) {
  extern __shared__ __align__(16) uint16_t tab[];
  load_table<true>(tab);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t gw = gate[i] | (uint32_t(gate[i]) << 16), uw = up[i] | (uint32_t(up[i]) << 16);
    const uint32_t pair = swiglu_pair(gw, uw, tab);
    const float p = __fmul_rn(bf16_to_f32(tab[gate[i]]), bf16_to_f32(up[i]));
    const uint32_t pa = __float_as_uint(p) & 0x7FFFFFFFu;
    const uint32_t p1 = (pa >= 0x7F800000u ? pa : (bf16x2_rn(__uint_as_float(pa), 0.0f) << 16)) >> 16;
    Slice s;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      s.g[k] = gw;
      s.u[k] = uw;
    }
    const float bound = slice_bound(s);
    const uint32_t lo = pair & 0xFFFFu, hi = pair >> 16;
    const bool nan_h = (lo & 0x7FFFu) > 0x7F80u;
    const bool bound_ok = nan_h || isnan(bound) || bf16_to_f32(lo & 0x7FFFu) <= bound;
    const bool ok = lo == hi && ((lo & 0x7FFFu) == p1 || (nan_h && p1 > 0x7F80u)) && bound_ok;
    h[i] = static_cast<uint16_t>(ok ? lo : 0x7FFFu);
  }
}

__device__ __forceinline__ uint32_t diag_code(int which, uint32_t bits) {
  const float f = __uint_as_float(bits);
  if (which == 0) {
    // the packed encoder in both slots; a slot disagreement shows up as an
    // out-of-range code
    const uint32_t lo = e2m1x2_code(f, 0.0f) & 0xFu, hi = e2m1x2_code(0.0f, f) >> 4;
    return lo == hi ? lo : 0x100u | lo;
  }
  return e4m3_code(f);
}

__global__ void k_diag_transitions(int which, uint32_t* trans, uint32_t cap, uint32_t* count,
                                   uint32_t* first_code) {
  const uint64_t total = uint64_t(1) << 32;
  for (uint64_t p = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; p < total;
       p += uint64_t(gridDim.x) * blockDim.x) {
    const uint32_t b = static_cast<uint32_t>(p);
    if (b == 0) {
      *first_code = diag_code(which, 0u);
      continue;
    }
    const uint32_t a = b - 1u;
    if (((a >> 23) & 0xFFu) == 0xFFu || ((b >> 23) & 0xFFu) == 0xFFu) continue;
    const uint32_t cb = diag_code(which, b), ca = diag_code(which, a);
    if (cb != ca) {
      const uint32_t i = atomicAdd(count, 1u);
      if (i < cap) {
        trans[3 * i] = b;
        trans[3 * i + 1] = cb;
        trans[3 * i + 2] = ca;
      }
    }
  }
}

// Every (global max, block-scale code, h) through block_codes, against the
// definition E2M1(RN(h / sc)) with RN(h / sc) from the correctly rounded
// division.  Global maxima A are the BF16 patterns a_first .. a_first +
// a_count - 1 (g = RN(A / 2688), as pass 2 forms it), block-scale codes
// 1..126 (sc = RN(E4M3(bs) * g), blocks with sc = 0 are never encoded), and
// every BF16 h of either sign with |h| <= A (a block's values never exceed
// the global max), 16 to a block.
// counts[0] += codes that differ, counts[1] += codes compared.
__global__ void k_diag_quotient_codes(uint32_t a_first, uint32_t a_count, unsigned long long* counts) {
  constexpr uint32_t kFinite = 0x7F80u;            // non-negative finite BF16 patterns
  constexpr uint32_t kChunks = 2 * kFinite / 16;  // blocks of 16 values, both signs
  unsigned long long bad = 0, seen = 0;
  const uint64_t items = uint64_t(a_count) * 126u * kChunks;
  for (uint64_t it = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; it < items;
       it += uint64_t(gridDim.x) * blockDim.x) {
    const uint32_t chunk = uint32_t(it % kChunks);
    const uint32_t bs = 1u + uint32_t((it / kChunks) % 126u);
    const uint32_t abits = a_first + uint32_t(it / (uint64_t(kChunks) * 126u));
    const float g = __fdiv_rn(bf16_to_f32(abits), 2688.0f);
    const float sc = __fmul_rn(e4m3_value(bs), g);
    if (!(sc > 0.0f)) continue;
    uint32_t hb[16], hw[8];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t k = chunk * 16u + uint32_t(j);
      hb[j] = k < kFinite ? k : 0x8000u + (k - kFinite);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) hw[i] = hb[2 * i] | (hb[2 * i + 1] << 16);
    const uint2 c = block_codes(hw, sc, __frcp_rn(sc));
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if ((hb[j] & 0x7FFFu) > abits) continue;
      const uint32_t got = ((j < 8 ? c.x : c.y) >> (4 * (j & 7))) & 0xFu;
      const uint32_t want = e2m1x2_code(__fdiv_rn(bf16_to_f32(hb[j]), sc), 0.0f) & 0xFu;
      bad += got != want ? 1u : 0u;
      ++seen;
    }
  }
  atomicAdd(&counts[0], bad);
  atomicAdd(&counts[1], seen);
}

// Every (global max, block max) through block_scale_code, against the
// definition E4M3(RN(bmax / d)) with d = RN(6 g), g = RN(A / 2688) as pass 2
// forms them and RN(bmax / d) the correctly rounded division.  Global
// maxima A are the BF16 patterns a_first .. a_first + a_count - 1; block
// maxima every finite non-negative BF16 pattern (above A too, so that the
// saturating end of the encoder is reached).
// counts[0] += codes that differ, counts[1] += codes compared.
__global__ void k_diag_block_scale_codes(uint32_t a_first, uint32_t a_count, unsigned long long* counts) {
  constexpr uint32_t kFinite = 0x7F80u;  // non-negative finite BF16 patterns
  unsigned long long bad = 0, seen = 0;
  const uint64_t items = uint64_t(a_count) * kFinite;
  for (uint64_t it = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; it < items;
       it += uint64_t(gridDim.x) * blockDim.x) {
    const uint32_t bbits = uint32_t(it % kFinite);
    const uint32_t abits = a_first + uint32_t(it / kFinite);
    const float g = __fdiv_rn(bf16_to_f32(abits), 2688.0f);
    const float d = __fmul_rn(6.0f, g);
    const float rd = d == 0.0f ? 0.0f : __frcp_rn(d);
    const float bmax = bf16_to_f32(bbits);
    const uint32_t got = block_scale_code(bmax, d, rd);
    const uint32_t want = d == 0.0f ? 0u : e4m3_code(__fdiv_rn(bmax, d));
    bad += got != want ? 1u : 0u;
    ++seen;
  }
  atomicAdd(&counts[0], bad);
  atomicAdd(&counts[1], seen);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_quantize_weight(const void* w_bf16, int64_t rows, int64_t cols, int64_t ld,
                                              void* qdata, void* scales, nvfp4_scale_rec* rec,
                                              nvfp4_stream_t stream) {
  return quantize(w_bf16, rows, cols, ld, false, qdata, scales, rec, reinterpret_cast<cudaStream_t>(stream),
                  "nvfp4_quantize_weight");
}

extern "C" nvfp4_status swiglu_nvfp4_quantize(const void* gate_up_bf16, int64_t m, int64_t k, int64_t ld,
                                              void* qdata, void* scales, nvfp4_scale_rec* rec,
                                              nvfp4_stream_t stream) {
  return quantize(gate_up_bf16, m, k, ld, true, qdata, scales, rec, reinterpret_cast<cudaStream_t>(stream),
                  "swiglu_nvfp4_quantize");
}

extern "C" nvfp4_status nvfp4_quantize_with_amax(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                                                 void* qdata, void* scales, nvfp4_scale_rec* rec,
                                                 nvfp4_stream_t stream) {
  return quantize(x_bf16, rows, cols, ld, false, qdata, scales, rec, reinterpret_cast<cudaStream_t>(stream),
                  "nvfp4_quantize_with_amax", true);
}

extern "C" nvfp4_status nvfp4_diag_silu_all(uint16_t* out, nvfp4_stream_t stream) {
  if (!out || !aligned16(out)) return fail(NVFP4_EINVAL, "nvfp4_diag_silu_all: bad pointer");
  nvfp4_status st = cuda_check(
      cudaFuncSetAttribute(k_diag_silu_all, cudaFuncAttributeMaxDynamicSharedMemorySize, kTableBytes), "diag silu");
  if (st != NVFP4_OK) return st;
  k_diag_silu_all<<<64, 256, kTableBytes, reinterpret_cast<cudaStream_t>(stream)>>>(out);
  return cuda_check(cudaGetLastError(), "launch k_diag_silu_all");
}

extern "C" nvfp4_status nvfp4_diag_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t n,
                                          nvfp4_stream_t stream) {
  if (!gate || !up || !h || n < 1) return fail(NVFP4_EINVAL, "nvfp4_diag_swiglu: bad arguments");
  nvfp4_status st = cuda_check(
      cudaFuncSetAttribute(k_diag_swiglu, cudaFuncAttributeMaxDynamicSharedMemorySize, kTableBytes), "diag swiglu");
  if (st != NVFP4_OK) return st;
  k_diag_swiglu<<<64, 256, kTableBytes, reinterpret_cast<cudaStream_t>(stream)>>>(gate, up, h, n);
  return cuda_check(cudaGetLastError(), "launch k_diag_swiglu");
}

extern "C" nvfp4_status nvfp4_diag_code_transitions(int which, uint32_t* trans, uint32_t cap, uint32_t* count,
                                                    uint32_t* first_code, nvfp4_stream_t stream) {
  if ((which != 0 && which != 1) || !trans || !count || !first_code || cap == 0)
    return fail(NVFP4_EINVAL, "nvfp4_diag_code_transitions: bad arguments");
  k_diag_transitions<<<sm_count() * 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(which, trans, cap, count,
                                                                                          first_code);
  return cuda_check(cudaGetLastError(), "launch k_diag_transitions");
}

extern "C" nvfp4_status nvfp4_diag_quotient_codes(uint32_t a_first, uint32_t a_count, uint64_t* counts,
                                                  nvfp4_stream_t stream) {
  if (!counts || a_count < 1 || a_first >= 0x7F80u || a_count > 0x7F80u - a_first)
    return fail(NVFP4_EINVAL, "nvfp4_diag_quotient_codes: bad arguments");
  k_diag_quotient_codes<<<sm_count() * 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      a_first, a_count, reinterpret_cast<unsigned long long*>(counts));
  return cuda_check(cudaGetLastError(), "launch k_diag_quotient_codes");
}

extern "C" nvfp4_status nvfp4_diag_block_scale_codes(uint32_t a_first, uint32_t a_count, uint64_t* counts,
                                                     nvfp4_stream_t stream) {
  if (!counts || a_count < 1 || a_first >= 0x7F80u || a_count > 0x7F80u - a_first)
    return fail(NVFP4_EINVAL, "nvfp4_diag_block_scale_codes: bad arguments");
  k_diag_block_scale_codes<<<sm_count() * 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      a_first, a_count, reinterpret_cast<unsigned long long*>(counts));
  return cuda_check(cudaGetLastError(), "launch k_diag_block_scale_codes");
}
