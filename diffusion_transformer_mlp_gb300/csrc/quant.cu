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
// Work unit: one warp handles 256 consecutive elements of one row; lane l
// owns elements 8l..8l+7 (one 16-byte load of gate, one of up), a lane pair
// owns one 16-element block, eight lanes one 4-column group of scales.
#include <cuda_bf16.h>

#include <cstdio>

#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSiluEntries = 3840;
constexpr int kSegElems = 512;  // elements of one row handled by one warp per unit (16 per lane)

// Correctly rounded BF16 silu for gates with exponent field 117..129 (g > 0,
// entries 0..1663) and 117..133 (g < 0, entries 1664..3839), indexed by
// (g & 0x7FFF) - 117*128; generated at build time by gen_silu_table.py.
__device__ const uint16_t k_silu_mid[kSiluEntries] = {
#include "silu_mid_table.inc"
};

__device__ __forceinline__ float bf16_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// silu(g) rounded once to BF16, for the gates outside the table:
//   |g| < 2^-10 : silu(g) = g/2 + g^2/4 - ..., so the result is g/2, and when
//                 g/2 falls between two BF16 values the exact value lies
//                 above the midpoint: round toward +inf.
//   g >= 8      : the relative gap g - silu(g) < e^-8 < 2^-9: the result is g.
//   g <= -128   : |silu(g)| < 2^-134: the result is -0.
//   +inf -> +inf, -inf and NaN -> NaN (a non-finite gate stays non-finite).
__device__ __noinline__ float silu_outside_table(uint32_t g) {
  const uint32_t mag = g & 0x7FFFu;
  const uint32_t neg = g >> 15;
  uint32_t out;
  if (mag < 117u * 128u) {
    const uint32_t u = __float_as_uint(bf16_to_f32(g) * 0.5f);  // exact, no flush to zero
    out = (u + (neg ? 0x7FFFu : 0x8000u)) >> 16;
  } else if (mag >= 0x7F80u) {
    out = (g == 0x7F80u) ? 0x7F80u : 0x7FC0u;
  } else {
    out = neg ? 0x8000u : g;
  }
  return bf16_to_f32(out);
}

// silu(g) rounded once to BF16 (returned as its binary32 value); the common
// case is one shared-memory load from the table (entries stored as binary32).
__device__ __forceinline__ float silu_bf16(uint32_t g, const float* tab) {
  const uint32_t rel = (g & 0x7FFFu) - 117u * 128u;
  const bool neg = (g & 0x8000u) != 0;
  if (rel < (neg ? 2176u : 1664u)) return tab[rel + (neg ? 1664u : 0u)];
  return silu_outside_table(g);
}

// The exact binary32 product silu_bf16(g) * u (two BF16 significands: no
// rounding); h = RNE_bf16 of it.
__device__ __forceinline__ float swiglu_product(uint32_t g, uint32_t u, const float* tab) {
  return __fmul_rn(silu_bf16(g, tab), bf16_to_f32(u));
}

// Two SwiGLU outputs as BF16 bits (lo in bits 0..15).
__device__ __forceinline__ uint32_t swiglu_pair(uint32_t gw, uint32_t uw, const float* tab) {
  return bf16x2_rn(swiglu_product(gw & 0xFFFFu, uw & 0xFFFFu, tab), swiglu_product(gw >> 16, uw >> 16, tab));
}

template <bool kSwiglu>
__device__ __forceinline__ void load_table(float* tab) {
  if constexpr (kSwiglu) {
    for (int i = threadIdx.x; i < kSiluEntries; i += blockDim.x) tab[i] = bf16_to_f32(k_silu_mid[i]);
    __syncthreads();
  }
}

// Raw 16-element slice of one lane: 2 x 16 B of gate (or W) and, with
// SwiGLU, 2 x 16 B of up.
struct Slice {
  uint4 g[2];
  uint4 u[2];
};

template <bool kSwiglu, bool kStream>
__device__ __forceinline__ void load_slice(const uint16_t* row, int64_t cols, int64_t c0, Slice& s) {
  const uint4* pg = reinterpret_cast<const uint4*>(row + c0);
  if constexpr (kStream) {
    s.g[0] = __ldcs(pg);
    s.g[1] = __ldcs(pg + 1);
  } else {
    s.g[0] = __ldg(pg);
    s.g[1] = __ldg(pg + 1);
  }
  if constexpr (kSwiglu) {
    const uint4* pu = reinterpret_cast<const uint4*>(row + cols + c0);
    if constexpr (kStream) {
      s.u[0] = __ldcs(pu);
      s.u[1] = __ldcs(pu + 1);
    } else {
      s.u[0] = __ldg(pu);
      s.u[1] = __ldg(pu + 1);
    }
  }
}

__device__ __forceinline__ uint32_t word(const Slice& s, int i, bool up) {
  const uint4& v = up ? s.u[i >> 2] : s.g[i >> 2];
  return (i & 3) == 0 ? v.x : (i & 3) == 1 ? v.y : (i & 3) == 2 ? v.z : v.w;
}

// max |h| of a slice as a binary32 bit pattern.  With SwiGLU the exact
// products are compared and the largest is rounded to BF16 once: rounding is
// monotone, so max |RNE(p)| = RNE(max |p|).  Integer max keeps NaN (its bit
// patterns sort above +inf).
template <bool kSwiglu>
__device__ __forceinline__ uint32_t slice_absmax_bits(const Slice& s, const float* tab) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t gw = word(s, i, false);
    if constexpr (kSwiglu) {
      const uint32_t uw = word(s, i, true);
      m = max(m, __float_as_uint(swiglu_product(gw & 0xFFFFu, uw & 0xFFFFu, tab)) & 0x7FFFFFFFu);
      m = max(m, __float_as_uint(swiglu_product(gw >> 16, uw >> 16, tab)) & 0x7FFFFFFFu);
    } else {
      m = max(m, (gw << 16) & 0x7FFFFFFFu);
      m = max(m, gw & 0x7FFF0000u);
    }
  }
  return m;
}

__device__ __forceinline__ uint32_t round_max_to_bf16(uint32_t m) {
  if (m >= 0x7F800000u) return m;  // Inf / NaN stay as they are
  return bf16x2_rn(__uint_as_float(m), 0.0f) << 16;
}

// Walks the units (row, segment) of a [rows, cols] grid, grid-strided over
// warps, without a division in the loop.
struct UnitWalker {
  int64_t row, seg;
  int64_t step_rows, step_segs, segs;
  __device__ UnitWalker(int64_t first, int64_t stride, int64_t segs_) : segs(segs_) {
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
// Two units in flight per warp.  Loads keep the default L2 policy so the
// tail of the tensor is still in L2 when pass 2 (which walks backwards)
// starts.
template <bool kSwiglu>
__global__ void __launch_bounds__(kThreads) k_amax(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ld, nvfp4_scale_rec* rec) {
  __shared__ float tab[kSwiglu ? kSiluEntries : 1];
  __shared__ uint32_t wmax[kWarps];
  load_table<kSwiglu>(tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t segs = (cols + kSegElems - 1) / kSegElems;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  uint32_t amax = 0;
  UnitWalker w(first, stride, segs);
  while (w.row < rows) {
    const int64_t r0 = w.row, c0 = w.seg * kSegElems + lane * 16;
    w.next();
    const int64_t r1 = w.row, c1 = w.seg * kSegElems + lane * 16;
    w.next();
    Slice s0, s1;
    const bool v0 = c0 < cols, v1 = r1 < rows && c1 < cols;
    if (v0) load_slice<kSwiglu, false>(x + r0 * ld, cols, c0, s0);
    if (v1) load_slice<kSwiglu, false>(x + r1 * ld, cols, c1, s1);
    if (v0) amax = max(amax, slice_absmax_bits<kSwiglu>(s0, tab));
    if (v1) amax = max(amax, slice_absmax_bits<kSwiglu>(s1, tab));
  }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) m = max(m, wmax[i]);
    if constexpr (kSwiglu) m = round_max_to_bf16(m);
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

// Block scale code of a block with max |h| = bmax: E4M3(RN(bmax / d)).
__device__ __forceinline__ uint32_t block_scale_code(float bmax, float d, float rd) {
  if (d == 0.0f) return 0u;
  float r = __fmul_rn(bmax, rd);
  if (near_boundary<5>(r)) r = __fdiv_rn(bmax, d);
  return e4m3_code(r);
}

// Pass 2: quantise.  Units cover rows [0, rows_pad), walked from the end so
// that the first reads hit what pass 1 left in L2; rows >= rows are zeros.
template <bool kSwiglu>
__global__ void __launch_bounds__(kThreads) k_quant(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                    int64_t ld, int64_t rows_pad, uint8_t* __restrict__ qdata,
                                                    uint8_t* __restrict__ scales, nvfp4_scale_rec* rec) {
  __shared__ float tab[kSwiglu ? kSiluEntries : 1];
  load_table<kSwiglu>(tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const uint32_t amax_bits = *reinterpret_cast<volatile uint32_t*>(&rec->amax_bits);
  const bool finite = amax_bits < 0x7F800000u;
  const float g = finite ? __fdiv_rn(__uint_as_float(amax_bits), 2688.0f) : __uint_as_float(0x7FC00000u);
  const float d = __fmul_rn(6.0f, g);
  const float rd = (d == 0.0f || !finite) ? 0.0f : __frcp_rn(d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    rec->global_scale = g;
    rec->status = finite ? NVFP4_OK : NVFP4_ENONFINITE;
  }

  const int64_t segs = (cols + kSegElems - 1) / kSegElems;
  const int64_t cpad4 = (cols / 16 + 3) / 4;  // 4-column scale groups per row
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  for (UnitWalker w(first, stride, segs); w.row < rows_pad; w.next()) {
    const int64_t r = rows_pad - 1 - w.row;
    const int64_t seg = segs - 1 - w.seg;
    const int64_t c0 = seg * kSegElems + lane * 16;
    const bool valid = c0 < cols;
    uint32_t hw[8];  // 16 BF16 values of h, two per word
    if (valid && finite && r < rows) {
      Slice s;
      load_slice<kSwiglu, true>(x + r * ld, cols, c0, s);
#pragma unroll
      for (int i = 0; i < 8; ++i) hw[i] = kSwiglu ? swiglu_pair(word(s, i, false), word(s, i, true), tab)
                                                  : word(s, i, false);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) hw[i] = 0u;
    }
    uint32_t mbits = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mbits = max(mbits, max((hw[i] << 16) & 0x7FFFFFFFu, hw[i] & 0x7FFF0000u));
    const uint32_t bs = finite ? block_scale_code(__uint_as_float(mbits), d, rd) : 0u;
    const float sc = __fmul_rn(e4m3_value(bs), g);
    uint2 packed = make_uint2(0u, 0u);
    if (sc != 0.0f && finite) {
      const float rs = __frcp_rn(sc);
      float q[16];
      bool near = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q[2 * i] = __fmul_rn(bf16_to_f32(hw[i] & 0xFFFFu), rs);
        q[2 * i + 1] = __fmul_rn(__uint_as_float(hw[i] & 0xFFFF0000u), rs);
        near |= near_boundary<3>(q[2 * i]) | near_boundary<3>(q[2 * i + 1]);
      }
      if (near) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          q[2 * i] = __fdiv_rn(bf16_to_f32(hw[i] & 0xFFFFu), sc);
          q[2 * i + 1] = __fdiv_rn(__uint_as_float(hw[i] & 0xFFFF0000u), sc);
        }
      }
      uint32_t b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) b[i] = e2m1x2_code(q[2 * i], q[2 * i + 1]);
      packed.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
      packed.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    }
    if (valid) *reinterpret_cast<uint2*>(qdata + r * (cols / 2) + c0 / 2) = packed;

    // scales: lanes 4j..4j+3 hold the four blocks of scale group j
    const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, bs, 1);
    const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, bs, 2);
    const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, bs, 3);
    const int64_t grp = seg * (kSegElems / 64) + (lane >> 2);
    if ((lane & 3) == 0 && grp < cpad4) {
      const int64_t off = ((r >> 7) * cpad4 + grp) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
      *reinterpret_cast<uint32_t*>(scales + off) = bs | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
  }
}

template <typename K>
int grid_for(K kernel) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return sm_count() * per_sm;
}

nvfp4_status quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, bool swiglu, void* qdata,
                      void* scales, nvfp4_scale_rec* rec, cudaStream_t stream, const char* name) {
  if (!x || !qdata || !scales || !rec) return fail(NVFP4_EINVAL, std::string(name) + ": null pointer");
  if (rows < 1 || cols < 16) return fail(NVFP4_EINVAL, std::string(name) + ": rows must be >= 1 and cols >= 16");
  if (cols % 16 != 0) return fail(NVFP4_EUNSUPPORTED, std::string(name) + ": cols must be a multiple of 16");
  const int64_t need = swiglu ? 2 * cols : cols;
  if (ld < need) return fail(NVFP4_EINVAL, std::string(name) + ": ld too small");
  if (ld % 8 != 0 || !aligned16(x) || !aligned16(qdata) || !aligned16(scales) || !aligned16(rec))
    return fail(NVFP4_EALIGN, std::string(name) + ": pointers must be 16-byte aligned and ld a multiple of 8");
  if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 30))
    return fail(NVFP4_EUNSUPPORTED, std::string(name) + ": tensor too large");
  const int64_t rows_pad = nvfp4_padded_rows(rows);
  const uint16_t* xin = static_cast<const uint16_t*>(x);
  uint8_t* q = static_cast<uint8_t*>(qdata);
  uint8_t* s = static_cast<uint8_t*>(scales);

  nvfp4_status st = cuda_check(cudaMemsetAsync(rec, 0, sizeof(nvfp4_scale_rec), stream), "memset rec");
  if (st != NVFP4_OK) return st;
  if (swiglu) {
    k_amax<true><<<grid_for(k_amax<true>), kThreads, 0, stream>>>(xin, rows, cols, ld, rec);
    st = cuda_check(cudaGetLastError(), "launch k_amax");
    if (st != NVFP4_OK) return st;
    k_quant<true><<<grid_for(k_quant<true>), kThreads, 0, stream>>>(xin, rows, cols, ld, rows_pad, q, s, rec);
  } else {
    k_amax<false><<<grid_for(k_amax<false>), kThreads, 0, stream>>>(xin, rows, cols, ld, rec);
    st = cuda_check(cudaGetLastError(), "launch k_amax");
    if (st != NVFP4_OK) return st;
    k_quant<false><<<grid_for(k_quant<false>), kThreads, 0, stream>>>(xin, rows, cols, ld, rows_pad, q, s, rec);
  }
  return cuda_check(cudaGetLastError(), "launch k_quant");
}

// ---- diagnostics: the same device functions on test-chosen inputs ----------

__global__ void k_diag_silu_all(uint16_t* out) {
  __shared__ float tab[kSiluEntries];
  load_table<true>(tab);
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < 65536u; g += gridDim.x * blockDim.x)
    out[g] = static_cast<uint16_t>(__float_as_uint(silu_bf16(g, tab)) >> 16);
}

// SwiGLU through the producer's pass-2 path (swiglu_pair) and, for the
// pass-1 path, the BF16 rounding of the exact product.
__global__ void k_diag_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t n) {
  __shared__ float tab[kSiluEntries];
  load_table<true>(tab);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t pair = swiglu_pair(gate[i] | (uint32_t(gate[i]) << 16), up[i] | (uint32_t(up[i]) << 16), tab);
    const uint32_t p1 = round_max_to_bf16(__float_as_uint(swiglu_product(gate[i], up[i], tab)) & 0x7FFFFFFFu) >> 16;
    const uint32_t lo = pair & 0xFFFFu, hi = pair >> 16;
    // both halves of the pair and |pass-1 value| must agree; a disagreement
    // is reported as the NaN pattern 0x7FFF, which never equals the oracle
    const bool ok = lo == hi && ((lo & 0x7FFFu) == p1 || ((lo & 0x7FFFu) > 0x7F80u && p1 > 0x7F80u));
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

extern "C" nvfp4_status nvfp4_diag_silu_all(uint16_t* out, nvfp4_stream_t stream) {
  if (!out || !aligned16(out)) return fail(NVFP4_EINVAL, "nvfp4_diag_silu_all: bad pointer");
  k_diag_silu_all<<<64, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out);
  return cuda_check(cudaGetLastError(), "launch k_diag_silu_all");
}

extern "C" nvfp4_status nvfp4_diag_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t n,
                                          nvfp4_stream_t stream) {
  if (!gate || !up || !h || n < 1) return fail(NVFP4_EINVAL, "nvfp4_diag_swiglu: bad arguments");
  k_diag_swiglu<<<256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(gate, up, h, n);
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
