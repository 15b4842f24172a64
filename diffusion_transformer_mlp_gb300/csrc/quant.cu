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

// Correctly rounded BF16 silu for gates with exponent field 117..129 (g > 0)
// and 117..133 (g < 0); generated at build time by gen_silu_table.py.
__device__ const uint16_t k_silu_mid[kSiluEntries] = {
#include "silu_mid_table.inc"
};

__device__ __forceinline__ float bf16_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// silu(g) rounded once to BF16 (returned as its binary32 value).
//   |g| < 2^-10 : silu(g) = g/2 + g^2/4 - ..., so the result is g/2, and when
//                 g/2 falls between two BF16 values the exact value lies
//                 above the midpoint: round toward +inf.
//   g >= 8      : the relative gap g - silu(g) < e^-8 < 2^-9: the result is g.
//   g <= -128   : |silu(g)| < 2^-134: the result is -0.
//   +inf -> +inf, -inf and NaN -> NaN (a non-finite gate stays non-finite).
//   otherwise   : table.
__device__ __forceinline__ float silu_bf16(uint32_t g, const uint16_t* tab) {
  const uint32_t e = (g >> 7) & 0xFFu;
  const uint32_t neg = g >> 15;
  uint32_t out;
  if (e < 117u) {
    const uint32_t u = __float_as_uint(bf16_to_f32(g) * 0.5f);  // exact, no flush to zero
    out = (u + (neg ? 0x7FFFu : 0x8000u)) >> 16;
  } else if (e == 0xFFu) {
    out = (g == 0x7F80u) ? 0x7F80u : 0x7FC0u;
  } else if (!neg) {
    out = (e >= 130u) ? g : tab[(e - 117u) * 128u + (g & 0x7Fu)];
  } else {
    out = (e >= 134u) ? 0x8000u : tab[1664u + (e - 117u) * 128u + (g & 0x7Fu)];
  }
  return bf16_to_f32(out);
}

// h = bf16(silu_bf16(g) * u): the binary32 product of two BF16 values is
// exact, so this is a single rounding.
__device__ __forceinline__ float swiglu(uint32_t g, uint32_t u, const uint16_t* tab) {
  const float p = __fmul_rn(silu_bf16(g, tab), bf16_to_f32(u));
  return __bfloat162float(__float2bfloat16_rn(p));
}

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// Eight h values of lane-chunk (row, c0).
template <bool kSwiglu>
__device__ __forceinline__ void load_h(const uint16_t* row, int64_t cols, int64_t c0, const uint16_t* tab,
                                       float h[8]) {
  const uint4 gv = ld_stream(row + c0);
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  if constexpr (kSwiglu) {
    const uint4 uv = ld_stream(row + cols + c0);
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h[2 * i] = swiglu(gw[i] & 0xFFFFu, uw[i] & 0xFFFFu, tab);
      h[2 * i + 1] = swiglu(gw[i] >> 16, uw[i] >> 16, tab);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h[2 * i] = bf16_to_f32(gw[i] & 0xFFFFu);
      h[2 * i + 1] = bf16_to_f32(gw[i] >> 16);
    }
  }
}

template <bool kSwiglu>
__device__ __forceinline__ void load_table(uint16_t* tab) {
  if constexpr (kSwiglu) {
    for (int i = threadIdx.x; i < kSiluEntries; i += blockDim.x) tab[i] = k_silu_mid[i];
    __syncthreads();
  }
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
template <bool kSwiglu>
__global__ void __launch_bounds__(kThreads) k_amax(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ld, nvfp4_scale_rec* rec) {
  __shared__ uint16_t tab[kSwiglu ? kSiluEntries : 1];
  __shared__ uint32_t wmax[kWarps];
  load_table<kSwiglu>(tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t segs = (cols + 255) / 256;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  uint32_t amax = 0;
  for (UnitWalker w(first, stride, segs); w.row < rows; w.next()) {
    const int64_t c0 = w.seg * 256 + lane * 8;
    if (c0 < cols) {
      float h[8];
      load_h<kSwiglu>(x + w.row * ld, cols, c0, tab, h);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(h[i]) & 0x7FFFFFFFu);
    }
  }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) m = max(m, wmax[i]);
    if (m != 0) atomicMax(&rec->amax_bits, m);
  }
}

// Pass 2: quantise.  Units cover rows [0, rows_pad); rows >= rows are zeros.
template <bool kSwiglu>
__global__ void __launch_bounds__(kThreads) k_quant(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                    int64_t ld, int64_t rows_pad, uint8_t* __restrict__ qdata,
                                                    uint8_t* __restrict__ scales, nvfp4_scale_rec* rec) {
  __shared__ uint16_t tab[kSwiglu ? kSiluEntries : 1];
  load_table<kSwiglu>(tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const uint32_t amax_bits = *reinterpret_cast<volatile uint32_t*>(&rec->amax_bits);
  const bool finite = amax_bits < 0x7F800000u;
  const float g = finite ? __fdiv_rn(__uint_as_float(amax_bits), 2688.0f) : __uint_as_float(0x7FC00000u);
  const float d = __fmul_rn(6.0f, g);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    rec->global_scale = g;
    rec->status = finite ? NVFP4_OK : NVFP4_ENONFINITE;
  }

  const int64_t segs = (cols + 255) / 256;
  const int64_t nblk = cols / 16;
  const int64_t cpad4 = (nblk + 3) / 4;  // 4-column groups per row (= tiles per 128-row block)
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
  for (UnitWalker w(first, stride, segs); w.row < rows_pad; w.next()) {
    const int64_t r = w.row;
    const int64_t c0 = w.seg * 256 + lane * 8;
    const bool valid = c0 < cols;
    float h[8];
    if (valid && finite && r < rows) {
      load_h<kSwiglu>(x + r * ld, cols, c0, tab, h);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = 0.0f;
    }
    float lmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) lmax = fmaxf(lmax, fabsf(h[i]));
    const float bmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, 1));
    const float ratio = (d == 0.0f) ? 0.0f : __fdiv_rn(bmax, d);
    const uint32_t bs = finite ? e4m3_code(ratio) : 0u;
    const float s = __fmul_rn(e4m3_value(bs), g);
    uint32_t packed = 0;
    if (s != 0.0f && finite) {
#pragma unroll
      for (int i = 0; i < 8; ++i) packed |= e2m1_code(__fdiv_rn(h[i], s)) << (4 * i);
    }
    if (valid) *reinterpret_cast<uint32_t*>(qdata + r * (cols / 2) + c0 / 2) = packed;

    // scales: lanes 8j, 8j+2, 8j+4, 8j+6 hold blocks 4j..4j+3 of this segment
    const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, bs, 2);
    const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, bs, 4);
    const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, bs, 6);
    const int64_t grp = w.seg * 4 + (lane >> 3);  // 4-column group index
    if ((lane & 7) == 0 && grp < cpad4) {
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
  __shared__ uint16_t tab[kSiluEntries];
  load_table<true>(tab);
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < 65536u; g += gridDim.x * blockDim.x)
    out[g] = static_cast<uint16_t>(__float_as_uint(silu_bf16(g, tab)) >> 16);
}

__global__ void k_diag_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t n) {
  __shared__ uint16_t tab[kSiluEntries];
  load_table<true>(tab);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    h[i] = static_cast<uint16_t>(__float_as_uint(swiglu(gate[i], up[i], tab)) >> 16);
}

__device__ __forceinline__ uint32_t diag_code(int which, uint32_t bits) {
  const float f = __uint_as_float(bits);
  return which == 0 ? e2m1_code(f) : e4m3_code(f);
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
