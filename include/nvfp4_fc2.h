/*
 * nvfp4_fc2.h -- C ABI of libnvfp4fc2.so: the FC2 step of a video diffusion
 * transformer's MLP on one GB300 (sm_103a).
 *
 *   gate|up (BF16) --swiglu_nvfp4_quantize--> NVFP4 activation
 *   W (BF16)       --nvfp4_quantize_weight--> NVFP4 weight      (once)
 *   NVFP4 x NVFP4  --nvfp4_fc2_gemm---------> BF16 output
 *
 * Sources (page title, section):
 *   "FC2 NVFP4 Scheduling Results", Canonical Operation -- logical GEMM
 *     M=37,810 N=5,376 K=14,336; packed NVFP4 E2M1 activation and weight with
 *     vector-16 UE4M3 scales; FP32 accumulation and scalars; BF16 output;
 *     producer pads M; the accepted producer fuses SwiGLU into quantisation.
 *   "FC2 NVFP4 Scheduling Results", Decision and Traffic Attribution -- a
 *     split-K-1 schedule with zero workspace, no global atomics or reduction
 *     traffic, one BF16 output write.
 *   "GB10 component-2 nsys summary", nvfp4 -- absmax partials, scale
 *     finalize, block-scale zeroing and activation packing: the global scale
 *     must be known before any element is quantised (two passes).
 *   "GB10 component-2 nsys summary", native_pack_validation -- block scales
 *     in the general 128-row by 4-scale-column tiled layout, exact at feature
 *     widths 5376, 7168 and 14336.
 *
 * NVFP4 recipe (global/block/element):
 *   amax   = max |h| over the whole tensor
 *   g      = RN_f32(amax / 2688)                       (2688 = 6 * 448)
 *   bs     = RNE_E4M3_satfinite(RN_f32(block_amax / RN_f32(6 g)))  per 16 elements
 *   s      = RN_f32(E4M3(bs) * g)
 *   code   = RNE_E2M1_satfinite(RN_f32(h / s))  (0x0 when s == 0; sign kept)
 *   QDATA byte j of a row = code(2j) | code(2j+1) << 4
 *
 * Layouts (all row-major, bytes):
 *   rows_pad        = ceil(rows / 128) * 128; rows >= rows are zero bytes.
 *   QDATA           [rows_pad, cols/2] uint8.
 *   scale columns   C = cols/16, padded to C4 = ceil(C/4)*4 (pad bytes zero).
 *   scale (r, c)    at ((r/128)*(C4/4) + c/4)*512 + (r%32)*16 + ((r/32)%4)*4 + c%4.
 *   nvfp4_scale_rec 16 bytes in device memory (below).
 *
 * Ownership and threading: the caller allocates every buffer (device memory
 * unless stated) and keeps it alive until the stream work completes.  The
 * library allocates nothing, keeps no state between calls, is safe to call
 * from several host threads, and enqueues all work asynchronously on the
 * given stream (NULL = legacy default stream).
 *
 * Errors: a non-zero nvfp4_status returned by a call means nothing was
 * enqueued (argument errors) or a CUDA launch failed (NVFP4_ECUDA; the CUDA
 * error is cleared from the runtime's sticky-free state and described by
 * nvfp4_last_error()).  Errors found on the device (non-finite input, a
 * bounded wait that ran out) are written to device status words and read by
 * the caller after synchronising the stream.
 */
#ifndef NVFP4_FC2_H
#define NVFP4_FC2_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* same object as cudaStream_t */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_EINVAL = 1,       /* null pointer, non-positive size, ld too small */
  NVFP4_EUNSUPPORTED = 2, /* shape outside what the kernels handle */
  NVFP4_EALIGN = 3,       /* pointer not 16-byte aligned or ld not a multiple of 8 */
  NVFP4_ENONFINITE = 4,   /* device: the quantised tensor holds Inf or NaN */
  NVFP4_ETIMEOUT = 5,     /* device: a bounded pipeline wait ran out */
  NVFP4_ECUDA = 6         /* a CUDA runtime call or launch failed */
} nvfp4_status;

/* Global-scale record of one NVFP4 tensor, written on the device by the
 * quantisers and read on the device by the GEMM (never copied to the host
 * by the library).  16 bytes, 16-byte aligned.
 *   global_scale  g above; NaN when status == NVFP4_ENONFINITE
 *   amax_bits     bit pattern of max |h| (binary32; >= 0x7F800000 if non-finite)
 *   status        NVFP4_OK or NVFP4_ENONFINITE */
typedef struct {
  float global_scale;
  uint32_t amax_bits;
  uint32_t status;
  uint32_t reserved;
} nvfp4_scale_rec;

/* ceil(rows / 128) * 128 (rows >= 0). */
int64_t nvfp4_padded_rows(int64_t rows);
/* Bytes of QDATA for a [rows, cols] tensor: padded_rows * cols / 2. */
int64_t nvfp4_qdata_bytes(int64_t rows, int64_t cols);
/* Bytes of the tiled block-scale array: padded_rows * ceil(cols/16/4)*4. */
int64_t nvfp4_scale_bytes(int64_t rows, int64_t cols);
/* Byte offset of scale (r, c) (c = column/16) in the tiled layout. */
int64_t nvfp4_scale_offset(int64_t r, int64_t c, int64_t cols);

/* Weight quantiser: two-pass NVFP4 of a BF16 [rows, cols] matrix.
 *   w_bf16  device, row stride ld elements (ld >= cols, ld % 8 == 0), 16-B aligned
 *   rows    >= 1;  cols >= 16, cols % 16 == 0
 *   qdata   device, nvfp4_qdata_bytes(rows, cols) bytes, 16-B aligned (written
 *           in full, pad rows zero)
 *   scales  device, nvfp4_scale_bytes(rows, cols) bytes, 16-B aligned
 *           (written in full, pad rows and pad columns zero)
 *   rec     device, 16-B aligned; written
 * Enqueues a memset of rec and two kernels (absmax pass, quantise pass). */
nvfp4_status nvfp4_quantize_weight(const void* w_bf16, int64_t rows, int64_t cols, int64_t ld,
                                   void* qdata, void* scales, nvfp4_scale_rec* rec,
                                   nvfp4_stream_t stream);

/* SwiGLU activation producer: h = bf16(bf16(silu(gate)) * up) with
 * gate = columns [0, k) and up = columns [k, 2k) of a BF16 [m, 2k] matrix,
 * silu rounded once (correctly) to BF16, then two-pass NVFP4 of h [m, k].
 *   gate_up  device, row stride ld elements (ld >= 2k, ld % 8 == 0), 16-B aligned
 *   m >= 1;  k >= 16, k % 16 == 0
 *   qdata, scales, rec as for nvfp4_quantize_weight with rows = m, cols = k.
 * h is never stored: both passes recompute it from gate|up. */
nvfp4_status swiglu_nvfp4_quantize(const void* gate_up_bf16, int64_t m, int64_t k, int64_t ld,
                                   void* qdata, void* scales, nvfp4_scale_rec* rec,
                                   nvfp4_stream_t stream);

/* Block-scaled NVFP4 GEMM (persistent tcgen05 kernel, FP32 accumulation in
 * tensor memory, BF16 output):
 *   out[i, j] = bf16_rn( RN_f32(a_rec.g * w_rec.g) * sum_k A[i,k] W[j,k] )
 * where A[i,k] = E2M1(a) * UE4M3(a scale) and likewise W, i < m, j < n.
 *   a_q, a_s, a_rec   activation QDATA [pad(m), k/2], scales, record (device)
 *   w_q, w_s, w_rec   weight QDATA [n, k/2], scales, record (device)
 *   m >= 1; n >= 128, n % 128 == 0; k >= 256, k % 256 == 0
 *   out_bf16          device [m, ldo] BF16, 16-byte aligned, ldo >= n,
 *                     ldo % 8 == 0 (else NVFP4_EALIGN); written by TMA stores
 *                     through a tensor map of [m, n], so rows >= m and
 *                     columns >= n are not touched
 *   dev_status        device uint32 or NULL; set to NVFP4_ETIMEOUT if a
 *                     bounded wait ran out (never cleared by the library)
 * No workspace, no atomics; K is reduced in increasing order inside one CTA,
 * so row i of the output does not depend on m. */
nvfp4_status nvfp4_fc2_gemm(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                            const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec,
                            int64_t m, int64_t n, int64_t k, void* out_bf16, int64_t ldo,
                            uint32_t* dev_status, nvfp4_stream_t stream);

/* FC1 with the SwiGLU producer's first pass in its epilogue (the fusion the
 * pages leave open, "FC2 NVFP4 Scheduling Results", Canonical Operation:
 * SwiGLU into the NVFP4 quantisation).  The same GEMM as nvfp4_fc2_gemm with
 * W = [gate; up], 2f rows: each output tile pairs gate rows j and up rows
 * f + j, and the epilogue writes, for i < m and j < f,
 *   g = bf16_rn(RN_f32(a_rec.g * w_rec.g) * sum_k A[i,k] W[j,k])
 *   u = bf16_rn(... W[f + j, k] ...)          (the BF16 FC1 outputs)
 *   h[i, j] = bf16(bf16(silu(g)) * u)         (silu correctly rounded)
 * which is byte for byte what nvfp4_fc2_gemm followed by the SwiGLU of
 * swiglu_nvfp4_quantize computes.  It also writes h_rec->amax_bits = the bit
 * pattern of max |h| (the producer's first pass), after zeroing h_rec.
 *   a_q, a_s, a_rec, w_q, w_s, w_rec, m, k   as for nvfp4_fc2_gemm; W has 2f rows
 *   f >= 128, f % 128 == 0
 *   h_bf16   device [m, ldh] BF16, ldh >= f, ldh % 8 == 0; other bytes untouched
 *   h_rec    device record, 16-B aligned: zeroed, then amax_bits set
 *   dev_status as for nvfp4_fc2_gemm
 * Follow with nvfp4_quantize_with_amax(h, m, f, ldh, ..., h_rec) for the
 * NVFP4 activation of FC2: the two calls give the bytes of
 * swiglu_nvfp4_quantize on FC1's BF16 gate|up output, without writing or
 * re-reading that 2f-wide output. */
nvfp4_status nvfp4_fc1_swiglu(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                              const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec,
                              int64_t m, int64_t f, int64_t k, void* h_bf16, int64_t ldh,
                              nvfp4_scale_rec* h_rec, uint32_t* dev_status, nvfp4_stream_t stream);

/* The quantise pass of nvfp4_quantize_weight alone, for a BF16 [rows, cols]
 * matrix whose global max is already in rec->amax_bits (as
 * nvfp4_fc1_swiglu leaves it); rec->global_scale and rec->status are
 * written.  Arguments as for nvfp4_quantize_weight; rec is not zeroed. */
nvfp4_status nvfp4_quantize_with_amax(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                                      void* qdata, void* scales, nvfp4_scale_rec* rec,
                                      nvfp4_stream_t stream);

/* One FC2 step from host memory to host memory ("FC2 NVFP4 Scheduling
 * Results", Production Integration: forward_swiglu = the accepted producer,
 * then the FC2 GEMM): the host gate|up is copied into the caller's device
 * buffer, swiglu_nvfp4_quantize and nvfp4_fc2_gemm run on it, and the BF16
 * output is copied back to host memory.  Everything is enqueued on
 * `stream`; the host output is valid once the stream has reached this
 * point (the call itself does not synchronise).  Pinned host memory makes
 * both copies asynchronous; with pageable memory the runtime copies
 * synchronously.
 *   gate_up_host  host BF16 [m, ld_host], ld_host >= 2k
 *   m >= 1; k, n as for swiglu_nvfp4_quantize and nvfp4_fc2_gemm
 *   w_q, w_s, w_rec   the NVFP4 weight [n, k] (device)
 *   x_dev         device BF16 [m, 2k], contiguous: receives the input
 *   a_q, a_s, a_rec   device NVFP4 activation buffers of [m, k] (sizes as
 *                 for swiglu_nvfp4_quantize); written
 *   out_dev       device BF16 [m, n], contiguous: the GEMM output
 *   out_host      host BF16 [m, n], contiguous: receives the output
 *   dev_status    as for nvfp4_fc2_gemm
 * All device buffers belong to the caller; the library allocates no device
 * memory.  The host-to-device copies of all calls on a device run one at a
 * time in call order: before its copy, `stream` waits for an event that the
 * library records after the previous call's copy (one CUDA event per device,
 * created by the first call; the current device must be the stream's).  One
 * copy at a time keeps the host link, which bounds this step, moving at the
 * rate of a single copy; callers that pipeline steps on several streams
 * still overlap one step's copy with another's kernels and output copy.
 * While `stream` is being captured into a graph the wait is left out.
 * Every argument is checked before anything is enqueued (the shapes that
 * nvfp4_fc2_gemm accepts: k % 256 == 0, n % 128 == 0). */
nvfp4_status nvfp4_fc2_host(const void* gate_up_host, int64_t m, int64_t k, int64_t ld_host, const void* w_q,
                            const void* w_s, const nvfp4_scale_rec* w_rec, int64_t n, void* x_dev, void* a_q,
                            void* a_s, nvfp4_scale_rec* a_rec, void* out_dev, void* out_host,
                            uint32_t* dev_status, nvfp4_stream_t stream);

/* nvfp4_fc2_host for callers that cannot allocate device memory.  The pages
 * have no counterpart: it exists for callers such as a plug-in whose host
 * program owns the GPU's memory and forbids cudaMalloc, or code that must not
 * allocate once running (an allocation can block, synchronise the device or
 * fail under fragmentation).  The step's three device buffers (the copy of
 * gate|up, the NVFP4 activation, the BF16 output) come from one 32 MiB
 * (33,554,432-byte) array inside the library, which every GPU that loads the
 * library holds until the process exits; no cudaMalloc, cudaFree or other
 * call that allocates device memory is made.  The caller still provides the inputs (gate|up in
 * host memory, the NVFP4 weight on the device) and the host output.
 *   Arguments as for nvfp4_fc2_host without the device buffers.
 *   Sizes: 256-byte-rounded m*2k*2 + QDATA + scale bytes + 16 + m*n*2 must
 *   fit in the 32 MiB, else NVFP4_EUNSUPPORTED with the bytes needed in
 *   nvfp4_last_error() (FC2 widths, k = 14336 and n = 5376: up to 432 rows;
 *   the tiny FC2 shape, m = 256, k = 1024, n = 512: 1.4 MiB).  Argument and
 *   size errors are found before any CUDA call.
 *   The first call with a device current looks up the array's address on
 *   that device (cudaGetSymbolAddress, a synchronous runtime call) and keeps
 *   it, and nvfp4_fc2_host's first call creates its copy-order event; make
 *   that first call before any stream capture on the device.
 *   All calls share the one array and find the last call's bytes in it.
 *   Nothing in it needs to start at zero (each call writes every byte it
 *   later reads), but calls whose work overlaps on the GPU (two streams, two
 *   host threads) race on it: order them on one stream or wait in between. */
nvfp4_status nvfp4_fc2_host_noalloc(const void* gate_up_host, int64_t m, int64_t k, int64_t ld_host,
                                    const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec, int64_t n,
                                    void* out_host, uint32_t* dev_status, nvfp4_stream_t stream);

/* Message describing the last non-zero status returned on this host thread. */
const char* nvfp4_last_error(void);

/* Library version, (major << 16) | minor. */
uint32_t nvfp4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_FC2_H */
