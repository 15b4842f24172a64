/*
 * nvfp4_fc2_diag.h -- diagnostic entry points of libnvfp4fc2.so.
 *
 * They run the exact device functions the production kernels use (the BF16
 * silu, the E2M1 and E4M3 encoders, the bounded pipeline wait) on inputs the
 * tests choose, so that each can be checked exhaustively against the CPU
 * oracle.  They are not on the FC2 path.  Same conventions as nvfp4_fc2.h:
 * device pointers, caller-owned memory, asynchronous on `stream`, synchronous
 * argument errors.
 */
#ifndef NVFP4_FC2_DIAG_H
#define NVFP4_FC2_DIAG_H

#include <stdint.h>
#include "nvfp4_fc2.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[g] = BF16 bits of the producer's silu for every BF16 gate g
 * (65536 entries, device).  The SwiGLU step of the activation producer:
 * "GB10 component-2 nsys summary", other_boundaries (separate BF16 silu). */
nvfp4_status nvfp4_diag_silu_all(uint16_t* out, nvfp4_stream_t stream);

/* out[g] = BF16 bits of the silu the SwiGLU epilogue of nvfp4_fc1_swiglu
 * takes (a shared-memory slice of the producer's table for 2^-10 <= |g| <
 * 8, g itself for g >= 8, the table in global memory otherwise) for every
 * BF16 gate g (65536 entries, device); must equal nvfp4_diag_silu_all. */
nvfp4_status nvfp4_diag_silu_epilogue(uint16_t* out, nvfp4_stream_t stream);

/* h[i] = the producer's SwiGLU output for (gate[i], up[i]), BF16 bits,
 * n elements (device arrays). */
nvfp4_status nvfp4_diag_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t n,
                               nvfp4_stream_t stream);

/* Scan every binary32 bit pattern p in [0, 2^32) through the device encoder
 * (which = 0: E2M1 element code, which = 1: E4M3 block-scale code) and list
 * the patterns where the code differs from that of p - 1, skipping pairs
 * where either pattern is Inf or NaN.  Entry i of `trans` is
 * {p, code(p), code(p-1)}; code of pattern 0 goes to first_code.  At most
 * `cap` entries are stored; *count (device) receives the number found.
 * All of trans, count, first_code are device memory; *count must be zero on
 * entry. */
nvfp4_status nvfp4_diag_code_transitions(int which, uint32_t* trans, uint32_t cap,
                                         uint32_t* count, uint32_t* first_code,
                                         nvfp4_stream_t stream);

/* Run the bounded wait used by the GEMM pipeline on an mbarrier that nothing
 * arrives at, with the given limit in nanoseconds (1 .. 10^9).  Writes
 * NVFP4_ETIMEOUT to *dev_status when the wait runs out (device uint32).
 * Exercises the timeout path without faulting or hanging the GPU. */
nvfp4_status nvfp4_diag_wait_timeout(uint64_t limit_ns, uint32_t* dev_status,
                                     nvfp4_stream_t stream);

/* The element encoder of pass 2 (h -> E2M1 code of h / sc), swept against
 * its definition ("FC2 NVFP4 Scheduling Results", Canonical Operation: E2M1
 * elements of h divided by the decoded block scale): for every global max
 * A among the BF16 patterns a_first .. a_first + a_count - 1 (g =
 * RN(A / 2688)), every block-scale code 1..126 with sc = RN(E4M3 * g) > 0,
 * and every BF16 h of either sign with |h| <= A (the values of a block never
 * exceed the global max), the producer's code is compared
 * with E2M1(RN(h / sc)), RN(h / sc) the correctly rounded division.
 * counts (device, two uint64, zeroed by the caller) receives += {codes that
 * differ, codes compared}.  a_first + a_count <= 0x7F80 (finite maxima),
 * a_count >= 1, else NVFP4_EINVAL.  All 32,639 nonzero maxima take a few
 * seconds in total. */
nvfp4_status nvfp4_diag_quotient_codes(uint32_t a_first, uint32_t a_count, uint64_t* counts,
                                       nvfp4_stream_t stream);

/* The block-scale encoder of pass 2 swept against its definition ("GB10
 * component-2 nsys summary", nvfp4: scale finalize, then block scales from
 * block absmax; the two-level NVFP4 recipe bs = E4M3(block_amax / (6 g))):
 * for every global max A among the BF16 patterns a_first .. a_first +
 * a_count - 1 (g = RN(A / 2688), d = RN(6 g)) and every finite non-negative
 * BF16 block max b, the producer's code is compared with E4M3(RN(b / d)),
 * RN(b / d) the correctly rounded division (0 when d == 0).  counts
 * (device, two uint64, zeroed by the caller) receives += {codes that
 * differ, codes compared}.  a_first + a_count <= 0x7F80, a_count >= 1, else
 * NVFP4_EINVAL.  All 32,640 maxima (about 10^9 pairs) take well under a
 * second. */
nvfp4_status nvfp4_diag_block_scale_codes(uint32_t a_first, uint32_t a_count, uint64_t* counts,
                                          nvfp4_stream_t stream);

/* The tensor core's reading of packed E2M1 bytes ("FC2 NVFP4 Scheduling
 * Results", Canonical Operation: packed E2M1 operands).  qdata holds 128
 * rows of 16 bytes (32 E2M1 elements each, row-major, device, 16-B
 * aligned); one tcgen05.mma.kind::f8f6f4 multiplies them by the 32 x 32
 * identity in E4M3 (one byte per element), so out[r * 32 + n] (device
 * float, 128 x 32) is the value the tensor core gives element n of row r.
 * An E2M1 x E2M1 GEMM cannot show which nibble holds which element (the
 * same swap in both operands leaves every dot product unchanged); this
 * can.  NVFP4_ETIMEOUT goes to *dev_status (device uint32, may be NULL) if
 * the MMA's completion is not seen within about a second. */
nvfp4_status nvfp4_diag_tc_e2m1_read(const uint8_t* qdata, float* out, uint32_t* dev_status,
                                     nvfp4_stream_t stream);

/* Dense NVFP4 tensor-core throughput of this GPU, the denominator of the
 * GEMM's roofline ("FC2 NVFP4 Scheduling Results", Canonical Operation: the
 * FC2 is a dense E2M1 x E2M1 contraction with UE4M3 vector-16 scales).
 * P SM pairs (nvfp4_diag_mma_peak_pairs()) each run `iters` back-to-back
 * tcgen05.mma.cta_group::2.kind::mxf4nvf4 (M=256, N=256, K=64, i.e.
 * 2*256*256*64 = 8388608 FLOP each) on operands resident in shared memory
 * (fixed pseudo-random bytes, all scales 1.0) with nothing else on the
 * tensor pipe.  The caller times the launch on `stream`: FLOP per launch =
 * P * iters * 8388608.  1 <= iters <= 2^22, else NVFP4_EINVAL.  If the
 * final bounded wait runs out, NVFP4_ETIMEOUT is written to *dev_status
 * (device uint32; may be NULL); the accumulators are discarded.
 * clk (device, 8-byte aligned, may be NULL) receives the first pair's
 * clock record: {globaltimer ns when its first MMA is issued, ns when its
 * last has completed, the SM's clock64 at those two points}.  Cycles per
 * MMA = (clk[3] - clk[2]) / iters; the SM clock in MHz =
 * 1000 * (clk[3] - clk[2]) / (clk[1] - clk[0]). */
nvfp4_status nvfp4_diag_mma_peak(int64_t iters, uint32_t* dev_status, uint64_t* clk, nvfp4_stream_t stream);

/* nvfp4_fc2_gemm with a clock record: the same kernel and arguments, and
 * block 0 (the first CTA pair's leader) writes {globaltimer ns after its
 * prologue, ns at the end of its teardown barrier, its SM's clock64 at both
 * points} to clk (device, four uint64, 8-byte aligned, else NVFP4_EINVAL).
 * The kernel's time in SM cycles and the clock it ran at follow as for
 * nvfp4_diag_mma_peak.  The pages measure their FC2 kernel in wall time
 * only ("FC2 NVFP4 Scheduling Results", Timing); this record separates the
 * kernel's cycle count from the SM clock the part chose under its load. */
nvfp4_status nvfp4_diag_fc2_gemm_clock(const void* a_q, const void* a_s, const nvfp4_scale_rec* a_rec,
                                       const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec, int64_t m,
                                       int64_t n, int64_t k, void* out_bf16, int64_t ldo, uint32_t* dev_status,
                                       uint64_t* clk, nvfp4_stream_t stream);

/* P above: the SM pairs that hold one two-CTA cluster of the loop each at
 * the same time on the current device (SMs / 2 unless fewer fit); -1 if
 * the CUDA query fails. */
int64_t nvfp4_diag_mma_peak_pairs(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_FC2_DIAG_H */
