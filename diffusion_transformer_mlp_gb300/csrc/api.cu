// Host-side pieces of libnvfp4fc2 shared by every entry point: sizes of the
// NVFP4 buffers, the tiled scale offset, per-thread error messages and the
// per-device SM count.
//
// Sizes follow "FC2 NVFP4 Scheduling Results", Canonical Operation (rows
// padded by the producer; QDATA half a byte per element) and Traffic
// Attribution (activation QDATA + scales 305,012,736 B at 37,824 x 14,336,
// i.e. 9/16 byte per element); the scale offset is the general 128-row by
// 4-scale-column tiled layout of "GB10 component-2 nsys summary",
// native_pack_validation.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"

namespace nvfp4 {

namespace {
thread_local std::string g_last_error;
}

nvfp4_status fail(nvfp4_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

nvfp4_status cuda_check(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return NVFP4_OK;
  char buf[256];
  std::snprintf(buf, sizeof(buf), "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
  return fail(NVFP4_ECUDA, buf);
}

int sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

// The host-to-device copies of nvfp4_fc2_host run one at a time across all
// calls on a device, in call order: before its copy, a call's stream waits
// for an event recorded after the previous call's copy (one event per
// device, created on first use).  The host link is the bound of that step
// (2.17 GB in against 0.41 GB out at ~210 GB/s a direction); two copies in
// flight at once, from two callers' streams on two copy engines, only share
// it, and on some machines they moved fewer bytes together than one alone.
// The wait is skipped while `stream` is being captured into a graph.
struct CopyOrder {
  std::mutex mu;
  cudaEvent_t ev[64] = {};
  bool recorded[64] = {};
};

CopyOrder& copy_order() {
  static CopyOrder c;
  return c;
}

}  // namespace nvfp4

extern "C" int64_t nvfp4_padded_rows(int64_t rows) { return rows <= 0 ? 0 : (rows + 127) / 128 * 128; }

extern "C" int64_t nvfp4_qdata_bytes(int64_t rows, int64_t cols) {
  return (rows <= 0 || cols <= 0) ? 0 : nvfp4_padded_rows(rows) * (cols / 2);
}

extern "C" int64_t nvfp4_scale_bytes(int64_t rows, int64_t cols) {
  return (rows <= 0 || cols <= 0) ? 0 : nvfp4_padded_rows(rows) * ((cols / 16 + 3) / 4 * 4);
}

extern "C" int64_t nvfp4_scale_offset(int64_t r, int64_t c, int64_t cols) {
  const int64_t groups = (cols / 16 + 3) / 4;
  return ((r / 128) * groups + c / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

extern "C" const char* nvfp4_last_error(void) { return nvfp4::g_last_error.c_str(); }

extern "C" uint32_t nvfp4_version(void) { return (1u << 16) | 0u; }

extern "C" nvfp4_status nvfp4_fc2_host(const void* gate_up_host, int64_t m, int64_t k, int64_t ld_host,
                                       const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec, int64_t n,
                                       void* x_dev, void* a_q, void* a_s, nvfp4_scale_rec* a_rec, void* out_dev,
                                       void* out_host, uint32_t* dev_status, nvfp4_stream_t stream) {
  using nvfp4::cuda_check;
  using nvfp4::fail;
  using nvfp4::aligned16;
  // Every argument is checked before the first copy is enqueued, so that an
  // error status still means that nothing was queued.
  if (!gate_up_host || !w_q || !w_s || !w_rec || !x_dev || !a_q || !a_s || !a_rec || !out_dev || !out_host)
    return fail(NVFP4_EINVAL, "nvfp4_fc2_host: null pointer");
  if (m < 1 || k < 1 || n < 1) return fail(NVFP4_EINVAL, "nvfp4_fc2_host: m, k and n must be positive");
  if (ld_host < 2 * k) return fail(NVFP4_EINVAL, "nvfp4_fc2_host: ld_host must be >= 2k");
  if (k % 256 != 0 || n % 128 != 0 || nvfp4_padded_rows(m) > (int64_t(1) << 30) || n > (int64_t(1) << 24) ||
      k > (int64_t(1) << 24))
    return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_host: k must be a multiple of 256 and n of 128 (or too large)");
  if (!aligned16(x_dev) || !aligned16(a_q) || !aligned16(a_s) || !aligned16(a_rec) || !aligned16(out_dev) ||
      !aligned16(w_q) || !aligned16(w_s) || !aligned16(w_rec))
    return fail(NVFP4_EALIGN, "nvfp4_fc2_host: device pointers must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  nvfp4_status st = cuda_check(cudaStreamIsCapturing(s, &capture), "nvfp4_fc2_host: cudaStreamIsCapturing");
  if (st != NVFP4_OK) return st;
  int dev = 0;
  if ((st = cuda_check(cudaGetDevice(&dev), "nvfp4_fc2_host: cudaGetDevice")) != NVFP4_OK) return st;
  if (dev < 0 || dev >= 64) return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_host: device ordinal above 63");
  nvfp4::CopyOrder& order = nvfp4::copy_order();
  std::unique_lock<std::mutex> lock(order.mu, std::defer_lock);
  const bool ordered = capture == cudaStreamCaptureStatusNone;
  if (ordered) {
    lock.lock();
    if (order.ev[dev] == nullptr &&
        (st = cuda_check(cudaEventCreateWithFlags(&order.ev[dev], cudaEventDisableTiming),
                         "nvfp4_fc2_host: cudaEventCreateWithFlags")) != NVFP4_OK)
      return st;
    if (order.recorded[dev] &&
        (st = cuda_check(cudaStreamWaitEvent(s, order.ev[dev], 0), "nvfp4_fc2_host: cudaStreamWaitEvent")) != NVFP4_OK)
      return st;
  }
  // packed host rows go as one linear copy (a pitched copy of the same bytes
  // moves them row by row, measurably slower over the host link)
  const size_t row_bytes = static_cast<size_t>(2 * k) * 2;
  const cudaError_t ce =
      ld_host == 2 * k
          ? cudaMemcpyAsync(x_dev, gate_up_host, row_bytes * static_cast<size_t>(m), cudaMemcpyHostToDevice, s)
          : cudaMemcpy2DAsync(x_dev, row_bytes, gate_up_host, static_cast<size_t>(ld_host) * 2, row_bytes,
                              static_cast<size_t>(m), cudaMemcpyHostToDevice, s);
  st = cuda_check(ce, "nvfp4_fc2_host: copy of gate|up to the device");
  if (st != NVFP4_OK) return st;
  if (ordered) {
    if ((st = cuda_check(cudaEventRecord(order.ev[dev], s), "nvfp4_fc2_host: cudaEventRecord")) != NVFP4_OK)
      return st;
    order.recorded[dev] = true;
    lock.unlock();
  }
  if ((st = swiglu_nvfp4_quantize(x_dev, m, k, 2 * k, a_q, a_s, a_rec, stream)) != NVFP4_OK) return st;
  if ((st = nvfp4_fc2_gemm(a_q, a_s, a_rec, w_q, w_s, w_rec, m, n, k, out_dev, n, dev_status, stream)) != NVFP4_OK)
    return st;
  return cuda_check(cudaMemcpyAsync(out_host, out_dev, static_cast<size_t>(m) * static_cast<size_t>(n) * 2,
                                    cudaMemcpyDeviceToHost, s),
                    "nvfp4_fc2_host: copy of the output to the host");
}
