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
