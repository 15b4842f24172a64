// The host-to-host FC2 step for callers that cannot allocate device memory.
//
// nvfp4_fc2_host needs three device buffers besides its inputs and outputs:
// the device copy of gate|up, the NVFP4 activation and the device BF16
// output.  Some callers have no way to provide them: a plug-in that runs
// inside a host program which owns the GPU's memory and forbids direct
// cudaMalloc calls, or code that must not allocate once it is running (an
// allocation can block, fail under fragmentation, or synchronise the device).
// nvfp4_fc2_host_noalloc serves them from one scratch array that lives in the
// library itself, so the call allocates nothing.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code never
// dereferences its name (on the host the name only stands in for the symbol);
// its device address is looked up once per device with cudaGetSymbolAddress
// and cached.  All calls share the array and find the previous call's bytes
// in it; nothing there has to start at zero (every byte the kernels read is
// written earlier in the same call), and two calls whose work overlaps on the
// GPU race on it.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"

namespace nvfp4 {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr size_t kAlign = 256;

static __device__ __align__(256) unsigned char g_fc2_scratch[kScratchBytes];

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Device address of g_fc2_scratch on the current device, looked up on the
// first call made with that device current and cached afterwards.
nvfp4_status scratch_address(unsigned char** out) {
  static std::mutex mu;
  static unsigned char* cache[64] = {};
  int dev = 0;
  nvfp4_status st = cuda_check(cudaGetDevice(&dev), "nvfp4_fc2_host_noalloc: cudaGetDevice");
  if (st != NVFP4_OK) return st;
  if (dev < 0 || dev >= 64) return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_host_noalloc: device ordinal above 63");
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_fc2_scratch), "nvfp4_fc2_host_noalloc: cudaGetSymbolAddress");
    if (st != NVFP4_OK) return st;
    if (p == nullptr) return fail(NVFP4_ECUDA, "nvfp4_fc2_host_noalloc: the scratch array has no device address");
    cache[dev] = static_cast<unsigned char*>(p);
  }
  *out = cache[dev];
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_fc2_host_noalloc(const void* gate_up_host, int64_t m, int64_t k, int64_t ld_host,
                                               const void* w_q, const void* w_s, const nvfp4_scale_rec* w_rec,
                                               int64_t n, void* out_host, uint32_t* dev_status,
                                               nvfp4_stream_t stream) {
  using nvfp4::fail;
  using nvfp4::round_up;
  if (!gate_up_host || !w_q || !w_s || !w_rec || !out_host)
    return fail(NVFP4_EINVAL, "nvfp4_fc2_host_noalloc: null pointer");
  if (m < 1 || k < 1 || n < 1) return fail(NVFP4_EINVAL, "nvfp4_fc2_host_noalloc: m, k and n must be positive");
  if (ld_host < 2 * k) return fail(NVFP4_EINVAL, "nvfp4_fc2_host_noalloc: ld_host must be >= 2k");
  if (k % 256 != 0 || n % 128 != 0 || k > (int64_t(1) << 24) || n > (int64_t(1) << 24) || m > (int64_t(1) << 30))
    return fail(NVFP4_EUNSUPPORTED, "nvfp4_fc2_host_noalloc: k must be a multiple of 256 and n of 128 (or too large)");
  if (!nvfp4::aligned16(w_q) || !nvfp4::aligned16(w_s) || !nvfp4::aligned16(w_rec))
    return fail(NVFP4_EALIGN, "nvfp4_fc2_host_noalloc: weight pointers must be 16-byte aligned");
  // the scratch regions, each 256-byte aligned: gate|up, QDATA, scales,
  // record, output
  const size_t x_bytes = round_up(size_t(m) * size_t(2 * k) * 2);
  const size_t q_bytes = round_up(size_t(nvfp4_qdata_bytes(m, k)));
  const size_t s_bytes = round_up(size_t(nvfp4_scale_bytes(m, k)));
  const size_t r_bytes = round_up(sizeof(nvfp4_scale_rec));
  const size_t o_bytes = round_up(size_t(m) * size_t(n) * 2);
  const size_t need = x_bytes + q_bytes + s_bytes + r_bytes + o_bytes;
  if (need > nvfp4::kScratchBytes) {
    char buf[200];
    std::snprintf(buf, sizeof(buf),
                  "nvfp4_fc2_host_noalloc: the step needs %zu bytes of scratch, more than the library's fixed %zu",
                  need, nvfp4::kScratchBytes);
    return fail(NVFP4_EUNSUPPORTED, buf);
  }
  unsigned char* base = nullptr;
  nvfp4_status st = nvfp4::scratch_address(&base);
  if (st != NVFP4_OK) return st;
  unsigned char* x_dev = base;
  unsigned char* a_q = x_dev + x_bytes;
  unsigned char* a_s = a_q + q_bytes;
  auto* a_rec = reinterpret_cast<nvfp4_scale_rec*>(a_s + s_bytes);
  unsigned char* out_dev = a_s + s_bytes + r_bytes;
  return nvfp4_fc2_host(gate_up_host, m, k, ld_host, w_q, w_s, w_rec, n, x_dev, a_q, a_s, a_rec, out_dev, out_host,
                        dev_status, stream);
}
