// kernel_calib.cu -- the read-only streaming kernel of mla_calib_stream_read:
// the fastest one launch of this library's launch shape can read a given
// number of bytes (a measurement aid; the stage itself is elsewhere).
//
// Every thread issues eight 16-byte streaming loads before it uses any of
// them, the grid covers the range in one pass when it fits four 256-thread
// CTAs per SM (else the threads loop), and nothing is written unless the xor
// of all the data equals a fixed pattern.  Optional dependent round trips
// come first: each reads one word at an address that depends on the word
// before, and the stream waits on the last one.  Launched with programmatic
// stream serialization, like the stage's kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "device_common.cuh"
#include "mla_calibration.h"

namespace mla {

namespace {

constexpr int kCalibThreads = 256;
constexpr int kCalibInFlight = 8;
constexpr uint32_t kNeverWord = 0x7FC00001u;  // a NaN pattern the caller's data does not hold
constexpr uint32_t kSinkPattern = 0x9E3779B9u;

__device__ __forceinline__ uint32_t ld_cg_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kCalibThreads) calib_kernel(const uint4 *src, long long n16, int nrt,
                                                               uint32_t *sink) {
  grid_launch_dependents();
  grid_dependency_wait();
  const uint32_t *w32 = reinterpret_cast<const uint32_t *>(src);
  uint32_t dep = 0u;
  for (int i = 0; i < nrt; ++i) dep = ld_cg_u32(w32 + 4 * i + (dep == kNeverWord ? 1 : 0));
  if (dep == kNeverWord) return;  // not for the caller's data: the loads below wait for the chain
  const long long stride = (long long)gridDim.x * kCalibThreads;
  uint32_t x = 0u;
  for (long long b = (long long)blockIdx.x * kCalibThreads + threadIdx.x; b < n16; b += kCalibInFlight * stride) {
    uint4 v[kCalibInFlight];
#pragma unroll
    for (int k = 0; k < kCalibInFlight; ++k) {
      const long long j = b + k * stride;
      v[k] = j < n16 ? __ldcs(src + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kCalibInFlight; ++k) x ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  if (x == kSinkPattern) sink[0] = x;
}

std::mutex g_calib_mu;
int g_calib_sms[64] = {};

}  // namespace

}  // namespace mla

extern "C" int32_t mla_calib_stream_read(const void *src, int64_t bytes, int32_t dependent_round_trips,
                                         uint32_t *sink, void *stream) {
  if (!src || !sink) return 1;
  if (bytes < 64 || bytes % 16 || dependent_round_trips < 0 || dependent_round_trips > 4) return 2;
  if (reinterpret_cast<uintptr_t>(src) % 16) return 4;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 7;
  int sms;
  {
    std::lock_guard<std::mutex> lk(mla::g_calib_mu);
    if (!mla::g_calib_sms[dev] &&
        cudaDeviceGetAttribute(&mla::g_calib_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 7;
    sms = mla::g_calib_sms[dev];
  }
  const long long n16 = bytes / 16;
  const long long per_cta = (long long)mla::kCalibThreads * mla::kCalibInFlight;
  long long grid = (n16 + per_cta - 1) / per_cta;
  if (grid > 4LL * sms) grid = 4LL * sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(mla::kCalibThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mla::calib_kernel, static_cast<const uint4 *>(src), n16, (int)dependent_round_trips,
                         sink) != cudaSuccess)
    return 7;
  return cudaGetLastError() == cudaSuccess ? 0 : 7;
}
