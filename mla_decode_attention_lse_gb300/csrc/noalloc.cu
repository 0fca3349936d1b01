// noalloc.cu -- mla_attn_combine_uv_noalloc: the fused decode step with its
// scratch in this library's own fixed device buffer, for callers that cannot
// allocate device memory when they run the step.
//
// A serving engine typically reserves nearly all free device memory for its
// KV cache when it starts and may not allocate afterwards; and cudaMalloc can
// synchronise the whole device, which a latency-bound decode loop cannot
// afford.  Such a caller still owns its inputs and outputs, but the step's
// scratch -- the attention's partials and the work-queue / arrival counters
// -- comes from the array below, which every device that loads the library
// holds until the process exits.
//
// The array is one per device and shared by every call: calls whose work
// overlaps on the GPU (two streams, or two threads) race on it and give
// undefined results; run them one after another.  The counters must start at
// zero: the first call on a device clears them once (a memset enqueued on
// that call's stream, before its kernel), and every call leaves them zero
// when it ends.  The partials need no clearing: every element is written
// before it is read.  Because the first call on a device does this set-up
// (the array's address lookup and the clear), make that first call before
// any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mla_combine_uv.h"

namespace {

// 16 MiB: the counter region first, then the partials' LSE and latents.
constexpr int64_t kScratchBytes = 16ll << 20;
constexpr int64_t kCounterWords = 4096;  // 16 KiB: 3 + ceil(B q / 8) words at most
constexpr int64_t kCounterBytes = kCounterWords * 4;

static __device__ __align__(256) unsigned char g_step_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_scratch_ptr[kMaxDevices] = {};

// The array's device address on the current device.  Set-up on the first
// call per device, with that device current: the address lookup (in host
// code the array's name is only a stand-in, never a device address) and the
// counters' clear, enqueued on the caller's stream ahead of its kernel.
int32_t scratch_of_current_device(cudaStream_t stream, unsigned char **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_step_scratch) != cudaSuccess || !ptr) return MLA_ERR_CUDA;
    if (cudaMemsetAsync(ptr, 0, (size_t)kCounterBytes, stream) != cudaSuccess) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(ptr);
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" int32_t mla_attn_combine_uv_noalloc(const mla_attn_combine_uv_args *args, void *stream) {
  if (!args) return MLA_ERR_NULL;
  const mla_attn_combine_uv_args &a = *args;
  if (a.B < 0 || a.q < 1 || a.q > 32 || a.H < 1 || a.H > 65535 || a.spr < 1 || a.spr > 32) return MLA_ERR_SHAPE;
  // what this call's scratch needs, against what the array holds (the token
  // count is bounded first, so nothing below overflows)
  const int64_t S = (int64_t)a.B * a.q;
  if (3 + (S + 7) / 8 > kCounterWords) return MLA_ERR_SCRATCH;
  const int64_t rows = (int64_t)a.spr * S * a.H;
  const int64_t lse_bytes = round_up(rows * 4, 256);
  const int64_t o_bytes = rows * 512 * 2;
  if (kCounterBytes + lse_bytes + o_bytes > kScratchBytes) return MLA_ERR_SCRATCH;
  unsigned char *base = nullptr;
  const int32_t st = scratch_of_current_device(static_cast<cudaStream_t>(stream), &base);
  if (st != MLA_OK) return st;
  mla_attn_combine_uv_args c = a;
  c.workspace = reinterpret_cast<int32_t *>(base);
  c.workspace_words = kCounterWords;
  c.part_lse = reinterpret_cast<float *>(base + kCounterBytes);
  c.part_o = base + kCounterBytes + lse_bytes;
  return mla_attn_combine_uv(&c, stream);
}
