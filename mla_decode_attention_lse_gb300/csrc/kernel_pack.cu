// kernel_pack.cu -- the DCP producer side on one GPU: every rank's attention
// partials (each over all R*H global heads) packed into one destination
// rank's combine buffer, with the LSE masking of the vLLM page
// "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
// (stage_push): the row of global head dst*H + h of token t from rank r goes
// to packed row (r, t, h) unchanged; its LSE is copied bit for bit, or set to
// -inf when rank r holds no KV of the token's request (seq_lens == 0) or the
// token is past the batch (t >= qsl[S/q]).  The packed buffer is the compact
// [R, S, H, 512] layout the combine reads with P = R.
//
// A data move, bound by HBM: one warp moves one 1-KiB row (two 16-byte
// pieces per lane) per iteration, lane 0 its LSE; rows are grid-strided over
// 64 warps per SM.  Measured on the 8-rank decode batch: 1 row per warp at 64
// warps per SM 10.5 us, 2 rows 10.8 us, 4 rows at 32 warps 12.4 us, 8 rows
// 16.9 us -- many warps with little each beat deep batches per warp.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kPackWarps = 8;
constexpr int kPackThreads = kPackWarps * 32;
constexpr int kPackRows = 1;  // rows per warp and iteration

__global__ void __launch_bounds__(kPackThreads, 8) pack_kernel(const __grid_constant__ PackParams p) {
  const int lane = threadIdx.x & 31;
  // rows < 2^31 (the host bounds R*S*H*512 below 2^40): 32-bit index math
  const uint32_t nrows = (uint32_t)p.R * (uint32_t)p.S * (uint32_t)p.H;
  const uint32_t H = (uint32_t)p.H, S = (uint32_t)p.S;
  const uint32_t warps = gridDim.x * kPackWarps;
  const uint32_t w0 = blockIdx.x * kPackWarps + (threadIdx.x >> 5);
  // the partials come from the previous kernel on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  const int rows_live = p.S > 0 ? __ldg(p.qsl + p.S / p.q) : 0;
  const uint32_t neg_inf = 0xFF800000u;
  for (uint32_t base = w0 * kPackRows; base < nrows; base += warps * kPackRows) {
    uint4 v[kPackRows][2];
    uint32_t bits[kPackRows];
    // every load of the batch first: the rows, and (lane 0) each row's
    // request length and LSE
#pragma unroll
    for (int k = 0; k < kPackRows; ++k) {
      const uint32_t row = base + k;  // packed row (r, t, h), h fastest
      bits[k] = neg_inf;
      if (row < nrows) {
        const uint32_t rt = row / H, h = row - rt * H;
        const uint32_t r = rt / S, t = rt - r * S;
        const long long g = (long long)p.dst * p.H + h;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(p.o + (long long)r * p.o_sr + (long long)t * p.o_st + g * p.o_sh);
        v[k][0] = __ldcs(s4 + lane);
        v[k][1] = __ldcs(s4 + lane + 32);
        if (lane == 0) {
          const bool empty = __ldg(p.seq_lens + (long long)r * p.sl_sr + (long long)(t / (uint32_t)p.q)) == 0 ||
                             (int)t >= rows_live;
          const uint32_t b = __float_as_uint(__ldg(p.lse + (long long)r * p.l_sr + (long long)t * p.l_st + g * p.l_sh));
          bits[k] = empty ? neg_inf : b;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPackRows; ++k) {
      const uint32_t row = base + k;
      if (row < nrows) {
        uint4 *d4 = reinterpret_cast<uint4 *>(p.cmb_o + (long long)row * kD);
        d4[lane] = v[k][0];
        d4[lane + 32] = v[k][1];
        if (lane == 0) reinterpret_cast<uint32_t *>(p.cmb_lse)[row] = bits[k];
      }
    }
  }
}

}  // namespace

int pack_threads() { return kPackThreads; }
int pack_grid(long long rows, int num_sms) {
  const long long per_cta = (long long)kPackWarps * kPackRows;
  long long g = (rows + per_cta - 1) / per_cta;
  const long long cap = (long long)num_sms * 8;  // resident CTAs: 8 of 256 threads per SM
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_pack(const PackParams &p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kPackThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pack_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
