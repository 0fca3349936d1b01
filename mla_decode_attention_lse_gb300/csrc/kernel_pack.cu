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
// pieces per lane), four rows per warp and iteration, all loads issued
// before the stores; lane 0 writes the row's LSE.  Rows are grid-strided.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kPackWarps = 8;
constexpr int kPackThreads = kPackWarps * 32;
constexpr int kPackRows = 4;  // rows per warp and iteration

__global__ void __launch_bounds__(kPackThreads, 4) pack_kernel(const __grid_constant__ PackParams p) {
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)p.R * p.S * p.H;
  const long long warps = (long long)gridDim.x * kPackWarps;
  const long long w0 = (long long)blockIdx.x * kPackWarps + (threadIdx.x >> 5);
  // the partials come from the previous kernel on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  const int rows_live = p.S > 0 ? __ldg(p.qsl + p.S / p.q) : 0;
  const uint32_t neg_inf = 0xFF800000u;
  for (long long base = w0 * kPackRows; base < nrows; base += warps * kPackRows) {
    uint4 v[kPackRows][2];
    const uint16_t *src[kPackRows];
#pragma unroll
    for (int k = 0; k < kPackRows; ++k) {
      const long long row = base + k;  // packed row (r, t, h), h fastest
      src[k] = nullptr;
      if (row < nrows) {
        const int h = (int)(row % p.H);
        const long long rt = row / p.H;
        const int t = (int)(rt % p.S), r = (int)(rt / p.S);
        src[k] = p.o + (long long)r * p.o_sr + (long long)t * p.o_st + (long long)(p.dst * p.H + h) * p.o_sh;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src[k]);
        v[k][0] = __ldcs(s4 + lane);
        v[k][1] = __ldcs(s4 + lane + 32);
      }
    }
#pragma unroll
    for (int k = 0; k < kPackRows; ++k) {
      const long long row = base + k;
      if (row < nrows) {
        uint4 *d4 = reinterpret_cast<uint4 *>(p.cmb_o + row * kD);
        d4[lane] = v[k][0];
        d4[lane + 32] = v[k][1];
        if (lane == 0) {
          const int h = (int)(row % p.H);
          const long long rt = row / p.H;
          const int t = (int)(rt % p.S), r = (int)(rt / p.S);
          const bool empty = __ldg(p.seq_lens + (long long)r * p.sl_sr + t / p.q) == 0 || t >= rows_live;
          const uint32_t bits =
              empty ? neg_inf
                    : __float_as_uint(__ldg(p.lse + (long long)r * p.l_sr + (long long)t * p.l_st +
                                            (long long)(p.dst * p.H + h) * p.l_sh));
          reinterpret_cast<uint32_t *>(p.cmb_lse)[row] = bits;
        }
      }
    }
  }
}

}  // namespace

int pack_threads() { return kPackThreads; }
int pack_grid(long long rows, int num_sms) {
  const long long per_cta = (long long)kPackWarps * kPackRows;
  long long g = (rows + per_cta - 1) / per_cta;
  const long long cap = (long long)num_sms * 4;  // resident CTAs: 4 of 256 threads per SM
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
