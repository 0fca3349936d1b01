// kernel_oproj.h -- launch entry of the o_proj shard kernel (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// This rank's o_proj shard: out[t][j] = sum_k x[t][k] W[j][k] (x = core rows,
// W = the rank's slice of the linear layer's weight, [Nout, K]).  Both
// operands come by TMA through `wmap` (W, boxes of 64 x 64) and `xmap` (x,
// boxes of 64 x NT rows), both with the 128-byte swizzle.
struct OprojParams {
  int S, K, Nout;   // tokens, input width, output features (K % 64 == 0, Nout % 64 == 0)
  int nt;           // tokens per unit (64, 128 or 256)
  uint16_t *out;    // bf16 [S, Nout], row stride out_st
  long long out_st;
  int *err;         // device error word
};

int oproj_tokens_per_unit(int S);  // NT
size_t oproj_smem_bytes(int nt);
cudaError_t launch_oproj(const OprojParams &p, const CUtensorMap &wmap, const CUtensorMap &xmap, int num_sms,
                         cudaStream_t stream);

}  // namespace mla
