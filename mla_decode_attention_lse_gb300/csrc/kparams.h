// kparams.h -- launch parameters shared by the host dispatcher and kernels.
#pragma once

#include <stdint.h>

namespace mla {

enum Layout : int { kPassthrough = 0, kCompact = 1, kRequestMajor = 2 };

// Error codes a kernel writes into the device error word (first one wins).
enum KernelError : int { kErrNone = 0, kErrWaitLatent = 1, kErrWaitMma = 2, kErrWaitAccEmpty = 3,
                         kErrWaitWv = 4, kErrWaitTeardown = 5,
                         kErrWaitPeer = 6 };

struct KParams {
  int S, S_out, H;
  int layout;        // Layout
  int n_part;        // partials per token (1 for passthrough)
  int q, spr;        // queries / splits per request (request-major)
  const uint16_t *o; // bf16 bits
  long long o_sp, o_st, o_sh;
  const float *lse;
  long long l_sp, l_st, l_sh;
  const void *w_v;
  long long w_sh, w_sv;
  const uint8_t *w_scale;
  long long s_sh, s_sv;
  int w_fmt;         // 0 bf16, 1 MXFP4
  const uint16_t *gate;
  uint16_t *out;
  int tile;          // tokens per work unit
  int tiles_per_head;
  int units;         // H * tiles_per_head
  int off32;         // every element offset into o, lse, gate and out that is
                     // read or written is below 2^32 (32-bit address arithmetic)
  int *err;          // device error word
};

}  // namespace mla
