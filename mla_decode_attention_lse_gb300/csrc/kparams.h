// kparams.h -- launch parameters shared by the host dispatcher and kernels.
#pragma once

#include <stdint.h>

namespace mla {

enum Layout : int { kPassthrough = 0, kCompact = 1, kRequestMajor = 2 };

// Default limit of a bounded wait (ns); a healthy wait lasts microseconds.
constexpr unsigned long long kDefaultWaitNs = 500ull * 1000ull * 1000ull;

// Error codes a kernel writes into the device error word (first one wins).
enum KernelError : int { kErrNone = 0, kErrWaitLatent = 1, kErrWaitMma = 2, kErrWaitAccEmpty = 3,
                         kErrWaitWv = 4, kErrWaitTeardown = 5,
                         kErrWaitPeer = 6, kErrWaitAttn = 7,
                         kErrKvLen = 8, kErrWaitFlag = 9, kErrWaitTile = 10 };

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
  unsigned long long wait_ns;  // limit of the pipeline's bounded waits (ns)
  const int *ready_flag;       // optional: wait until non-zero before reading inputs
  int *err;          // device error word
};

// The partial producer: split-KV MLA decode attention (absorbed form).  One
// CTA per (request, split, head group); the cached rows come by TMA through
// a tensor map passed beside these parameters.
struct AttnParams {
  int B, q, H, spr;  // requests, queries per request, heads, splits per request
  int G, groups;     // heads per CTA, head groups (ceil(H / G))
  int Lmax;          // cached positions per request in the cache tensor
  float scale_log2;  // softmax scale times log2(e)
  const uint16_t *qv;  // bf16 [S, H, 576] (latent query, then rope query)
  long long q_st, q_sh;
  const int32_t *kv_len;  // [B]
  uint16_t *o;       // bf16 [spr, S, H, 512] dense
  float *lse;        // f32 [spr, S, H] dense
  int *err;          // device error word
  // The combine fused behind the attention (mla_attn_combine_uv) only:
  int *ws;           // workspace: [0] work queue, [1] CTAs done, [2 + k] arrivals of token tile k,
                     // [2 + ntiles] combine units stored
  int ntiles;        // 8-token tiles of the batch, ceil(S / 8)
  int S_out;         // rows of out (rows S .. S_out - 1 are zeroed)
  const uint16_t *gate;  // bf16 [S, H*128] dense
  uint16_t *out;     // bf16 [S_out, H*128] dense
  unsigned long long wait_ns;  // limit of the waits for a tile's partials
  // o_proj in the same launch (n_out > 0): y[t][j] = sum_k out[t][k] w_o[j][k]
  // over k < H*128, units of 64 outputs x 64 tokens behind the combine units
  int n_out;         // outputs, a multiple of 64 (0: no o_proj)
  int op_units;      // (n_out / 64) * ceil(S / 64)
  uint16_t *y;       // bf16 [S, y_st]
  long long y_st;
};

// The DCP producer side (pack into one destination rank's combine buffer).
struct PackParams {
  int S, H, R, q, dst;  // tokens, heads per rank, ranks, queries per request, destination
  const uint16_t *o;    // bf16 [R, S, R*H, 512]
  long long o_sr, o_st, o_sh;
  const float *lse;     // f32 [R, S, R*H]
  long long l_sr, l_st, l_sh;
  const int32_t *seq_lens;  // int32 [R, S/q]
  long long sl_sr;
  const int32_t *qsl;   // int32 [S/q + 1]
  uint16_t *cmb_o;      // bf16 [R, S, H, 512] dense
  float *cmb_lse;       // f32 [R, S, H] dense
};

}  // namespace mla
