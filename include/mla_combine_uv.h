/*
 * mla_combine_uv.h -- C ABI of the GB300 (sm_103a) MLA decode post-attention
 * stage: LSE-weighted merge of partial attention outputs, bf16 or MXFP4
 * rounding of the merged latents, per-head W_UV up-projection, gate.
 *
 * The operation is the one the vLLM API page
 * "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
 * defines (module docstring; functions sane, combine_ranks, combine_splits,
 * stage_combine, stage_uv, wv_loads, host_args, mla_post).  For every token
 * t < S and head h:
 *
 *   R(t)  = the partials token t merges (see "Layouts" below)
 *   l_r   = sane(lse[r, t, h])            NaN and +inf become -inf
 *   m     = max_r l_r  (0 if that is -inf)
 *   e_r   = 2^((l_r - m) * log2 e)        (lse is a natural log)
 *   w_r   = 0 if e_r == 0 or sum e == 0, else e_r / sum e
 *   lat   = bf16( sum_{r : w_r != 0} w_r * o[r, t, h, :] )   fp32 sum
 *   x     = lat (bf16 weights) or MXFP4(lat) (MXFP4 weights: per 32-wide
 *           block an E8M0 scale 2^(floor(log2 amax) - 2), E2M1 elements
 *           rounded to nearest even, saturating at 6)
 *   acc_v = sum_k W_V[h][v][k] * x[k]      fp32
 *   out[t, h*128 + v] = bf16( bf16(acc_v) * gate[t, h*128 + v] )
 *
 * and out[t, :] = 0 for S <= t < S_out.
 *
 * Layouts (chosen by P):
 *   P == 1                         passthrough: lat = o[0, t, h, :] as is;
 *                                  lse is ignored and may be NULL.
 *   P == splits_per_request        compact / stacked partials: every token
 *                                  merges partials 0 .. P-1.
 *   P == (S / q) * splits_per_request, S % q == 0
 *                                  request-major split-KV partials: token t
 *                                  merges (t/q)*spr .. (t/q)*spr + spr - 1.
 *   anything else                  MLA_ERR_LAYOUT.
 *
 * Ownership: the caller owns every buffer; the library allocates nothing per
 * call.  All pointers are DEVICE pointers of the current CUDA device except
 * where a field says otherwise.  Calls are asynchronous on `stream` (a
 * cudaStream_t passed as void*; NULL is the legacy default stream).
 * Validation errors return before anything is launched and leave `out`
 * untouched.  `out` must not overlap any input.
 */
#ifndef MLA_COMBINE_UV_H
#define MLA_COMBINE_UV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 6

/* W_V storage format. */
enum {
  MLA_W_BF16 = 0,  /* w_v: bf16 [H, 128, 512]                                  */
  MLA_W_MXFP4 = 1  /* w_v: u8 [H, 128, 256] E2M1 pairs (element 2i in the low
                      nibble of byte i); w_scale: u8 [H, 128, 16] E8M0, one per
                      32 elements along K                                      */
};

/* Status codes. */
enum {
  MLA_OK = 0,
  MLA_ERR_NULL = 1,    /* a required pointer is NULL                          */
  MLA_ERR_SHAPE = 2,   /* S < 0, S_out < S, H < 1, P < 1, q < 1, spr < 0, or a
                          size too large for 32-bit token / unit indexing     */
  MLA_ERR_STRIDE = 3,  /* a stride is not a multiple of 8 elements (16 bytes)
                          where 16-byte vector or TMA access needs it        */
  MLA_ERR_ALIGN = 4,   /* a base pointer is not 16-byte aligned               */
  MLA_ERR_FMT = 5,     /* w_fmt is not MLA_W_BF16 / MLA_W_MXFP4               */
  MLA_ERR_LAYOUT = 6,  /* (P, q, splits_per_request) is not one of the layouts */
  MLA_ERR_CUDA = 7,    /* a CUDA runtime / driver call failed                 */
  MLA_ERR_TIMEOUT = 8, /* a kernel gave up a bounded wait (reported by
                          mla_combine_uv_status)                              */
  MLA_ERR_KERNEL = 9,  /* the requested kernel cannot run this problem        */
  MLA_ERR_DATA = 10,   /* a kernel met invalid device data: a kv_len outside
                          [0, Lmax] (reported by mla_combine_uv_status)       */
  MLA_ERR_SCRATCH = 11 /* mla_attn_combine_uv_noalloc: the problem needs more
                          scratch than the library's fixed device buffer holds
                          (nothing launched)                                  */
};

/* Kernel selection. */
enum {
  MLA_KERNEL_AUTO = 0, /* pick by size (the plan says which)                  */
  MLA_KERNEL_SIMT = 1, /* CUDA-core kernel: any P; the small-batch path       */
  MLA_KERNEL_TC = 2,   /* fused tcgen05 kernel: partials per token <= 32
                          (<= 16 with 32-token tiles)                        */
  MLA_KERNEL_KSPLIT = 3 /* a (head, 16-token) unit per 4-CTA cluster, the
                          512 latents split over the cluster and the partial
                          GEMMs summed through distributed shared memory;
                          partials per token <= 16, S >= 1; on request only
                          (automatic choice never picks it)                   */
};

typedef struct {
  int32_t S;                  /* token rows of o (and of gate)                */
  int32_t S_out;              /* rows of out, >= S; rows S.. are zeroed       */
  int32_t H;                  /* heads; gate / out rows are H*128 wide        */
  int32_t P;                  /* partials along o's first dimension           */
  int32_t q_per_request;      /* queries per request (request-major layout)   */
  int32_t splits_per_request; /* splits each request's tokens merge           */

  const void *o;              /* bf16 [P, S, H, 512]: element (r,t,h,d) at
                                 r*o_sp + t*o_st + h*o_sh + d; strides in
                                 elements, multiples of 8; 16-byte aligned     */
  int64_t o_sp, o_st, o_sh;

  const float *lse;           /* f32 [P, S, H]: (r,t,h) at r*l_sp + t*l_st +
                                 h*l_sh; natural-log LSE; may be NULL iff P==1 */
  int64_t l_sp, l_st, l_sh;

  const void *w_v;            /* W_V[h][v][k] at h*w_sh + v*w_sv + k (bf16
                                 elements) or + k/2 (MXFP4 bytes); strides
                                 multiples of 8 elements (bf16) / 16 bytes     */
  int64_t w_sh, w_sv;
  const uint8_t *w_scale;     /* E8M0 scale of (h, v, k/32) at h*s_sh + v*s_sv
                                 + k/32 (MXFP4 only; NULL for bf16)           */
  int64_t s_sh, s_sv;
  int32_t w_fmt;              /* MLA_W_BF16 or MLA_W_MXFP4                   */

  const void *gate;           /* bf16 [S, H*128], dense row-major            */
  void *out;                  /* bf16 [S_out, H*128], dense row-major        */

  int32_t kernel;             /* MLA_KERNEL_*; 0 = automatic                  */
  int32_t tile_tokens;        /* tensor-core token tile (8, 16 or 32; 8 added
                                 in ABI version 4: two warps per token, each
                                 merging half of its latents; 17..31 added in
                                 version 5: the 32-token kernel with that many
                                 tokens per unit, <= 16 partials); 0 = auto  */
  int64_t wait_ns;            /* limit of the tensor-core kernel's bounded
                                 waits, in ns; 0 = the default 0.5 s.  A wait
                                 that runs out makes the kernel stop, drain its
                                 own copies and MMAs (those drains keep the
                                 default limit), free TMEM and return;
                                 mla_combine_uv_status then reports
                                 MLA_ERR_TIMEOUT and `out` is undefined.  The
                                 other kernels use the default.  (Added in ABI
                                 version 5.)                                  */
  const int32_t *ready_flag;  /* optional device int32 (NULL: none).  The
                                 producer's completion flag of the page's
                                 flag handshake (the combine polls the flags
                                 its producer raises once the partials are
                                 written): every CTA waits, bounded by wait_ns,
                                 until the value is non-zero before it reads
                                 o, lse or gate.  A flag still zero when the
                                 limit runs out ends the call with
                                 MLA_ERR_TIMEOUT.  The producer must not be a
                                 kernel that itself waits for this call.
                                 Tensor-core kernel only (other kernels:
                                 MLA_ERR_KERNEL).  (Added in ABI version 5.) */
} mla_combine_uv_args;

/* What a call would launch (host-side planning only). */
typedef struct {
  int32_t kernel;        /* MLA_KERNEL_SIMT, _TC or _KSPLIT                   */
  int32_t layout;        /* 0 passthrough, 1 compact, 2 request-major         */
  int32_t n_part;        /* partials each token merges                        */
  int32_t tile_tokens;   /* tokens per work unit                              */
  int32_t units;         /* (head, token tile) work units                     */
  int32_t grid;          /* CTAs launched (KSPLIT: 4 per unit, as clusters)   */
  int32_t threads;       /* threads per CTA                                   */
  int32_t smem_bytes;    /* dynamic shared memory per CTA                     */
  int32_t offsets32;     /* 1: every element offset the call dereferences in
                            o, lse, gate and out is below 2^32, and the kernel
                            computes addresses in 32-bit arithmetic; 0: 64-bit
                            (added in ABI version 2)                         */
} mla_plan;

/*
 * mla_combine_uv -- run the stage on `stream`.
 * Returns MLA_OK once the kernel is enqueued, or an MLA_ERR_* code (nothing
 * launched).  Kernel-side failures (a bounded wait that gave up) are reported
 * by mla_combine_uv_status.
 */
int32_t mla_combine_uv(const mla_combine_uv_args *args, void *stream);

/*
 * mla_combine_uv_plan -- validate `args` and describe the launch a call would
 * make on a GPU with `num_sms` SMs (pass 0 to ask the current device).
 * Pure host logic when num_sms > 0: no CUDA call is made.
 */
int32_t mla_combine_uv_plan(const mla_combine_uv_args *args, int32_t num_sms, mla_plan *plan);

/*
 * mla_combine_uv_status -- read and clear the device-side error word of the
 * current device, in order on `stream`: the read and the clear are enqueued
 * on `stream`, which is then synchronised.  The word is ONE per device: it
 * collects the first error of any kernel of this library on any stream of
 * the device, so a caller that runs the library on several streams should
 * synchronise them (or the device) before asking, or it may see (and clear)
 * another stream's error.  Returns MLA_OK, MLA_ERR_TIMEOUT (a kernel
 * abandoned a bounded wait; its output is undefined), MLA_ERR_DATA
 * (mla_attn_split_kv met a kv_len outside [0, Lmax]) or MLA_ERR_CUDA.
 */
int32_t mla_combine_uv_status(void *stream);

/*
 * The DCP producer side on one GPU -- stage_push of the vLLM page
 * "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
 * (section "stage_push(c)"): with decode context parallelism over R ranks,
 * rank r's attention leaves partials of every token for all R*H global heads;
 * destination rank p combines, for its H heads, the R ranks' partials.  Here
 * every rank's partials are resident on one GPU and one call packs rank p's
 * combine buffer: packed row (r, t, h) is the partial of global head
 * p*H + h of token t from rank r, copied unchanged; its LSE is copied bit for
 * bit, or set to -inf when rank r holds no KV of the token's request
 * (seq_lens[r][t/q] == 0) or the token is past the batch (t >= qsl[S/q]).
 * The packed buffer is the compact layout mla_combine_uv reads with P = R
 * (splits_per_request = R): cmb_o o_sp = S*H*512, o_st = H*512, o_sh = 512.
 */
typedef struct {
  int32_t S;             /* token rows of the (padded) batch; S % q == 0      */
  int32_t H;             /* heads per rank; a rank's partials have R*H heads  */
  int32_t R;             /* ranks, >= 1; R*H <= 65535                         */
  int32_t q_per_request; /* queries per request: token t is of request t / q  */
  int32_t dst_rank;      /* the destination rank p, 0 <= p < R                */

  const void *o;         /* bf16 [R, S, R*H, 512]: (r, t, g, d) at r*o_sr +
                            t*o_st + g*o_sh + d; strides in elements,
                            multiples of 8; 16-byte aligned                   */
  int64_t o_sr, o_st, o_sh;
  const float *lse;      /* f32 [R, S, R*H]: (r, t, g) at r*l_sr + t*l_st +
                            g*l_sh                                            */
  int64_t l_sr, l_st, l_sh;
  const int32_t *seq_lens; /* int32: rank r's local KV length of request j at
                              r*sl_sr + j (j < S/q); 0 = empty               */
  int64_t sl_sr;
  const int32_t *qsl;    /* int32 [S/q + 1] query start locations; rows
                            t >= qsl[S/q] are past the batch                  */

  void *cmb_o;           /* bf16 [R, S, H, 512], dense, 16-byte aligned; the
                            caller owns it                                    */
  float *cmb_lse;        /* f32 [R, S, H], dense                              */
} mla_dcp_pack_args;

/*
 * mla_dcp_pack -- enqueue the pack on `stream` (a copy bound by HBM: it reads
 * and writes R*S*H rows of 1 KiB).  Returns MLA_OK, or MLA_ERR_NULL /
 * _SHAPE / _STRIDE / _ALIGN before anything is launched (the outputs are
 * untouched), or MLA_ERR_CUDA.  S == 0 launches nothing.  (Added in ABI
 * version 2.)
 */
int32_t mla_dcp_pack(const mla_dcp_pack_args *args, void *stream);

/*
 * The partial producer: split-KV MLA decode attention in the absorbed form,
 * writing the partials mla_combine_uv merges.  The vLLM page
 * "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back" names
 * this producer (M1c, mla_attn: o / lse of dense [splits, S, 12, 512] bf16 /
 * [splits, S, 12] f32, a request's splits merged LSE-weighted) but does not
 * print it; the call computes the plain definition:
 *   S = B * q query tokens, token t = b*q + i of request b; head h's query row
 *   qv[t][h] is 576 wide (the latent query with W_UK absorbed, then the rope
 *   query); cached position j of request b is kv[b][j] (the latent, 512, then
 *   the rope key, 64).  Token i sees positions j < kv_len[b] - (q - 1 - i).
 *   Split r of request b covers [r C, (r + 1) C), C = ceil(kv_len[b] / spr).
 *   For split r, token t, head h over the positions of the split it sees:
 *     lse[r][t][h] = ln sum_j exp(scale * qv[t][h] . kv[b][j])   (f32)
 *     o[r][t][h][:] = sum_j exp(scale * qv . kv[b][j] - lse) kv[b][j][0:512]
 *   rounded to bf16; a split with no visible position has lse -inf, o 0.
 * The outputs are the compact layout of mla_combine_uv with P = spr
 * (splits_per_request = spr): o_sp = S*H*512, o_st = H*512, o_sh = 512.
 * Scores accumulate in fp32 on the tensor cores, the softmax weights enter the
 * latent sum as bf16, the sum accumulates in fp32.
 */
typedef struct {
  int32_t B;             /* requests, >= 0                                    */
  int32_t q;             /* queries per request, 1 <= q <= 32                 */
  int32_t H;             /* heads, >= 1                                       */
  int32_t spr;           /* splits per request, >= 1                          */
  float scale;           /* softmax scale on q . k (finite)                   */
  const void *qv;        /* bf16 [S, H, 576]: (t, h, k) at t*q_st + h*q_sh + k;
                            strides in elements, multiples of 8; 16-byte
                            aligned                                           */
  int64_t q_st, q_sh;
  const void *kv;        /* bf16 [B, Lmax, 576]: (b, j, k) at b*kv_sb +
                            j*kv_sl + k; strides multiples of 8 elements;
                            16-byte aligned.  Rows past kv_len[b] are never
                            used (they may hold anything)                     */
  int64_t kv_sb, kv_sl;
  int32_t Lmax;          /* cached positions per request in kv, >= 1          */
  const int32_t *kv_len; /* device int32 [B]: cached positions of request b,
                            its q new tokens included; a value outside
                            [0, Lmax] is clamped and reported as
                            MLA_ERR_DATA by mla_combine_uv_status              */
  void *o;               /* bf16 [spr, S, H, 512], dense, 16-byte aligned;
                            caller-owned, every element written               */
  float *lse;            /* f32 [spr, S, H], dense                            */
  int32_t kernel;        /* 0 automatic (= 1); 1 one CTA per (request, split,
                            head group); 2 on request: a 2-CTA cluster per
                            item, each CTA holding half of every cached row's
                            latents and the partial scores summed through
                            distributed shared memory (the fp32 score sum is
                            split in two and added once, so o / lse may
                            differ from kernel 1 in the last bits).  (Added
                            in ABI version 5.)                                */
} mla_attn_split_kv_args;

/*
 * mla_attn_split_kv -- enqueue the attention on `stream` (a persistent grid
 * over (request, split, group of heads) items; reads each cached row once
 * per group of up to 32 / q heads).  Returns MLA_OK, or MLA_ERR_NULL /
 * _SHAPE / _STRIDE / _ALIGN / _KERNEL before anything is launched (outputs
 * untouched), or MLA_ERR_CUDA.  B == 0 launches nothing.  The library
 * allocates nothing; kv_len is read on the device.  (Added in ABI version 3.)
 */
int32_t mla_attn_split_kv(const mla_attn_split_kv_args *args, void *stream);

/*
 * Downstream of the stage: this rank's o_proj shard.  The vLLM page
 * "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back" ends
 * the stage at "o_proj's input" (core); o_proj is a row-parallel linear layer,
 * so the rank computes out[t][j] = sum_k core[t][k] * W[j][k] over its own
 * H*128 inputs and the tensor-parallel all-reduce (multi-GPU, not part of
 * this library) sums the ranks' outputs.  Accumulation in fp32 on the tensor
 * cores, out rounded to bf16 once.
 */
typedef struct {
  int32_t S;             /* tokens, >= 0                                      */
  int32_t K;             /* input width (H*128), a multiple of 64             */
  int32_t Nout;          /* output features, a multiple of 64                 */
  const void *x;         /* bf16 [S, K] (core): row stride x_st (elements, a
                            multiple of 8, >= K); 16-byte aligned             */
  int64_t x_st;
  const void *w;         /* bf16 [Nout, K] (the linear layer's weight slice):
                            row stride w_sj (a multiple of 8, >= K); 16-byte
                            aligned                                           */
  int64_t w_sj;
  void *out;             /* bf16 [S, Nout]: row stride out_st (>= Nout);
                            caller-owned, every element written               */
  int64_t out_st;
} mla_o_proj_args;

/*
 * mla_o_proj -- enqueue the o_proj shard on `stream` (a persistent
 * tensor-core GEMM; at decode sizes it streams the weight from HBM).
 * Returns MLA_OK, or MLA_ERR_NULL / _SHAPE / _STRIDE / _ALIGN before anything
 * is launched (out untouched), or MLA_ERR_CUDA.  S == 0 launches nothing.
 * (Added in ABI version 3.)
 */
int32_t mla_o_proj(const mla_o_proj_args *args, void *stream);

/*
 * The decode step's attention and its combine in ONE launch: the partial
 * producer of mla_attn_split_kv followed, in the same persistent grid, by
 * mla_combine_uv on its partials (compact layout, P = spr) -- the pairing the
 * vLLM page "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.
 * mla_back" describes in its module docstring (M1c's partials, a token's
 * request's splits merged by the combine) and in combine_splits' branch that
 * runs with M1c in the same launch.  Each result is the same as the two calls
 * in sequence would give: o / lse partials as mla_attn_split_kv defines them
 * (they are written to part_o / part_lse and read back within the call), and
 * out[t, h*128 + v] as mla_combine_uv defines it, rows S .. S_out - 1 zero.
 *
 * The attention's work items come from a queue shared by the CTAs; once an
 * item's partials are written it adds one arrival to each 8-token tile its
 * request covers.  Behind the attention items the queue holds the combine's
 * (8-token tile, head) units; a CTA reaches one only after its own attention
 * items, and waits (bounded by wait_ns) until the tile's items have all
 * arrived -- items that running CTAs hold and that never wait on a combine
 * unit.  With n_out > 0 the queue then holds o_proj units (64 outputs x 64
 * tokens): a CTA reaches one only after its combine units; it copies its
 * weight rows at once and waits (bounded by wait_ns) until every combine unit
 * has stored its core rows -- units held by running CTAs that never wait on
 * an o_proj unit.  The workspace carries the queue, the arrival counters and
 * the count of stored combine units.
 */
typedef struct {
  /* the attention, as in mla_attn_split_kv_args */
  int32_t B, q, H, spr;  /* q <= 32; spr <= 32                                 */
  float scale;
  const void *qv;        /* bf16 [S, H, 576], S = B * q                        */
  int64_t q_st, q_sh;
  const void *kv;        /* bf16 [B, Lmax, 576]                                 */
  int64_t kv_sb, kv_sl;
  int32_t Lmax;
  const int32_t *kv_len; /* device int32 [B]                                    */
  void *part_o;          /* bf16 [spr, S, H, 512] dense: the partials (caller-
                            owned scratch, written and read in the call)      */
  float *part_lse;       /* f32 [spr, S, H] dense                               */
  /* the combine, as in mla_combine_uv_args with P = splits_per_request = spr */
  const void *w_v;       /* bf16 [H, 128, 512]: W_V[h][v][k] at h*w_sh + v*w_sv
                            + k; strides multiples of 8 elements; 16-byte
                            aligned                                           */
  int64_t w_sh, w_sv;
  const uint8_t *w_scale; /* must be NULL (MXFP4 W_V: MLA_ERR_FMT)             */
  int64_t s_sh, s_sv;
  int32_t w_fmt;         /* MLA_W_BF16                                         */
  const void *gate;      /* bf16 [S, H*128] dense                               */
  void *out;             /* bf16 [S_out, H*128] dense, caller-owned            */
  int32_t S_out;         /* >= S                                                */
  int32_t *workspace;    /* device int32 [mla_attn_combine_uv_workspace_words(
                            B, q)]: zero before the first call; every call
                            leaves it zero (also after a timeout).  One call
                            at a time per workspace.                          */
  int64_t workspace_words;
  int64_t wait_ns;       /* limit of the waits for a tile's partials (and of
                            o_proj's wait for the core rows), in ns; 0 = the
                            default 0.5 s                                     */
  /* o_proj in the same launch (ABI version 6; n_out == 0: none).  The page's
     stage ends at "o_proj's input"; with n_out > 0 the same grid then computes
     this rank's o_proj shard on the core rows it just wrote, exactly as
     mla_o_proj defines it: y[t][j] = bf16(sum_k out[t][k] w_o[j][k]) over
     k < H*128 (fp32 accumulation, one rounding), t < S.  The tensor-parallel
     all-reduce of the shards is the caller's.                                */
  const void *w_o;       /* bf16 [n_out, H*128]: w_o[j][k] at j*w_o_sj + k;
                            16-byte aligned                                   */
  int64_t w_o_sj;        /* >= H*128, multiple of 8 elements                  */
  int32_t n_out;         /* 0, or a multiple of 64                            */
  void *y;               /* bf16 [S, y_st], caller-owned                      */
  int64_t y_st;          /* >= n_out                                          */
} mla_attn_combine_uv_args;

/* Workspace words (int32) that mla_attn_combine_uv needs for B requests of q
 * tokens: 3 + ceil(B*q / 8) (ABI version 6; version 5 needed 2 + ...).
 * Returns -1 for B < 0 or q < 1. */
int64_t mla_attn_combine_uv_workspace_words(int32_t B, int32_t q);

/*
 * mla_attn_combine_uv -- enqueue the fused decode step on `stream`.  Returns
 * MLA_OK, or MLA_ERR_NULL / _SHAPE / _STRIDE / _ALIGN / _FMT before anything
 * is launched (outputs untouched), or MLA_ERR_CUDA.  B == 0 (S = 0) only
 * zeroes out's S_out rows (a memset on `stream`).
 * Kernel-side failures (a kv_len outside [0, Lmax]: MLA_ERR_DATA; a wait that
 * ran out: MLA_ERR_TIMEOUT) are reported by mla_combine_uv_status.
 * (Added in ABI version 5.)
 */
int32_t mla_attn_combine_uv(const mla_attn_combine_uv_args *args, void *stream);

/*
 * mla_attn_combine_uv_noalloc -- the same decode step as mla_attn_combine_uv,
 * for callers that cannot allocate device memory when they run it (a serving
 * engine that hands nearly all free device memory to its KV cache at start-up
 * and may not allocate afterwards; a decode loop that cannot afford the
 * device-wide synchronisation cudaMalloc can cause).  The pages have no
 * counterpart to this call: it exists for those callers only.
 *
 * The caller passes the inputs and `out` as for mla_attn_combine_uv; the
 * fields part_o, part_lse, workspace and workspace_words are not read.  The
 * step's scratch (the partials and the work-queue / arrival counters) lives
 * in one fixed 16 MiB device array inside the library, which every device
 * that loads the library holds until the process exits; the call allocates
 * nothing and calls no allocating routine.  Limits: 16 KiB of counters
 * (B*q <= 32744 tokens) and spr * B*q * H * (1024 + 4) bytes of partials
 * (LSE rounded up to 256 bytes) within the remaining 16 MiB - 16 KiB; a
 * bigger problem returns MLA_ERR_SCRATCH before anything is launched (the
 * decode step of 64 requests x 12 heads x 16 splits needs 12.6 MB).
 *
 * The array is shared by every call on a device, and keeps the last call's
 * contents: calls whose work overlaps on the GPU race on it (undefined
 * results), so run them one after another.  The first call on a device does
 * the set-up -- it looks the array's address up and clears its counters (a
 * memset on `stream`, ahead of the kernel) -- so make that first call before
 * any stream capture.  Every call leaves the counters zero.  Returns as
 * mla_attn_combine_uv does, plus MLA_ERR_SCRATCH.
 */
int32_t mla_attn_combine_uv_noalloc(const mla_attn_combine_uv_args *args, void *stream);

/* A short English description of a status code (static storage). */
const char *mla_status_str(int32_t status);

/* MLA_ABI_VERSION of the loaded library. */
int32_t mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_COMBINE_UV_H */
