/*
 * mla_oracle.h -- interface of the CPU oracle (test infrastructure only; the
 * CUDA library neither includes nor links it).
 *
 * Definition followed: the vLLM API page
 * "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back",
 * functions sane, combine_ranks, combine_splits, stage_combine, stage_uv,
 * mla_post and stage_push.  All strides are in elements.
 */
#ifndef MLA_ORACLE_H
#define MLA_ORACLE_H
#include <stdint.h>

typedef struct {
  int S, S_out, H;    /* tokens of o, rows of out, heads                    */
  int P, q, spr;      /* partials, queries per request, splits per request   */
  const uint16_t *o;  /* bf16 [P, S, H, 512]                                 */
  int64_t o_sp, o_st, o_sh;
  const float *lse;   /* f32 [P, S, H]; unused when P == 1                   */
  int64_t l_sp, l_st, l_sh;
  const void *w_v;    /* bf16 [H,128,512] (w_fmt 0) or u8 [H,128,256] (1)    */
  int64_t w_sh, w_sv;
  const uint8_t *w_scale; /* e8m0 [H,128,16], w_fmt 1 only                   */
  int64_t s_sh, s_sv;
  int w_fmt;
  const uint16_t *gate; /* bf16 [S, H*128] dense                            */
} orc_args;

float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);
float orc_e2m1_value(int code);
float orc_e8m0_value(int code);
int orc_e2m1_code(float y);
int orc_mx_scale_code(const uint16_t *blk);
void orc_mx_quant_block(const uint16_t *blk, uint8_t *codes, int *scale_code);
float orc_sane(float x);
int orc_partial_set(int t, int S, int P, int q, int spr, int *r0, int *n);
int orc_combine_latent(const orc_args *a, int t, int h, float *lat);
int orc_latent_bf16(const orc_args *a, int t, int h, uint16_t *latb);
int orc_row(const orc_args *a, int t, int h, uint16_t *seg);
int orc_rows(const orc_args *a, int n, const int *ts, const int *hs, uint16_t *segs);
int orc_mla_combine_uv(const orc_args *a, uint16_t *out);

/* stage_push (the DCP producer side) on one machine: every rank's attention
 * partials, each over all R*H global heads, packed into destination rank
 * dst's combine buffer, the LSE masked for empty requests and rows past the
 * batch. */
typedef struct {
  int S, H, R, q, dst;     /* tokens, heads per rank, ranks, queries per request, destination */
  const uint16_t *o;       /* bf16 [R, S, R*H, 512]: source rank r, token t, global head g */
  int64_t o_sr, o_st, o_sh;
  const float *lse;        /* f32 [R, S, R*H]                                 */
  int64_t l_sr, l_st, l_sh;
  const int32_t *seq_lens; /* int32 [R, S/q]: rank r's local KV length of request j at r*sl_sr + j */
  int64_t sl_sr;
  const int32_t *qsl;      /* int32 [S/q + 1]: query start locations; rows >= qsl[S/q] are past the batch */
} orc_pack_args;
/* cmb_o bf16 [R, S, H, 512] and cmb_lse f32 [R, S, H], dense.  Returns 0, or
 * -1 for invalid sizes. */
int orc_dcp_pack(const orc_pack_args *a, uint16_t *cmb_o, float *cmb_lse);

/* The partial producer: split-KV MLA decode attention in the absorbed form
 * (the page's M1c, whose partials the combine merges; its kernel is not on
 * the page, so this follows the plain definition -- see mla_oracle.c). */
typedef struct {
  int B, q, H, spr;        /* requests, queries per request (S = B*q), heads, splits per request */
  float scale;             /* softmax scale applied to q . k                  */
  const uint16_t *qv;      /* bf16 [S, H, 576]: latent query (512) then rope query (64) */
  int64_t q_st, q_sh;
  const uint16_t *kv;      /* bf16 [B, Lmax, 576]: latent (512) then rope key (64) per cached position */
  int64_t kv_sb, kv_sl;
  const int32_t *kv_len;   /* int32 [B]: cached positions of request b, its q new ones included */
} orc_attn_args;
/* o bf16 [spr, S, H, 512] and lse f32 [spr, S, H], dense (split r of token t
 * at [r, t, h]).  Returns 0, or -1 for invalid sizes. */
int orc_mla_attn_split(const orc_attn_args *a, uint16_t *o, float *lse);

/* Downstream: this rank's o_proj shard, out[t][j] = sum_k core[t][k] W[j][k]
 * (see mla_oracle.c).  out bf16 [S, Nout] dense. */
typedef struct {
  int S, K, Nout;          /* tokens, input width (H*128), output features      */
  const uint16_t *x;       /* bf16 [S, K] (core), row stride x_st               */
  int64_t x_st;
  const uint16_t *w;       /* bf16 [Nout, K], row stride w_sj                   */
  int64_t w_sj;
} orc_oproj_args;
int orc_o_proj(const orc_oproj_args *a, uint16_t *out);

#endif
