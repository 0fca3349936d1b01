/*
 * mla_oracle.c -- the CPU oracle for the MLA decode post-attention stage
 * (LSE combine -> W_UV up-projection -> gate).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file; only the tests, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Source of the definition: the vLLM API page
 * "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
 * (functions sane, combine_ranks, combine_splits, stage_combine, stage_uv,
 * wv_loads, mla_post, stage_push).  The module docstring and combine_ranks /
 * stage_combine state that the partials are merged with their LSE weights in
 * single precision, so the oracle computes in fp32, single-threaded, in a
 * fixed order:
 * partials in index order, K in ascending order, one rounding per operation
 * (this file is compiled with -ffp-contract=off so no multiply-add is fused).
 *
 * Readings taken where the page is silent:
 *  - LSE is a natural log: weights are exp2((lse - m) * log2(e)).
 *  - exp2 is the C library's exp2f; the reciprocal is a true division.
 *  - bf16 rounding is round-to-nearest-even.
 *  - The MX scale rule ("even_code" is not defined on the page) is the OCP
 *    MX v1.0 shared-exponent rule: code = floor(log2(amax)) - 2 + 127,
 *    clamped to [1, 254]; amax == 0 gives 1; a non-finite amax gives the
 *    E8M0 NaN code 255.  PARITY UNPINNED against the page's own (undefined)
 *    even_code variant.
 *  - E2M1 conversion is round-to-nearest, ties to the even code, saturating
 *    at 6; a value that rounds to magnitude 0 is stored as +0.
 *  - Element 2i of a packed E2M1 row sits in the low nibble of byte i.
 *  - Split layout is chosen by P: P == 1 passthrough (lse ignored),
 *    P == splits_per_request compact (every token merges 0..P-1),
 *    P == (S/q) * splits_per_request request-major (token t merges
 *    (t/q)*spr .. (t/q)*spr + spr - 1).
 *  - Output rows S <= t < S_out are zero.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "mla_oracle.h"

#define ORC_D 512 /* latent width (KVL) */
#define ORC_V 128 /* V head dim (VD)    */
#define ORC_BLK 32 /* MX block along K   */

/* ---- scalar formats ------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round an fp32 value to the nearest bf16, ties to even.  A bf16 keeps the
 * upper 16 bits of the fp32 pattern; the discarded lower half decides. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u); /* stay a quiet NaN */
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* E2M1 magnitudes by 3-bit code (OCP MX v1.0, FP4 E2M1). */
static const float orc_e2m1_grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float orc_e2m1_value(int code) {
  float m = orc_e2m1_grid[code & 7];
  return (code & 8) ? -m : m;
}

/* E8M0 scale: 2^(code - 127); code 255 is NaN. */
float orc_e8m0_value(int code) {
  if (code == 255) return NAN;
  return ldexpf(1.0f, code - 127);
}

/* Nearest E2M1 code to an already-scaled value y; ties go to the even code,
 * values past 6 saturate to 6 (the nearest grid point). */
int orc_e2m1_code(float y) {
  /* below 8 the distances are exact in double, so ties are real ties; from 6
   * up the nearest grid point is the largest one, 6 */
  double a = fabs((double)y);
  int best = 0;
  if (a >= 6.0) {
    best = 7;
  } else {
    double best_d = fabs(a - orc_e2m1_grid[0]);
    for (int c = 1; c < 8; ++c) {
      double d = fabs(a - orc_e2m1_grid[c]);
      if (d < best_d || (d == best_d && (c % 2 == 0))) {
        best = c;
        best_d = d;
      }
    }
  }
  if (best != 0 && signbit(y)) best |= 8;
  return best;
}

/* Shared scale code of one block of 32 bf16 values (page: stage_uv takes
 * amax over the bf16 patterns with the sign cleared, code >= 1). */
int orc_mx_scale_code(const uint16_t *blk) {
  uint16_t amax_bits = 0;
  for (int i = 0; i < ORC_BLK; ++i) {
    uint16_t m = (uint16_t)(blk[i] & 0x7FFFu);
    if (m > amax_bits) amax_bits = m;
  }
  float amax = orc_bf16_to_f32(amax_bits);
  if (!isfinite(amax)) return 255;
  if (amax == 0.0f) return 1;
  int e;
  frexpf(amax, &e); /* amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
  int code = (e - 1) - 2 + 127;
  if (code < 1) code = 1;
  if (code > 254) code = 254;
  return code;
}

/* Quantise one block of 32 bf16 values: scale code and 32 E2M1 codes. */
void orc_mx_quant_block(const uint16_t *blk, uint8_t *codes, int *scale_code) {
  int c = orc_mx_scale_code(blk);
  *scale_code = c;
  for (int i = 0; i < ORC_BLK; ++i) {
    if (c == 255) {
      codes[i] = 0;
      continue;
    }
    float y = ldexpf(orc_bf16_to_f32(blk[i]), 127 - c);
    codes[i] = (uint8_t)orc_e2m1_code(y);
  }
}

/* ---- step a1: sanitise ------------------------------------------------- */

/* page: sane -- NaN and +inf become -inf. */
float orc_sane(float x) {
  if (isnan(x) || x == INFINITY) return -INFINITY;
  return x;
}

/* ---- partial set by layout ------------------------------------------- */

/* Returns the layout: 0 passthrough, 1 compact, 2 request-major, -1 invalid.
 * On success *r0 / *n give token t's partials r0 .. r0 + n - 1. */
int orc_partial_set(int t, int S, int P, int q, int spr, int *r0, int *n) {
  if (P == 1) {
    *r0 = 0;
    *n = 1;
    return 0;
  }
  if (spr > 0 && P == spr) {
    *r0 = 0;
    *n = P;
    return 1;
  }
  if (q > 0 && spr > 0 && S % q == 0 && (int64_t)P == (int64_t)(S / q) * spr) {
    *r0 = (t / q) * spr;
    *n = spr;
    return 2;
  }
  return -1;
}

/* ---- steps a2-a3: weights and merge ---------------------------------- */

/* fp32 latents of token t, head h (before the bf16 rounding).  Returns the
 * layout code, or -1 for an invalid (P, q, spr) combination. */
int orc_combine_latent(const orc_args *a, int t, int h, float *lat) {
  int r0, n;
  int lay = orc_partial_set(t, a->S, a->P, a->q, a->spr, &r0, &n);
  if (lay < 0) return -1;
  if (lay == 0) {
    /* page: stage_combine without splits copies the o row as the latents */
    const uint16_t *row = a->o + (int64_t)t * a->o_st + (int64_t)h * a->o_sh;
    for (int d = 0; d < ORC_D; ++d) lat[d] = orc_bf16_to_f32(row[d]);
    return lay;
  }
  float ell[4096];
  float e[4096];
  if (n > 4096) return -1;
  /* a1 */
  for (int j = 0; j < n; ++j) {
    int r = r0 + j;
    ell[j] = orc_sane(a->lse[(int64_t)r * a->l_sp + (int64_t)t * a->l_st + (int64_t)h * a->l_sh]);
  }
  /* a2: m = max, an all -inf row shifts by 0 */
  float m = -INFINITY;
  for (int j = 0; j < n; ++j)
    if (ell[j] > m) m = ell[j];
  if (m == -INFINITY) m = 0.0f;
  const float log2e = 1.4426950408889634f;
  float Z = 0.0f;
  for (int j = 0; j < n; ++j) {
    e[j] = exp2f((ell[j] - m) * log2e);
    Z = Z + e[j];
  }
  float inv = (Z == 0.0f) ? 0.0f : 1.0f / Z;
  /* a3: weighted sum, zero-weight partials skipped (their o never read) */
  for (int d = 0; d < ORC_D; ++d) lat[d] = 0.0f;
  for (int j = 0; j < n; ++j) {
    float w = (e[j] == 0.0f) ? 0.0f : e[j] * inv;
    if (w == 0.0f) continue;
    const uint16_t *row =
        a->o + (int64_t)(r0 + j) * a->o_sp + (int64_t)t * a->o_st + (int64_t)h * a->o_sh;
    for (int d = 0; d < ORC_D; ++d) {
      float p = w * orc_bf16_to_f32(row[d]);
      lat[d] = lat[d] + p;
    }
  }
  return lay;
}

/* ---- steps a4-a7 for one (t, h) row ------------------------------------ */

/* W_V[h][v][k] as an exact fp32 value. */
static float orc_wv(const orc_args *a, int h, int v, int k) {
  if (a->w_fmt == 0) {
    const uint16_t *w = (const uint16_t *)a->w_v;
    return orc_bf16_to_f32(w[(int64_t)h * a->w_sh + (int64_t)v * a->w_sv + k]);
  }
  const uint8_t *w = (const uint8_t *)a->w_v;
  uint8_t byte = w[(int64_t)h * a->w_sh + (int64_t)v * a->w_sv + k / 2];
  int code = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  int sc = a->w_scale[(int64_t)h * a->s_sh + (int64_t)v * a->s_sv + k / ORC_BLK];
  return orc_e2m1_value(code) * orc_e8m0_value(sc);
}

/* One output row segment core[t, h*128 .. h*128+127] (bf16 patterns). */
int orc_row(const orc_args *a, int t, int h, uint16_t *seg) {
  if (t >= a->S) {
    for (int v = 0; v < ORC_V; ++v) seg[v] = 0;
    return 0;
  }
  float lat[ORC_D];
  if (orc_combine_latent(a, t, h, lat) < 0) return -1;
  /* a4: bf16 latents */
  uint16_t latb[ORC_D];
  for (int d = 0; d < ORC_D; ++d) latb[d] = orc_f32_to_bf16(lat[d]);
  /* a5 (MXFP4 only): latents to E2M1 + E8M0, then back to exact fp32 */
  float x[ORC_D];
  if (a->w_fmt == 0) {
    for (int d = 0; d < ORC_D; ++d) x[d] = orc_bf16_to_f32(latb[d]);
  } else {
    for (int b = 0; b < ORC_D / ORC_BLK; ++b) {
      uint8_t codes[ORC_BLK];
      int sc;
      orc_mx_quant_block(latb + b * ORC_BLK, codes, &sc);
      for (int i = 0; i < ORC_BLK; ++i)
        x[b * ORC_BLK + i] = orc_e2m1_value(codes[i]) * orc_e8m0_value(sc);
    }
  }
  /* a6 + a7 */
  for (int v = 0; v < ORC_V; ++v) {
    float acc = 0.0f;
    for (int k = 0; k < ORC_D; ++k) {
      float p = orc_wv(a, h, v, k) * x[k];
      acc = acc + p;
    }
    float accb = orc_bf16_to_f32(orc_f32_to_bf16(acc));
    float g = orc_bf16_to_f32(a->gate[(int64_t)t * a->H * ORC_V + (int64_t)h * ORC_V + v]);
    seg[v] = orc_f32_to_bf16(accb * g);
  }
  return 0;
}

/* ---- whole call ---------------------------------------------------------- */

int orc_mla_combine_uv(const orc_args *a, uint16_t *out) {
  if (a->S < 0 || a->S_out < a->S || a->H < 1 || a->P < 1) return -1;
  const int64_t W = (int64_t)a->H * ORC_V;
  for (int t = 0; t < a->S_out; ++t)
    for (int h = 0; h < a->H; ++h)
      if (orc_row(a, t, h, out + (int64_t)t * W + (int64_t)h * ORC_V) < 0) return -1;
  return 0;
}

int orc_rows(const orc_args *a, int n, const int *ts, const int *hs, uint16_t *segs) {
  for (int i = 0; i < n; ++i)
    if (orc_row(a, ts[i], hs[i], segs + (int64_t)i * ORC_V) < 0) return -1;
  return 0;
}

/* Exposed for the pins: the bf16 latents of (t, h) and, for MXFP4, their
 * codes (one byte per element) and block scale codes. */
int orc_latent_bf16(const orc_args *a, int t, int h, uint16_t *latb) {
  float lat[ORC_D];
  if (orc_combine_latent(a, t, h, lat) < 0) return -1;
  for (int d = 0; d < ORC_D; ++d) latb[d] = orc_f32_to_bf16(lat[d]);
  return 0;
}

/* ---- stage_push: the DCP producer side --------------------------------- */

/* The page's stage_push, for one destination rank: for every source rank r,
 * token t and head h of the destination, the row of global head dst*H + h is
 * copied unchanged; its LSE is copied bit for bit, or replaced by -inf when
 * rank r holds no KV of the token's request (seq_lens == 0) or the token lies
 * past the batch (t >= qsl[S/q]).  Loops in (r, t, h, d) order. */
int orc_dcp_pack(const orc_pack_args *a, uint16_t *cmb_o, float *cmb_lse) {
  if (a->S < 0 || a->H < 1 || a->R < 1 || a->q < 1 || a->dst < 0 || a->dst >= a->R) return -1;
  if (a->S % a->q) return -1;
  const int rows = a->S > 0 ? a->qsl[a->S / a->q] : 0;
  const uint32_t neg_inf = 0xFF800000u;
  for (int r = 0; r < a->R; ++r) {
    for (int t = 0; t < a->S; ++t) {
      const int empty = a->seq_lens[(int64_t)r * a->sl_sr + t / a->q] == 0 || t >= rows;
      for (int h = 0; h < a->H; ++h) {
        const int64_t g = (int64_t)a->dst * a->H + h;
        const uint16_t *src = a->o + (int64_t)r * a->o_sr + (int64_t)t * a->o_st + g * a->o_sh;
        uint16_t *dst = cmb_o + (((int64_t)r * a->S + t) * a->H + h) * ORC_D;
        for (int d = 0; d < ORC_D; ++d) dst[d] = src[d];
        uint32_t bits;
        memcpy(&bits, a->lse + (int64_t)r * a->l_sr + (int64_t)t * a->l_st + g * a->l_sh, 4);
        if (empty) bits = neg_inf;
        memcpy(cmb_lse + ((int64_t)r * a->S + t) * a->H + h, &bits, 4);
      }
    }
  }
  return 0;
}

/* ---- the partial producer: split-KV MLA decode attention ----------------
 *
 * The page names the producer of the split partials (M1c, mla_attn: o / lse
 * of dense [splits, S, 12, 512] bf16 / [splits, S, 12] f32) but does not
 * print it, so this is the plain definition of MLA decode attention in the
 * absorbed form, split over the KV positions (flash decoding).  Readings:
 *  - a query row is 576 wide: the latent query (512, W_UK already absorbed)
 *    then the rope query (64); a cached row is the latent (512) then the
 *    rope key (64); the score is scale * (q . row) over all 576, and the
 *    value is the row's latent (512) -- the o that the combine merges;
 *  - the q tokens of a request are its last q cached positions: token i of
 *    request b sees positions j < kv_len[b] - (q - 1 - i);
 *  - split r of request b covers positions [r C, (r + 1) C) with
 *    C = ceil(kv_len[b] / spr), cut to what the token sees; a split with no
 *    position has lse -inf and o 0;
 *  - lse is the natural log of sum_j exp(score_j).
 * Computed in double, one position at a time in ascending order; o is
 * rounded to fp32 then to bf16 (both to nearest even), lse to fp32. */
int orc_mla_attn_split(const orc_attn_args *a, uint16_t *o, float *lse) {
  if (a->B < 0 || a->q < 1 || a->H < 1 || a->spr < 1) return -1;
  const int S = a->B * a->q;
  const uint32_t neg_inf = 0xFF800000u;
  for (int b = 0; b < a->B; ++b) {
    const int L = a->kv_len[b];
    if (L < 0) return -1;
    const int C = (L + a->spr - 1) / a->spr;
    const uint16_t *kvb = a->kv + (int64_t)b * a->kv_sb;
    for (int i = 0; i < a->q; ++i) {
      const int t = b * a->q + i;
      int vis = L - (a->q - 1 - i);
      if (vis < 0) vis = 0;
      for (int h = 0; h < a->H; ++h) {
        const uint16_t *qr = a->qv + (int64_t)t * a->q_st + (int64_t)h * a->q_sh;
        for (int r = 0; r < a->spr; ++r) {
          const int j0 = r * C;
          const int j1 = (r + 1) * C < vis ? (r + 1) * C : vis;
          uint16_t *orow = o + (((int64_t)r * S + t) * a->H + h) * ORC_D;
          float *l = lse + ((int64_t)r * S + t) * a->H + h;
          if (j1 <= j0) {
            memset(orow, 0, ORC_D * sizeof *orow);
            memcpy(l, &neg_inf, 4);
            continue;
          }
          /* scores, their max, the sum of exp(score - max) */
          double m = -INFINITY;
          for (int j = j0; j < j1; ++j) {
            const uint16_t *kr = kvb + (int64_t)j * a->kv_sl;
            double s = 0.0;
            for (int k = 0; k < ORC_D + 64; ++k) s += (double)orc_bf16_to_f32(qr[k]) * (double)orc_bf16_to_f32(kr[k]);
            s *= (double)a->scale;
            if (s > m) m = s;
          }
          double sum = 0.0, acc[ORC_D];
          for (int d = 0; d < ORC_D; ++d) acc[d] = 0.0;
          for (int j = j0; j < j1; ++j) {
            const uint16_t *kr = kvb + (int64_t)j * a->kv_sl;
            double s = 0.0;
            for (int k = 0; k < ORC_D + 64; ++k) s += (double)orc_bf16_to_f32(qr[k]) * (double)orc_bf16_to_f32(kr[k]);
            const double p = exp(s * (double)a->scale - m);
            sum += p;
            for (int d = 0; d < ORC_D; ++d) acc[d] += p * (double)orc_bf16_to_f32(kr[d]);
          }
          for (int d = 0; d < ORC_D; ++d) orow[d] = orc_f32_to_bf16((float)(acc[d] / sum));
          *l = (float)(m + log(sum));
        }
      }
    }
  }
  return 0;
}

/* ---- downstream: the o_proj shard of this rank ---------------------------
 *
 * The page's stage ends at "o_proj's input" (core).  o_proj is a row-parallel
 * linear layer: this rank's shard multiplies its core row (H*128 wide) by its
 * slice of the weight, out[t][j] = sum_k core[t][k] * W[j][k] (W stored
 * [hidden, H*128] as a linear layer's weight), and the ranks' outputs are
 * summed by the tensor-parallel all-reduce (multi-GPU, not here).  Computed in
 * double, k ascending; out rounded to fp32 then to bf16. */
int orc_o_proj(const orc_oproj_args *a, uint16_t *out) {
  if (a->S < 0 || a->K < 1 || a->Nout < 1) return -1;
  for (int t = 0; t < a->S; ++t) {
    const uint16_t *x = a->x + (int64_t)t * a->x_st;
    for (int j = 0; j < a->Nout; ++j) {
      const uint16_t *w = a->w + (int64_t)j * a->w_sj;
      double acc = 0.0;
      for (int k = 0; k < a->K; ++k) acc += (double)orc_bf16_to_f32(x[k]) * (double)orc_bf16_to_f32(w[k]);
      out[(int64_t)t * a->Nout + j] = orc_f32_to_bf16((float)acc);
    }
  }
  return 0;
}
