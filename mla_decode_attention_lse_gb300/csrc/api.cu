// api.cu -- the C ABI of libmla_combine_uv: validation, planning, dispatch.
//
// Host-side conventions follow the launcher of the vLLM page
// "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
// (host_args / mla_post): strided o / lse rows and heads with a unit-stride
// last dimension, dense gate / core, launch on the caller's stream, every
// check done before anything is launched.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "mla_combine_uv.h"
#include "kernel_oproj.h"
#include "kernels.h"

namespace {

using mla::KParams;

// Device-side error word, one per device context (first error wins).
__device__ int g_mla_err_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Validate and plan.  Pure host logic when num_sms > 0.
int32_t plan_impl(const mla_combine_uv_args *a, int32_t num_sms, mla_plan *pl, KParams *kp) {
  if (!a || !pl) return MLA_ERR_NULL;
  if (a->w_fmt != MLA_W_BF16 && a->w_fmt != MLA_W_MXFP4) return MLA_ERR_FMT;
  if (a->S < 0 || a->S_out < a->S || a->H < 1 || a->H > 65535 || a->P < 1 || a->q_per_request < 1 ||
      a->splits_per_request < 0)
    return MLA_ERR_SHAPE;
  if ((int64_t)a->S_out * a->H * 128 >= (int64_t)1 << 40) return MLA_ERR_SHAPE;
  if (a->wait_ns < 0) return MLA_ERR_SHAPE;

  // layout, chosen by P
  int layout, n_part;
  const int S = a->S, q = a->q_per_request, spr = a->splits_per_request;
  if (a->P == 1) {
    layout = mla::kPassthrough;
    n_part = 1;
  } else if (spr > 0 && a->P == spr) {
    layout = mla::kCompact;
    n_part = spr;
  } else if (spr > 0 && S % q == 0 && (int64_t)a->P == (int64_t)(S / q) * spr) {
    layout = mla::kRequestMajor;
    n_part = spr;
  } else {
    return MLA_ERR_LAYOUT;
  }

  // pointers (only those the call will touch)
  if (a->S_out > 0 && !a->out) return MLA_ERR_NULL;
  if (S > 0) {
    if (!a->o || !a->w_v || !a->gate) return MLA_ERR_NULL;
    if (a->P > 1 && !a->lse) return MLA_ERR_NULL;
    if (a->w_fmt == MLA_W_MXFP4 && !a->w_scale) return MLA_ERR_NULL;
    if (!aligned(a->o, 16) || !aligned(a->w_v, 16) || !aligned(a->gate, 16)) return MLA_ERR_ALIGN;
    if (a->lse && !aligned(a->lse, 4)) return MLA_ERR_ALIGN;
    // 16-byte vector rows of o; strides in elements
    if (a->o_st < 0 || a->o_sh < 0 || a->o_sp < 0) return MLA_ERR_STRIDE;
    if (a->o_st % 8 || a->o_sh % 8 || (a->P > 1 && a->o_sp % 8)) return MLA_ERR_STRIDE;
    if (a->P > 1 && (a->l_sp < 0 || a->l_st < 0 || a->l_sh < 0)) return MLA_ERR_STRIDE;
    if (a->w_sh < 0 || a->w_sv < 0) return MLA_ERR_STRIDE;
    if (a->w_fmt == MLA_W_BF16 && (a->w_sh % 8 || a->w_sv % 8)) return MLA_ERR_STRIDE;
    if (a->w_fmt == MLA_W_MXFP4 && (a->w_sh % 16 || a->w_sv % 16)) return MLA_ERR_STRIDE;
    if (a->w_fmt == MLA_W_MXFP4 && (a->s_sh < 0 || a->s_sv < 0)) return MLA_ERR_STRIDE;
  }
  if (a->S_out > 0 && !aligned(a->out, 16)) return MLA_ERR_ALIGN;

  // kernel choice
  int kernel = a->kernel;
  if (kernel != MLA_KERNEL_AUTO && kernel != MLA_KERNEL_SIMT && kernel != MLA_KERNEL_TC &&
      kernel != MLA_KERNEL_KSPLIT)
    return MLA_ERR_KERNEL;
  if (a->tile_tokens != 0 && a->tile_tokens != 8 && (a->tile_tokens < 16 || a->tile_tokens > 32))
    return MLA_ERR_KERNEL;
  if (kernel == MLA_KERNEL_TC && n_part > mla::kTcMaxPart) return MLA_ERR_KERNEL;
  if (kernel == MLA_KERNEL_KSPLIT && (n_part > mla::kKsMaxPart || S == 0 ||
                                      (a->tile_tokens != 0 && a->tile_tokens != 16)))
    return MLA_ERR_KERNEL;
  const int64_t units16 = (int64_t)a->H * ((S + 15) / 16);
  // the persistent tensor-core kernel whenever it can run it: even a single
  // token (a 16-token tile with empty rows) is faster than the CUDA-core
  // kernel, and with its prologue overlapping the previous launch it also
  // beats the cluster kernel at every decode size measured; the cluster
  // kernel runs on request only
  if (kernel == MLA_KERNEL_AUTO) kernel = (n_part <= mla::kTcMaxPart) ? MLA_KERNEL_TC : MLA_KERNEL_SIMT;
  if (S == 0) kernel = MLA_KERNEL_SIMT;  // nothing to merge: zero rows only
  const bool simt_small = mla::simt_small_fits(S, n_part);
  if (kernel == MLA_KERNEL_SIMT && !simt_small && mla::simt_smem_bytes(n_part) > 200 * 1024) return MLA_ERR_KERNEL;
  if (a->ready_flag && (kernel != MLA_KERNEL_TC || !aligned(a->ready_flag, 4))) return MLA_ERR_KERNEL;

  std::memset(pl, 0, sizeof *pl);
  pl->kernel = kernel;
  pl->layout = layout;
  pl->n_part = n_part;
  if (kernel == MLA_KERNEL_SIMT && simt_small) {
    // small batches: one CTA per (head, 16 V rows), every token of the batch
    pl->tile_tokens = S;
    pl->units = mla::simt_small_grid(a->H);
    pl->grid = pl->units;
    pl->threads = 256;
    pl->smem_bytes = (int32_t)mla::simt_small_smem_bytes();
  } else if (kernel == MLA_KERNEL_SIMT) {
    pl->tile_tokens = 8;
    pl->units = a->H * ((a->S_out + 7) / 8);
    pl->grid = pl->units;
    pl->threads = 256;
    pl->smem_bytes = (int32_t)mla::simt_smem_bytes(n_part);
  } else if (kernel == MLA_KERNEL_KSPLIT) {
    if ((int64_t)units16 * mla::ks_ctas_per_unit() >= ((int64_t)1 << 31)) return MLA_ERR_SHAPE;
    pl->tile_tokens = 16;
    pl->units = (int32_t)units16;
    pl->grid = pl->units * mla::ks_ctas_per_unit();
    pl->threads = mla::ks_threads();
    pl->smem_bytes = (int32_t)mla::ks_smem_bytes(a->w_fmt);
  } else {
    if (num_sms <= 0) return MLA_ERR_SHAPE;
    int tile = a->tile_tokens;
    // 32-token tiles once they give every SM a unit; with bf16 W_V and 16
    // or more partials per token, 8-token tiles (two warps per token, half a
    // row each) when those still fit one unit per SM and make more units than
    // 16-token tiles (a split-KV decode step: the partial rows spread over
    // twice the SMs; with one partial, as many CTAs each copying W_V measured
    // slower); else 16-token tiles (with MXFP4 W_V on two CTAs per SM).  More
    // than 16 partials per token need 8- or 16-token tiles.
    if (tile == 0) {
      const int64_t u8 = (int64_t)a->H * ((S + 7) / 8);
      // more 16-token units than SMs, too few 32-token ones to fill the GPU:
      // units of ut tokens (17..31, the 32-token kernel) so that each SM
      // takes exactly one (a stacked decode batch: 144 22-token units instead
      // of 192 16-token units, 40 SMs of which would run two)
      const int64_t tph = a->H <= num_sms ? num_sms / a->H : 0;
      const int64_t ut = tph > 0 ? (S + tph - 1) / tph : 0;
      if ((int64_t)a->H * ((S + 31) / 32) >= num_sms && n_part <= 16)
        tile = 32;
      else if (a->w_fmt == MLA_W_BF16 && n_part >= 16 && u8 <= num_sms && u8 > units16)
        tile = 8;
      else if (n_part <= 16 && units16 > num_sms && ut > 16 && ut < 32)
        tile = (int)ut;
      else
        tile = 16;
    }
    if (n_part > mla::tc_max_part(tile, a->w_fmt)) return MLA_ERR_KERNEL;
    pl->tile_tokens = tile;
    pl->units = a->H * ((S + tile - 1) / tile);
    const int slots = num_sms * mla::tc_ctas_per_sm(tile, a->w_fmt, n_part);
    pl->grid = pl->units < slots ? pl->units : slots;
    pl->threads = mla::tc_warps(tile, a->w_fmt, n_part) * 32;
    pl->smem_bytes = (int32_t)mla::tc_smem_bytes(tile, a->w_fmt, n_part);
  }

  // 32-bit offsets when the largest offset the kernels dereference fits
  // (terms are checked one by one, so nothing here can overflow)
  const int64_t lim = (int64_t)1 << 32;
  auto fits = [lim](int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t n2, int64_t s2, int64_t extra) {
    const int64_t n[3] = {n0, n1, n2}, st[3] = {s0, s1, s2};
    int64_t sum = extra;
    for (int i = 0; i < 3; ++i) {
      if (n[i] > 0 && st[i] >= lim) return false;
      sum += n[i] * st[i];  // < 2^31 * 2^32
      if (sum >= lim) return false;
    }
    return true;
  };
  const int64_t last_t = S > 0 ? S - 1 : 0;
  const bool o_ok = fits(a->P - 1, a->o_sp, last_t, a->o_st, a->H - 1, a->o_sh, 512);
  const bool l_ok = !a->lse || fits(a->P - 1, a->l_sp, last_t, a->l_st, a->H - 1, a->l_sh, 1);
  const bool g_ok = (int64_t)a->S_out * a->H * 128 < lim;
  pl->offsets32 = (o_ok && l_ok && g_ok) ? 1 : 0;

  if (kp) {
    KParams &k = *kp;
    std::memset(&k, 0, sizeof k);
    k.S = S;
    k.S_out = a->S_out;
    k.H = a->H;
    k.layout = layout;
    k.n_part = n_part;
    k.q = q;
    k.spr = spr;
    k.o = static_cast<const uint16_t *>(a->o);
    k.o_sp = a->o_sp;
    k.o_st = a->o_st;
    k.o_sh = a->o_sh;
    k.lse = a->lse;
    k.l_sp = a->l_sp;
    k.l_st = a->l_st;
    k.l_sh = a->l_sh;
    k.w_v = a->w_v;
    k.w_sh = a->w_sh;
    k.w_sv = a->w_sv;
    k.w_scale = a->w_scale;
    k.s_sh = a->s_sh;
    k.s_sv = a->s_sv;
    k.w_fmt = a->w_fmt;
    k.gate = static_cast<const uint16_t *>(a->gate);
    k.out = static_cast<uint16_t *>(a->out);
    k.tile = pl->tile_tokens;
    k.tiles_per_head = (kernel == MLA_KERNEL_SIMT) ? (a->S_out + 7) / 8 : (S + pl->tile_tokens - 1) / pl->tile_tokens;
    k.units = pl->units;
    k.off32 = pl->offsets32;
    k.wait_ns = a->wait_ns > 0 ? (unsigned long long)a->wait_ns : mla::kDefaultWaitNs;
    k.ready_flag = a->ready_flag;
  }
  return MLA_OK;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time
// dependency on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// TMA descriptor of the cache tensor [B, Lmax, 576] bf16: boxes of 64
// elements x box_rows positions (a tile of the attention kernel: 64 or 128)
// x 1 request with the 128-byte swizzle (the layout the tensor-core
// descriptors of the attention kernels read); positions past Lmax read as
// zero.
int32_t make_kv_tmap(const mla_attn_split_kv_args *a, int box_rows, CUtensorMap *tm) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return MLA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[3] = {576, (cuuint64_t)a->Lmax, (cuuint64_t)a->B};
  cuuint64_t strides[2] = {(cuuint64_t)a->kv_sl * 2, (cuuint64_t)a->kv_sb * 2};
  if (a->B == 1) strides[1] = (cuuint64_t)a->Lmax * (cuuint64_t)a->kv_sl * 2;  // unused dimension
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a->kv), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_STRIDE;
}

// TMA descriptor of W_V [H, 128, 512] bf16 (element strides w_sv, w_sh): boxes
// of 64 K elements x 128 V rows x 1 head with the 128-byte swizzle -- one K
// block of the [128 x 512] A tile of a head.
int32_t make_wv_tmap(const void *w_v, int H, int64_t w_sh, int64_t w_sv, CUtensorMap *tm) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return MLA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[3] = {512, 128, (cuuint64_t)H};
  cuuint64_t strides[2] = {(cuuint64_t)w_sv * 2, (cuuint64_t)(H > 1 ? w_sh : 128 * w_sv) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(w_v), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_STRIDE;
}

// TMA descriptor of a bf16 matrix [rows, cols] (row stride in elements) as
// a 3-D map with a unit third dimension: boxes of 64 columns x box_rows rows,
// 128-byte swizzle; rows past the matrix read as zero.
int32_t make_rows_tmap(const void *base, int64_t rows, int64_t cols, int64_t row_stride, int box_rows,
                       CUtensorMap *tm) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return MLA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2, (cuuint64_t)row_stride * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_STRIDE;
}

// Per-device state: SM count and the error word's device address.
int32_t device_state(int *dev_out, int *sms_out, int **err_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_mla_err_word) != cudaSuccess) return MLA_ERR_CUDA;
    g_num_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<int *>(ptr);
  }
  *dev_out = dev;
  *sms_out = g_num_sms[dev];
  *err_out = g_err_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" {

int32_t mla_abi_version(void) { return MLA_ABI_VERSION; }

const char *mla_status_str(int32_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_NULL: return "a required pointer is NULL";
    case MLA_ERR_SHAPE: return "invalid sizes";
    case MLA_ERR_STRIDE: return "a stride is not a multiple of 16 bytes or is negative";
    case MLA_ERR_ALIGN: return "a base pointer is not 16-byte aligned";
    case MLA_ERR_FMT: return "unknown W_V format";
    case MLA_ERR_LAYOUT: return "P matches neither passthrough, compact nor request-major layout";
    case MLA_ERR_CUDA: return "a CUDA call failed";
    case MLA_ERR_TIMEOUT: return "a kernel abandoned a bounded wait";
    case MLA_ERR_KERNEL: return "the requested kernel cannot run this problem";
    case MLA_ERR_DATA: return "a kernel met invalid device data (a kv_len outside [0, Lmax])";
    case MLA_ERR_SCRATCH: return "the problem needs more scratch than the library's fixed device buffer holds";
    default: return "unknown status";
  }
}

int32_t mla_combine_uv_plan(const mla_combine_uv_args *args, int32_t num_sms, mla_plan *plan) {
  if (num_sms <= 0) {
    int dev, sms;
    int *err;
    int32_t st = device_state(&dev, &sms, &err);
    if (st != MLA_OK) return st;
    num_sms = sms;
  }
  return plan_impl(args, num_sms, plan, nullptr);
}

int32_t mla_combine_uv(const mla_combine_uv_args *args, void *stream) {
  int dev, sms;
  int *err;
  int32_t st = device_state(&dev, &sms, &err);
  if (st != MLA_OK) return st;
  mla_plan pl;
  KParams kp;
  st = plan_impl(args, sms, &pl, &kp);
  if (st != MLA_OK) return st;
  if (args->S_out == 0) return MLA_OK;
  kp.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (pl.kernel == MLA_KERNEL_SIMT) {
    e = mla::simt_small_fits(kp.S, kp.n_part) ? mla::launch_simt_small(kp, s) : mla::launch_simt(kp, s);
  } else if (pl.kernel == MLA_KERNEL_KSPLIT) {
    e = mla::launch_ks(kp, s);
  } else {
    e = mla::launch_tc(kp, pl.grid, s);
  }
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_dcp_pack(const mla_dcp_pack_args *a, void *stream) {
  if (!a) return MLA_ERR_NULL;
  if (a->S < 0 || a->H < 1 || a->R < 1 || a->q_per_request < 1 || a->dst_rank < 0 || a->dst_rank >= a->R)
    return MLA_ERR_SHAPE;
  if (a->S % a->q_per_request) return MLA_ERR_SHAPE;
  if ((int64_t)a->R * a->H > 65535 || (int64_t)a->R * a->S * a->H * 512 >= ((int64_t)1 << 40)) return MLA_ERR_SHAPE;
  if (a->S == 0) return MLA_OK;
  if (!a->o || !a->lse || !a->seq_lens || !a->qsl || !a->cmb_o || !a->cmb_lse) return MLA_ERR_NULL;
  if (!aligned(a->o, 16) || !aligned(a->cmb_o, 16)) return MLA_ERR_ALIGN;
  if (!aligned(a->lse, 4) || !aligned(a->cmb_lse, 4) || !aligned(a->seq_lens, 4) || !aligned(a->qsl, 4))
    return MLA_ERR_ALIGN;
  if (a->o_sr < 0 || a->o_st < 0 || a->o_sh < 0 || a->o_sr % 8 || a->o_st % 8 || a->o_sh % 8) return MLA_ERR_STRIDE;
  if (a->l_sr < 0 || a->l_st < 0 || a->l_sh < 0 || a->sl_sr < 0) return MLA_ERR_STRIDE;
  int dev, sms;
  int *err;
  int32_t st = device_state(&dev, &sms, &err);
  if (st != MLA_OK) return st;
  mla::PackParams p;
  std::memset(&p, 0, sizeof p);
  p.S = a->S;
  p.H = a->H;
  p.R = a->R;
  p.q = a->q_per_request;
  p.dst = a->dst_rank;
  p.o = static_cast<const uint16_t *>(a->o);
  p.o_sr = a->o_sr;
  p.o_st = a->o_st;
  p.o_sh = a->o_sh;
  p.lse = a->lse;
  p.l_sr = a->l_sr;
  p.l_st = a->l_st;
  p.l_sh = a->l_sh;
  p.seq_lens = a->seq_lens;
  p.sl_sr = a->sl_sr;
  p.qsl = a->qsl;
  p.cmb_o = static_cast<uint16_t *>(a->cmb_o);
  p.cmb_lse = a->cmb_lse;
  const long long rows = (long long)a->R * a->S * a->H;
  const cudaError_t e = mla::launch_pack(p, mla::pack_grid(rows, sms), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_attn_split_kv(const mla_attn_split_kv_args *a, void *stream) {
  if (!a) return MLA_ERR_NULL;
  if (a->B < 0 || a->q < 1 || a->q > 32 || a->H < 1 || a->H > 65535 || a->spr < 1 || a->Lmax < 1 ||
      !std::isfinite(a->scale))
    return MLA_ERR_SHAPE;
  const int G = mla::attn_heads_per_cta(a->q, a->H);
  const int groups = (a->H + G - 1) / G;
  if ((int64_t)a->B * a->q >= ((int64_t)1 << 31) || (int64_t)a->B * a->spr * groups >= ((int64_t)1 << 31))
    return MLA_ERR_SHAPE;
  if (a->B == 0) return MLA_OK;
  if (!a->qv || !a->kv || !a->kv_len || !a->o || !a->lse) return MLA_ERR_NULL;
  if (!aligned(a->qv, 16) || !aligned(a->kv, 16) || !aligned(a->o, 16)) return MLA_ERR_ALIGN;
  if (!aligned(a->lse, 4) || !aligned(a->kv_len, 4)) return MLA_ERR_ALIGN;
  if (a->q_st < 0 || a->q_sh < 0 || a->q_st % 8 || a->q_sh % 8) return MLA_ERR_STRIDE;
  if (a->kv_sl < 576 || a->kv_sl % 8 || a->kv_sb < 0 || a->kv_sb % 8 || (a->B > 1 && a->kv_sb == 0))
    return MLA_ERR_STRIDE;
  if (a->kernel < 0 || a->kernel > 2) return MLA_ERR_KERNEL;
  CUtensorMap tm;
  const int rows = ((a->q * G + 15) / 16) * 16;
  int32_t st = make_kv_tmap(a, a->kernel == 2 ? 128 : mla::attn_tile_positions(rows, false), &tm);
  if (st != MLA_OK) return st;
  int dev, sms;
  int *err;
  st = device_state(&dev, &sms, &err);
  if (st != MLA_OK) return st;
  mla::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.B = a->B;
  p.q = a->q;
  p.H = a->H;
  p.spr = a->spr;
  p.G = G;
  p.groups = groups;
  p.Lmax = a->Lmax;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.qv = static_cast<const uint16_t *>(a->qv);
  p.q_st = a->q_st;
  p.q_sh = a->q_sh;
  p.kv_len = a->kv_len;
  p.o = static_cast<uint16_t *>(a->o);
  p.lse = a->lse;
  p.err = err;
  // one CTA per item unless the 2-CTA cluster kernel is asked for (measured
  // slower on the decode step: 135.9 against 87.6 us, its per-tile chain is
  // latency-bound and each SM pair walks twice the tiles)
  const cudaError_t e = a->kernel == 2 ? mla::launch_attn_pair(p, tm, sms, static_cast<cudaStream_t>(stream))
                                       : mla::launch_attn(p, tm, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int64_t mla_attn_combine_uv_workspace_words(int32_t B, int32_t q) {
  if (B < 0 || q < 1) return -1;
  return 3 + mla::attn_combine_tiles((int)std::min<int64_t>((int64_t)B * q, INT32_MAX));
}

int32_t mla_attn_combine_uv(const mla_attn_combine_uv_args *a, void *stream) {
  if (!a) return MLA_ERR_NULL;
  if (a->w_fmt != MLA_W_BF16 || a->w_scale) return MLA_ERR_FMT;  // bf16 W_V only
  if (a->B < 0 || a->q < 1 || a->q > 32 || a->H < 1 || a->H > 65535 || a->spr < 1 || a->spr > 32 || a->Lmax < 1 ||
      !std::isfinite(a->scale) || a->wait_ns < 0)
    return MLA_ERR_SHAPE;
  const int64_t S = (int64_t)a->B * a->q;
  if (S >= ((int64_t)1 << 31) || a->S_out < S || (int64_t)a->S_out * a->H * 128 >= ((int64_t)1 << 40))
    return MLA_ERR_SHAPE;
  const int G = mla::attn_heads_per_cta(a->q, a->H);
  const int groups = (a->H + G - 1) / G;
  const int ntiles = mla::attn_combine_tiles((int)S);
  // o_proj in the same launch: n_out outputs (a multiple of 64) of K = H*128 inputs
  const int64_t K = (int64_t)a->H * 128;
  const int64_t op_units = a->n_out > 0 ? (int64_t)(a->n_out / 64) * ((S + 63) / 64) : 0;
  if (a->n_out < 0 || a->n_out % 64 || (int64_t)a->n_out * K >= ((int64_t)1 << 40)) return MLA_ERR_SHAPE;
  if ((int64_t)a->B * a->spr * groups + (int64_t)ntiles * a->H + op_units >= ((int64_t)1 << 31)) return MLA_ERR_SHAPE;
  if (a->S_out > 0 && !a->out) return MLA_ERR_NULL;
  if (a->S_out > 0 && !aligned(a->out, 16)) return MLA_ERR_ALIGN;
  if (a->B > 0) {
    if (!a->qv || !a->kv || !a->kv_len || !a->part_o || !a->part_lse || !a->w_v || !a->gate || !a->workspace)
      return MLA_ERR_NULL;
    if (a->workspace_words < 3 + ntiles) return MLA_ERR_SHAPE;
    if (a->n_out > 0) {
      if (!a->w_o || !a->y) return MLA_ERR_NULL;
      if (!aligned(a->w_o, 16) || !aligned(a->y, 2)) return MLA_ERR_ALIGN;
      if (a->w_o_sj < K || a->w_o_sj % 8 || a->y_st < a->n_out) return MLA_ERR_STRIDE;
    }
    if (!aligned(a->qv, 16) || !aligned(a->kv, 16) || !aligned(a->part_o, 16) || !aligned(a->w_v, 16) ||
        !aligned(a->gate, 16))
      return MLA_ERR_ALIGN;
    if (!aligned(a->part_lse, 4) || !aligned(a->kv_len, 4) || !aligned(a->workspace, 4)) return MLA_ERR_ALIGN;
    if (a->q_st < 0 || a->q_sh < 0 || a->q_st % 8 || a->q_sh % 8) return MLA_ERR_STRIDE;
    if (a->kv_sl < 576 || a->kv_sl % 8 || a->kv_sb < 0 || a->kv_sb % 8 || (a->B > 1 && a->kv_sb == 0))
      return MLA_ERR_STRIDE;
    if (a->w_sv < 512 || a->w_sv % 8 || a->w_sh < 0 || a->w_sh % 8 || (a->H > 1 && a->w_sh == 0))
      return MLA_ERR_STRIDE;
  }
  int dev, sms;
  int *err;
  int32_t st = device_state(&dev, &sms, &err);
  if (st != MLA_OK) return st;
  if (a->B == 0) {
    if (a->S_out == 0) return MLA_OK;
    return cudaMemsetAsync(a->out, 0, (size_t)a->S_out * a->H * 128 * 2, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
  }
  mla_attn_split_kv_args aa;
  std::memset(&aa, 0, sizeof aa);
  aa.B = a->B;
  aa.q = a->q;
  aa.H = a->H;
  aa.spr = a->spr;
  aa.scale = a->scale;
  aa.qv = a->qv;
  aa.q_st = a->q_st;
  aa.q_sh = a->q_sh;
  aa.kv = a->kv;
  aa.kv_sb = a->kv_sb;
  aa.kv_sl = a->kv_sl;
  aa.Lmax = a->Lmax;
  CUtensorMap tm, wm, om, xm;
  st = make_kv_tmap(&aa, mla::attn_tile_positions(((a->q * G + 15) / 16) * 16, true), &tm);
  if (st != MLA_OK) return st;
  st = make_wv_tmap(a->w_v, a->H, a->w_sh, a->w_sv, &wm);
  if (st != MLA_OK) return st;
  std::memset(&om, 0, sizeof om);
  std::memset(&xm, 0, sizeof xm);
  if (a->n_out > 0) {
    st = make_rows_tmap(a->w_o, a->n_out, K, a->w_o_sj, 64, &om);  // W_o [n_out, K]
    if (st != MLA_OK) return st;
    st = make_rows_tmap(a->out, S, K, K, 64, &xm);  // core rows 0 .. S - 1 (later rows read as zero)
    if (st != MLA_OK) return st;
  }
  mla::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.B = a->B;
  p.q = a->q;
  p.H = a->H;
  p.spr = a->spr;
  p.G = G;
  p.groups = groups;
  p.Lmax = a->Lmax;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.qv = static_cast<const uint16_t *>(a->qv);
  p.q_st = a->q_st;
  p.q_sh = a->q_sh;
  p.kv_len = a->kv_len;
  p.o = static_cast<uint16_t *>(a->part_o);
  p.lse = a->part_lse;
  p.err = err;
  p.ws = a->workspace;
  p.ntiles = ntiles;
  p.S_out = a->S_out;
  p.gate = static_cast<const uint16_t *>(a->gate);
  p.out = static_cast<uint16_t *>(a->out);
  p.wait_ns = a->wait_ns > 0 ? (unsigned long long)a->wait_ns : mla::kDefaultWaitNs;
  p.n_out = a->n_out;
  p.op_units = (int)op_units;
  p.y = static_cast<uint16_t *>(a->y);
  p.y_st = a->y_st;
  const cudaError_t e = mla::launch_attn_combine(p, tm, wm, om, xm, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_o_proj(const mla_o_proj_args *a, void *stream) {
  if (!a) return MLA_ERR_NULL;
  if (a->S < 0 || a->K < 64 || a->K % 64 || a->Nout < 64 || a->Nout % 64) return MLA_ERR_SHAPE;
  if (a->S == 0) return MLA_OK;
  if (!a->x || !a->w || !a->out) return MLA_ERR_NULL;
  if (!aligned(a->x, 16) || !aligned(a->w, 16) || !aligned(a->out, 2)) return MLA_ERR_ALIGN;
  if (a->x_st < a->K || a->x_st % 8 || a->w_sj < a->K || a->w_sj % 8 || a->out_st < a->Nout) return MLA_ERR_STRIDE;
  const int nt = mla::oproj_tokens_per_unit(a->S);
  CUtensorMap wm, xm;
  int32_t st = make_rows_tmap(a->w, a->Nout, a->K, a->w_sj, 64, &wm);
  if (st != MLA_OK) return st;
  st = make_rows_tmap(a->x, a->S, a->K, a->x_st, nt, &xm);
  if (st != MLA_OK) return st;
  int dev, sms;
  int *err;
  st = device_state(&dev, &sms, &err);
  if (st != MLA_OK) return st;
  mla::OprojParams p;
  std::memset(&p, 0, sizeof p);
  p.S = a->S;
  p.K = a->K;
  p.Nout = a->Nout;
  p.nt = nt;
  p.out = static_cast<uint16_t *>(a->out);
  p.out_st = a->out_st;
  p.err = err;
  const cudaError_t e = mla::launch_oproj(p, wm, xm, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_combine_uv_status(void *stream) {
  int dev, sms;
  int *err;
  int32_t st = device_state(&dev, &sms, &err);
  if (st != MLA_OK) return st;
  // read and clear in order on the caller's stream (the word itself is one per
  // device, shared by every stream)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(err, 0, sizeof word, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    return word == mla::kErrKvLen ? MLA_ERR_DATA : MLA_ERR_TIMEOUT;
  }
  return MLA_OK;
}

}  // extern "C"
