// kernel_ks.cu -- the fused kernel for decode-sized batches: one (head,
// 16-token tile) unit per 4-CTA thread-block cluster, the 512-wide latent
// (K) dimension split over the cluster.
//
// With few units (a decode step of S = 64 tokens and 12 heads is 48 units of
// 16 tokens) the persistent kernel leaves most SMs idle, and each working SM
// pulls its whole W_V[h] (128 KiB bf16) and every partial row alone.  Here
// CTA r of a cluster owns latents [128 r, 128 r + 128): it reads that 256-byte
// slice of every partial row of the tile, the matching quarter of W_V[h],
// merges and rounds (or quantises) its slice, and runs a K = 128 tcgen05 GEMM
// into its own TMEM accumulator D_r[v, t] (M = 128 V rows, N = 16 tokens).
// The four partial accumulators meet through distributed shared memory: CTA
// q receives the V rows 32 q .. 32 q + 31 of every other CTA's D_r by
// st.async (completing on an mbarrier of q), adds the four in rank order, and
// runs the gate epilogue for those rows.  Rows, W_V and the epilogue are thus
// spread over four times as many SMs, and nothing outside the caller's
// buffers is written.
//
// Semantics are those of the vLLM page "vllm.models.kimi_k3.amd.
// specialized_decode.mono.attention.mla_back": combine_splits (sane, LSE
// weights, zero-weight partials skipped), stage_combine (bf16 latents, one
// partial passes through, padded rows zero), stage_uv (MXFP4 latents per
// 32-element K block, W_UV, bf16(acc) * gate).  Each 32-element MX block lies
// inside one CTA's slice, so the quantisation is unchanged by the split; only
// the GEMM's fp32 summation order differs (four K = 128 partial sums, added
// in rank order).  Every wait is bounded; on timeout the kernel records an
// error, still meets its cluster peers at the closing cluster barrier, frees
// TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kKs = 4;                    // CTAs per cluster = K slices
constexpr int kKsBN = 16;                 // tokens per unit
constexpr int kKsWarps = 8;               // two tokens per warp
constexpr int kKsThreads = kKsWarps * 32;
constexpr int kKsK = kD / kKs;            // latents per CTA (128)
constexpr uint32_t kKsSlot = 32u * kKsBN * 4u;  // one peer's V quadrant: 32 rows x 16 tokens fp32

// Shared memory of one CTA (offsets from a 1024-byte aligned base).
struct KsLayout {
  uint32_t b_off, sfa_off, sfb_off, recv_off, bar_off, total, tmem_cols;
};
__host__ __device__ constexpr KsLayout ks_layout(int WFMT) {
  KsLayout L{};
  // A: the W_V slice, K-major with the 128-byte swizzle: bf16 two K blocks of
  // [128 rows x 128 B]; MXFP4 one [128 x 128 B] block, 64 B of codes per row
  L.b_off = WFMT ? 128u * 128u : 2u * 128u * 128u;
  // B: the latent slice: bf16 two K blocks of [16 x 128 B]; MXFP4 one block
  L.sfa_off = L.b_off + (WFMT ? 16u * 128u : 2u * 16u * 128u);
  L.sfb_off = L.sfa_off + 512u;  // MXFP4 scale atoms (32 lines x 16 B each)
  L.recv_off = L.sfb_off + 512u;
  L.bar_off = L.recv_off + kKs * kKsSlot;  // slot of each peer rank (own slot unused)
  L.total = L.bar_off + 64u;
  // TMEM: accumulator columns 0..15; MXFP4 scales at columns 16 (W_V) and 32 (latents)
  L.tmem_cols = WFMT ? 64u : 32u;
  return L;
}

template <int WFMT>
__global__ void __launch_bounds__(kKsThreads, 2) ks_kernel(const __grid_constant__ KParams p) {
  constexpr KsLayout L = ks_layout(WFMT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t sA = sbase, sB = sbase + L.b_off;
  uint8_t *gB = gbase + L.b_off;
  uint8_t *gSFA = gbase + L.sfa_off;
  uint8_t *gSFB = gbase + L.sfb_off;
  const float *recv = reinterpret_cast<const float *>(gbase + L.recv_off);
  uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + L.bar_off);
  uint32_t *misc = reinterpret_cast<uint32_t *>(bars + 2);  // misc[0]: TMEM base
  const uint32_t bar_mma = smem_u32(&bars[0]), bar_recv = smem_u32(&bars[1]);
  const float kNegInf = __int_as_float(0xFF800000);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int unit = (int)cluster_id_x();
  const int h = unit / p.tiles_per_head, tile = unit - h * p.tiles_per_head;
  const int Wrow = p.H * kV;

  if (threadIdx.x == 0) {
    mbar_init(bar_mma, 1u);
    mbar_init(bar_recv, 1u);
    // the three peers' quadrants; the phase completes when all have landed
    mbar_arrive_expect_tx(bar_recv, (uint32_t)(kKs - 1) * kKsSlot);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc[0]), L.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // every CTA's barriers exist before a peer signals them
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // the next launch on the stream may start its own prologue now; its
  // token-dependent work still waits for this grid to complete
  grid_launch_dependents();

  auto load_wv_slice = [&]() {
    if (WFMT == 0) {
      // bf16 slice: 128 rows x 256 B, 16-byte chunk c of row v to K block c / 8
      const uint16_t *wb = static_cast<const uint16_t *>(p.w_v) + (long long)h * p.w_sh + (int)rank * kKsK;
      for (int s = threadIdx.x; s < kV * 16; s += kKsThreads) {
        const int v = s >> 4, c = s & 15;
        cp_async_16(sA + (uint32_t)(c >> 3) * (kV * 128u) + (uint32_t)v * 128u + (uint32_t)(((c & 7) ^ (v & 7)) << 4),
                    wb + (long long)v * p.w_sv + 8 * c);
      }
    } else {
      // MXFP4 slice: 128 rows x 64 B of codes, and the four scales of K blocks
      // 4 rank .. 4 rank + 3 of row v -> atom line v % 32, word v / 32
      const uint8_t *wb = static_cast<const uint8_t *>(p.w_v) + (long long)h * p.w_sh + (int)rank * (kKsK / 2);
      for (int s = threadIdx.x; s < kV * 4; s += kKsThreads) {
        const int v = s >> 2, c = s & 3;
        cp_async_16(sA + (uint32_t)v * 128u + (uint32_t)((c ^ (v & 7)) << 4), wb + (long long)v * p.w_sv + 16 * c);
      }
      const uint8_t *sb = p.w_scale + (long long)h * p.s_sh + 4 * (int)rank;
      const bool al4 = ((reinterpret_cast<uintptr_t>(sb) | (uintptr_t)p.s_sv) & 3u) == 0;
      for (int v = threadIdx.x; v < kV; v += kKsThreads) {
        const uint8_t *sr = sb + (long long)v * p.s_sv;
        uint8_t *dst = gSFA + (v & 31) * 16 + (v >> 5) * 4;
        if (al4) {
          cp_async_4(smem_u32(dst), sr);
        } else {
          *reinterpret_cast<uint32_t *>(dst) = (uint32_t)__ldg(sr) | ((uint32_t)__ldg(sr + 1) << 8) |
                                               ((uint32_t)__ldg(sr + 2) << 16) | ((uint32_t)__ldg(sr + 3) << 24);
        }
      }
    }
    cp_async_commit();
  };

  // ---- W_V's slice (a weight: no earlier kernel writes it), then, once the
  // previous grid on the stream is complete, the token-dependent loads ----
  load_wv_slice();
  grid_dependency_wait();
  const int n = p.n_part;
  const bool pass = (p.layout == kPassthrough);
  const int tl = 2 * warp + (lane >> 4);  // token within the tile
  const int l16 = lane & 15;              // 8 latents 8 l16 .. 8 l16 + 7 of the slice
  const int t = tile * kKsBN + tl;
  const bool tv = t < p.S;
  const int r0 = (p.layout == kRequestMajor && tv) ? (t / p.q) * p.spr : 0;
  float lv = kNegInf;  // LSE of (token t, partial l16)
  if (!pass && tv && l16 < n)
    lv = __ldg(p.lse + (long long)(r0 + l16) * p.l_sp + (long long)t * p.l_st + (long long)h * p.l_sh);
  // every partial's slice, issued before the weights are known (rows that
  // turn out dead are loaded but never merged)
  const uint16_t *ob = p.o + (long long)t * p.o_st + (long long)h * p.o_sh + (long long)r0 * p.o_sp +
                       (int)rank * kKsK + 8 * l16;
  uint4 rows[kKsMaxPart];
#pragma unroll
  for (int j = 0; j < kKsMaxPart; ++j) {
    if (j < n && tv) {
      rows[j] = __ldcs(reinterpret_cast<const uint4 *>(ob + (long long)j * p.o_sp));
    } else {
      rows[j] = make_uint4(0, 0, 0, 0);
    }
  }
  // the gate values of the V rows this CTA finishes (warps of lane quadrant
  // q == rank; tokens 8 ch .. 8 ch + 7), loaded now so that their round trip
  // overlaps everything up to the epilogue
  const int q = warp & 3, ch = warp >> 2;
  const bool owner = (q == (int)rank);
  const int v = (int)rank * 32 + lane;
  uint16_t gv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int te = tile * kKsBN + 8 * ch + e;
    gv[e] = (owner && te < p.S) ? p.gate[(long long)te * Wrow + h * kV + v] : (uint16_t)0;
  }

  // ---- weights: lane (token tl, partial l16); 16 lanes per token ----
  float wg;
  if (pass) {
    wg = (l16 == 0) ? 1.0f : 0.0f;
  } else {
    int np2 = 1;  // n rounded up to a power of two (<= 16)
    while (np2 < n) np2 <<= 1;
    const float l = sane(lv);
    float m = l;
    for (int s = 1; s < np2; s <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    if (m == kNegInf) m = 0.0f;
    const float e = (l16 < n) ? ex2_approx(__fmul_rn(__fsub_rn(l, m), kLog2e)) : 0.0f;
    float Z = 0.0f;  // sequential fp32 sum in partial order
    for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, (lane & 16) + j));
    const float inv = (Z == 0.0f) ? 0.0f : rcp_approx(Z);
    wg = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
  }

  // ---- merge in partial order, one rounding per multiply and per add ----
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < kKsMaxPart; ++j) {
    if (j < n) {
      const float w = __shfl_sync(0xffffffffu, wg, (lane & 16) + j);
      if (w != 0.0f && tv) {
        const uint64_t w2 = f2_pack(w, w);
        const uint32_t uu[4] = {rows[j].x, rows[j].y, rows[j].z, rows[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = f2_add(acc[q], f2_mul(w2, f2_pack(bf16_lo(uu[q]), bf16_hi(uu[q]))));
      }
    }
  }
  uint4 x;
  if (pass) {
    x = rows[0];  // one partial: the o row is the latent
  } else {
    uint32_t pk[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float lo, hi;
      f2_unpack(acc[q], lo, hi);
      pk[q] = pack_bf16(lo, hi);
    }
    x = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }

  // ---- latents into the B tile (bf16, or E2M1 codes + E8M0 scales) ----
  if (WFMT == 0) {
    if (!tv) x = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4 *>(gB + (l16 >> 3) * (kKsBN * 128) + tl * 128 + (((l16 & 7) ^ (tl & 7)) << 4)) = x;
  } else {
    uint32_t sc;
    uint32_t w = mx_codes(x, sc);  // K block l16 / 4 of the slice
    if (!tv) {
      w = 0u;
      sc = 127u;
    }
    *reinterpret_cast<uint32_t *>(gB + tl * 128 + (((l16 >> 2) ^ (tl & 7)) << 4) + 4 * (l16 & 3)) = w;
    if ((l16 & 3) == 0) gSFB[tl * 16 + (l16 >> 2)] = (uint8_t)sc;
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  __syncthreads();

  // ---- the slice's GEMM: D_r[v, t] = sum over the slice of W_V[h][v][k] lat[t][k] ----
  if (threadIdx.x == 0) {
    tc_fence_after();
    const uint32_t dA = (uint32_t)smem_desc_sw128(sA), dB = (uint32_t)smem_desc_sw128(sB);
    if (WFMT == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, kKsBN);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t kb = k >> 2, kk = k & 3;
        tc_mma_f16(tmem, desc_sw128_at(dA, kb * (kV * 128u) + kk * 32u), desc_sw128_at(dB, kb * (kKsBN * 128u) + kk * 32u),
                   kIdesc, k > 0 ? 1u : 0u);
      }
    } else {
      constexpr uint32_t kIdesc = idesc_mxf4(128, kKsBN);
      const uint32_t sfa = tmem + 16u, sfb = tmem + 32u;
      tc_cp_32x128b_warpx4(sfa, smem_desc_rows16(smem_u32(gSFA)));
      tc_cp_32x128b_warpx4(sfb, smem_desc_rows16(smem_u32(gSFB)));
#pragma unroll
      for (int k = 0; k < 2; ++k)  // K = 64 per step: scale bytes 2k, 2k + 1 of word 0
        tc_mma_mxf4(tmem, desc_sw128_at(dA, k * 32u), desc_sw128_at(dB, k * 32u), kIdesc | idesc_sf_ids(2u * k), sfa,
                    sfb, k > 0 ? 1u : 0u);
    }
    tc_commit(bar_mma);
  }

  // ---- exchange and epilogue: warp (quadrant q = warp % 4, tokens 8 ch .. 8 ch + 7) ----
  bool ok = mbar_wait(bar_mma, 0u, p.err, kErrWaitMma);
  ok = __all_sync(0xffffffffu, ok);
  uint32_t d[8];
  if (ok) {
    tc_fence_after();
    tmem_ld_x8(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(8 * ch), d);
    tc_wait_ld();
  }
  if (!owner) {
    if (ok) {
      // lane's V row 32 q + lane, tokens 8 ch .. 8 ch + 7 -> slot `rank` of CTA q
      const uint32_t dst = mapa_shared(smem_u32(recv) + rank * kKsSlot + (uint32_t)(lane * kKsBN + 8 * ch) * 4u, (uint32_t)q);
      const uint32_t rb = mapa_shared(bar_recv, (uint32_t)q);
      st_async_v4(dst, __uint_as_float(d[0]), __uint_as_float(d[1]), __uint_as_float(d[2]), __uint_as_float(d[3]), rb);
      st_async_v4(dst + 16u, __uint_as_float(d[4]), __uint_as_float(d[5]), __uint_as_float(d[6]), __uint_as_float(d[7]),
                  rb);
    }
  } else {
    bool ok2 = ok && mbar_wait(bar_recv, 0u, p.err, kErrWaitPeer);
    ok2 = __all_sync(0xffffffffu, ok2);
    if (ok2) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float s = 0.0f;
#pragma unroll
        for (int rr = 0; rr < kKs; ++rr) {  // the four K slices in rank order
          const float part = (rr == (int)rank) ? __uint_as_float(d[e]) : recv[rr * (kKsSlot / 4) + lane * kKsBN + 8 * ch + e];
          s = (rr == 0) ? part : __fadd_rn(s, part);
        }
        const int te = tile * kKsBN + 8 * ch + e;
        if (te < p.S) {
          const float a = round_bf16(s);
          const float g = __uint_as_float((uint32_t)gv[e] << 16);
          const __nv_bfloat16 o = __float2bfloat16_rn(__fmul_rn(a, g));
          p.out[(long long)te * Wrow + h * kV + v] = *reinterpret_cast<const uint16_t *>(&o);
        }
      }
    }
  }

  // rows S .. S_out-1 of core are zero (this CTA's slice of them)
  const long long n16 = (long long)(p.S_out - p.S) * p.H * (kV * 2 / 16);
  if (n16 > 0) {
    const long long zb = (long long)blockIdx.x * n16 / gridDim.x;
    const long long ze = (long long)(blockIdx.x + 1) * n16 / gridDim.x;
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (long long)p.S * Wrow);
    for (long long k = zb + threadIdx.x; k < ze; k += kKsThreads) dst[k] = make_uint4(0, 0, 0, 0);
  }

  // teardown: after a timed-out MMA wait, wait (bounded) once more so no MMA
  // still writes TMEM; meet the peers (none exits while another may still
  // store into its shared memory), then free TMEM
  if (threadIdx.x == 0 && !ok) mbar_wait(bar_mma, 0u, p.err, kErrWaitTeardown);
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L.tmem_cols);
  }
}

template <int WFMT>
cudaError_t launch_ks_one(const KParams &p, cudaStream_t stream) {
  const size_t smem = 1024 + ks_layout(WFMT).total;
  cudaError_t e = cudaFuncSetAttribute(ks_kernel<WFMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.units * kKs), 1, 1);
  cfg.blockDim = dim3(kKsThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kKs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: may begin while the previous kernel on the
  // stream finishes (the kernel waits for it before touching its outputs)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, ks_kernel<WFMT>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int ks_ctas_per_unit() { return kKs; }
int ks_threads() { return kKsThreads; }
size_t ks_smem_bytes(int w_fmt) { return 1024 + ks_layout(w_fmt ? 1 : 0).total; }

cudaError_t launch_ks(const KParams &p, cudaStream_t stream) {
  if (p.tile != kKsBN || p.n_part > kKsMaxPart || p.n_part < 1) return cudaErrorInvalidValue;
  return p.w_fmt ? launch_ks_one<1>(p, stream) : launch_ks_one<0>(p, stream);
}

}  // namespace mla
