// kernel_simt.cu -- CUDA-core kernel of the MLA decode post-attention stage.
//
// One CTA per (8-token tile, head); warp w owns token t0 + w.  It is the path
// for tiny token counts (where a 128-row tensor-core tile would be mostly
// empty) and for problems whose tokens merge more than 32 partials.
//
// Steps (vLLM page "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.
// mla_back"): sane + LSE weights (combine_ranks / combine_splits), the
// weighted merge in fp32 with zero-weight partials masked, bf16 latents
// (stage_combine), MXFP4 latent quantisation (stage_uv), W_UV against W_V[h]
// (stage_uv, wv_loads), bf16(acc) * gate -> core (stage_uv).
//
// The merge keeps one rounding per operation in partial order (separate
// multiply and add, sequential sum of the exponentials, correctly rounded
// reciprocal) so the bf16 latents match a straightforward fp32 evaluation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

constexpr int kSimtTok = 8;
constexpr int kSimtThreads = 256;

__global__ void __launch_bounds__(kSimtThreads) simt_kernel(const KParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int t0 = blockIdx.x * kSimtTok;
  const int W = p.H * kV;  // gate / out row width
  const int n = p.n_part;

  uint16_t *lat = reinterpret_cast<uint16_t *>(smem);                       // [8][512] bf16
  float *accs = reinterpret_cast<float *>(smem + kSimtTok * kD * 2);         // [8][128]
  float *wts = accs + kSimtTok * kV;                                         // [8][n]

  if (t0 >= p.S) {  // a tile of padded rows only: zero them
    for (int i = threadIdx.x; i < kSimtTok * kV / 4; i += kSimtThreads) {
      const int tk = i / (kV / 4), v4 = i % (kV / 4);
      const int t = t0 + tk;
      if (t < p.S_out)
        *reinterpret_cast<uint2 *>(p.out + (long long)t * W + h * kV + v4 * 4) = make_uint2(0, 0);
    }
    return;
  }

  // ---- combine: warp -> token --------------------------------------------
  {
    const int t = t0 + warp;
    uint4 *lrow = reinterpret_cast<uint4 *>(lat + warp * kD);
    if (t >= p.S) {
      lrow[lane] = make_uint4(0, 0, 0, 0);
      lrow[lane + 32] = make_uint4(0, 0, 0, 0);
    } else if (p.layout == kPassthrough) {
      const uint16_t *row = p.o + (long long)t * p.o_st + (long long)h * p.o_sh;
      uint4 a = __ldcs(reinterpret_cast<const uint4 *>(row) + lane);
      uint4 b = __ldcs(reinterpret_cast<const uint4 *>(row) + lane + 32);
      lrow[lane] = a;
      lrow[lane + 32] = b;
    } else {
      const int r0 = (p.layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
      float *wt = wts + warp * n;
      const float *lse_th = p.lse + (long long)t * p.l_st + (long long)h * p.l_sh;
      float m = __int_as_float(0xFF800000);
      for (int j = lane; j < n; j += 32) {
        const float x = sane(lse_th[(long long)(r0 + j) * p.l_sp]);
        wt[j] = x;
        m = fmaxf(m, x);
      }
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
      if (m == __int_as_float(0xFF800000)) m = 0.0f;
      for (int j = lane; j < n; j += 32) wt[j] = exp2f(__fmul_rn(__fsub_rn(wt[j], m), kLog2e));
      __syncwarp();
      float Z = 0.0f;
      if (lane == 0)
        for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, wt[j]);
      Z = __shfl_sync(0xffffffffu, Z, 0);
      const float inv = (Z == 0.0f) ? 0.0f : __frcp_rn(Z);
      for (int j = lane; j < n; j += 32) {
        const float e = wt[j];
        wt[j] = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
      }
      __syncwarp();
      float acc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
      const uint16_t *base = p.o + (long long)t * p.o_st + (long long)h * p.o_sh;
      for (int j0 = 0; j0 < n; j0 += 4) {
        uint4 v[4][2];
        float w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          w[k] = (j0 + k < n) ? wt[j0 + k] : 0.0f;
          if (w[k] != 0.0f) {
            const uint4 *row = reinterpret_cast<const uint4 *>(base + (long long)(r0 + j0 + k) * p.o_sp);
            v[k][0] = __ldcs(row + lane);
            v[k][1] = __ldcs(row + lane + 32);
          } else {
            v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (w[k] == 0.0f) continue;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t u[4] = {v[k][c].x, v[k][c].y, v[k][c].z, v[k][c].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[c * 8 + 2 * q] = __fadd_rn(acc[c * 8 + 2 * q], __fmul_rn(w[k], bf16_lo(u[q])));
              acc[c * 8 + 2 * q + 1] = __fadd_rn(acc[c * 8 + 2 * q + 1], __fmul_rn(w[k], bf16_hi(u[q])));
            }
          }
        }
      }
      lrow[lane] = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                              pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
      lrow[lane + 32] = make_uint4(pack_bf16(acc[8], acc[9]), pack_bf16(acc[10], acc[11]),
                                   pack_bf16(acc[12], acc[13]), pack_bf16(acc[14], acc[15]));
    }
    __syncwarp();
    // MXFP4: quantise the bf16 latents, keep the (exact) dequantised values.
    // Lane l holds elements 8l..8l+7 and 256+8l..; a 32-block spans 4 lanes.
    if (p.w_fmt == 1 && t < p.S) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint4 x = lrow[lane + 32 * c];
        uint32_t u[4] = {x.x, x.y, x.z, x.w};
        uint32_t am = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) am = max(am, max(u[q] & 0x7FFFu, (u[q] >> 16) & 0x7FFFu));
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const uint32_t sc = mx_scale_code(am);
        const float scale = e8m0_to_f32(sc), inv = e8m0_inverse(sc);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          u[q] = pack_bf16(mx_fake_quant(bf16_lo(u[q]), sc, scale, inv),
                           mx_fake_quant(bf16_hi(u[q]), sc, scale, inv));
        lrow[lane + 32 * c] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    }
  }
  __syncthreads();

  // ---- W_UV: warp -> 16 rows of W_V[h]; lane -> K chunks lane, lane+32 ----
  for (int vi = 0; vi < kV / 8; ++vi) {
    const int v = warp * (kV / 8) + vi;
    float wv[16];
    if (p.w_fmt == 0) {
      const uint4 *wrow = reinterpret_cast<const uint4 *>(
          static_cast<const uint16_t *>(p.w_v) + (long long)h * p.w_sh + (long long)v * p.w_sv);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 x = __ldg(wrow + lane + 32 * c);
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          wv[c * 8 + 2 * q] = bf16_lo(u[q]);
          wv[c * 8 + 2 * q + 1] = bf16_hi(u[q]);
        }
      }
    } else {
      const uint8_t *wrow =
          static_cast<const uint8_t *>(p.w_v) + (long long)h * p.w_sh + (long long)v * p.w_sv;
      const uint8_t *srow = p.w_scale + (long long)h * p.s_sh + (long long)v * p.s_sv;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int ch = lane + 32 * c;  // 8 elements = 4 bytes
        const uint32_t codes = __ldg(reinterpret_cast<const uint32_t *>(wrow) + ch);
        const float scale = e8m0_to_f32(__ldg(srow + (ch >> 2)));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t cd = (codes >> (4 * e)) & 0xFu;
          const float mag = e2m1_mag_value(cd & 7u) * scale;
          wv[c * 8 + e] = (cd & 8u) ? -mag : mag;
        }
      }
    }
#pragma unroll
    for (int tk = 0; tk < kSimtTok; ++tk) {
      const uint4 *lrow = reinterpret_cast<const uint4 *>(lat + tk * kD);
      float s = 0.0f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 x = lrow[lane + 32 * c];
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          s = fmaf(wv[c * 8 + 2 * q], bf16_lo(u[q]), s);
          s = fmaf(wv[c * 8 + 2 * q + 1], bf16_hi(u[q]), s);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) accs[tk * kV + v] = s;
    }
  }
  __syncthreads();

  // ---- gate + store: 4 consecutive outputs per thread ---------------------
  for (int i = threadIdx.x; i < kSimtTok * kV / 4; i += kSimtThreads) {
    const int tk = i / (kV / 4), v0 = (i % (kV / 4)) * 4;
    const int t = t0 + tk;
    if (t >= p.S_out) continue;
    uint2 res = make_uint2(0, 0);
    if (t < p.S) {
      const uint2 g = *reinterpret_cast<const uint2 *>(p.gate + (long long)t * W + h * kV + v0);
      const float *a = accs + tk * kV + v0;
      res.x = pack_bf16(round_bf16(a[0]) * bf16_lo(g.x), round_bf16(a[1]) * bf16_hi(g.x));
      res.y = pack_bf16(round_bf16(a[2]) * bf16_lo(g.y), round_bf16(a[3]) * bf16_hi(g.y));
    }
    *reinterpret_cast<uint2 *>(p.out + (long long)t * W + h * kV + v0) = res;
  }
}

size_t simt_smem_bytes(int n_part) {
  return (size_t)kSimtTok * kD * 2 + (size_t)kSimtTok * kV * 4 + (size_t)kSimtTok * n_part * 4;
}

cudaError_t launch_simt(const KParams &p, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes(p.n_part);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((p.S_out + kSimtTok - 1) / kSimtTok, p.H);
  simt_kernel<<<grid, kSimtThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
