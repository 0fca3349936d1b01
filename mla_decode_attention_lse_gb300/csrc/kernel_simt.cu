// kernel_simt.cu -- CUDA-core kernel of the MLA decode post-attention stage.
//
// One CTA per (8-token tile, head); warp w owns token t0 + w.  It is the path
// for problems whose tokens merge more than 32 partials (and for batches of
// more than 16 tokens on request; up to 16 tokens, the layout further below).
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

// ---- small batches: one CTA per (head, 16 V rows) ----------------------
//
// With a handful of tokens the tensor-core kernel's 128 x 16 GEMM is mostly
// empty and a whole W_V[h] goes through each of a few SMs.  Here the work of
// a head is spread over eight CTAs that each hold 16 rows of W_V[h] (16 KiB
// bf16 or 4 KiB of E2M1 codes, kept as fp32 and transposed, [512][16], so
// that the 16 threads of a token read consecutive words), merge the latents
// of every token of the batch (at most 16; the few partial rows are read
// again by each of the eight CTAs, from L2), and compute the 16 x S dot
// products on the CUDA cores: thread (token t, row v) sums four interleaved
// K chains in order (k = 4i + c), one rounding per multiply and per add, and
// adds the four chains at the end.  The weights, the merge and the MXFP4
// rounding are those of the kernel above.  W_V's rows are a weight (no
// earlier kernel writes them): they are loaded before the wait for the
// previous kernel on the stream (programmatic dependent launch).
//
// Measured against the tensor-core kernel (CUDA graph of 1000 launches over
// rotated inputs, one GB300, us per launch): 1 token x 12 heads 3.93 vs 4.01;
// the 4-token split case (2 heads, 4 request-major partials) 5.04 vs 4.12
// (the 8-token CUDA-core layout above: 27.7); 8 tokens x 12 heads x 16
// splits 9.87 vs 6.69; 16 tokens 17.1 vs 6.2.  The tensor-core kernel's
// floor at these sizes is its launch and its round trips, which this layout
// shares, while its dot products grow with the tokens: the automatic choice
// keeps the tensor cores, and this layout serves explicit requests.

constexpr int kSmallVR = 16;  // V rows per CTA
constexpr int kSmallMaxS = 16;
constexpr int kSmallLat = kD + 4;  // a latent row in shared memory (padded: two tokens, two banks)

__global__ void __launch_bounds__(kSimtThreads) simt_small_kernel(const KParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  float *wt = reinterpret_cast<float *>(smem);                // [512][16]: W_V rows vb*16.., transposed
  float *lat = wt + kD * kSmallVR;                            // [16][kSmallLat]: latents (bf16 or E2M1 values)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x / (kV / kSmallVR), vb = blockIdx.x % (kV / kSmallVR);
  const int W = p.H * kV;
  const int n = p.n_part;
  grid_launch_dependents();

  // ---- W_V[h] rows vb*16 .. vb*16+15 -> wt[k][r] (exact fp32) ----
  if (p.w_fmt == 0) {
    for (int i = threadIdx.x; i < kSmallVR * 64; i += kSimtThreads) {
      const int r = i & 15, c = i >> 4;  // row, 16-byte chunk (8 elements): lanes write consecutive words
      const uint4 x = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.w_v) + (long long)h * p.w_sh +
                                                            (long long)(vb * kSmallVR + r) * p.w_sv) + c);
      const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wt[(8 * c + 2 * q) * kSmallVR + r] = bf16_lo(u[q]);
        wt[(8 * c + 2 * q + 1) * kSmallVR + r] = bf16_hi(u[q]);
      }
    }
  } else {
    for (int i = threadIdx.x; i < kSmallVR * 64; i += kSimtThreads) {
      const int r = i & 15, c = i >> 4;  // row, 4-byte group (8 elements)
      const int v = vb * kSmallVR + r;
      const uint32_t codes = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(p.w_v) +
                                                                     (long long)h * p.w_sh + (long long)v * p.w_sv) + c);
      const float scale = e8m0_to_f32(__ldg(p.w_scale + (long long)h * p.s_sh + (long long)v * p.s_sv + (c >> 2)));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t cd = (codes >> (4 * e)) & 0xFu;
        const float mag = e2m1_mag_value(cd & 7u) * scale;
        wt[(8 * c + e) * kSmallVR + r] = (cd & 8u) ? -mag : mag;
      }
    }
  }
  grid_dependency_wait();

  // ---- latents: warp w merges tokens w and w + 8 ----
  for (int tk = warp; tk < kSmallMaxS; tk += kSimtThreads / 32) {
    float *lrow = lat + tk * kSmallLat;  // element 8 lane + e, and 256 + 8 lane + e
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
    if (tk < p.S && p.layout == kPassthrough) {
      const uint16_t *row = p.o + (long long)tk * p.o_st + (long long)h * p.o_sh;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 x = __ldcs(reinterpret_cast<const uint4 *>(row) + lane + 32 * c);
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[c * 8 + 2 * q] = bf16_lo(u[q]);
          acc[c * 8 + 2 * q + 1] = bf16_hi(u[q]);
        }
      }
    } else if (tk < p.S) {
      const int r0 = (p.layout == kRequestMajor) ? (tk / p.q) * p.spr : 0;
      // one lane per partial (n <= 32): sane, max, exponentials, sum in order
      float x = __int_as_float(0xFF800000);
      if (lane < n) x = sane(p.lse[(long long)(r0 + lane) * p.l_sp + (long long)tk * p.l_st + (long long)h * p.l_sh]);
      float m = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (m == __int_as_float(0xFF800000)) m = 0.0f;
      const float e = (lane < n) ? exp2f(__fmul_rn(__fsub_rn(x, m), kLog2e)) : 0.0f;
      float Z = 0.0f;
      for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, j));
      const float inv = (Z == 0.0f) ? 0.0f : __frcp_rn(Z);
      const float wl = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
      const uint16_t *base = p.o + (long long)tk * p.o_st + (long long)h * p.o_sh;
      for (int j0 = 0; j0 < n; j0 += 8) {
        uint4 v[8][2];
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          w[k] = __shfl_sync(0xffffffffu, wl, (j0 + k) & 31);  // 0 past n
          if (w[k] != 0.0f) {
            const uint4 *row = reinterpret_cast<const uint4 *>(base + (long long)(r0 + j0 + k) * p.o_sp);
            v[k][0] = __ldcs(row + lane);
            v[k][1] = __ldcs(row + lane + 32);
          } else {
            v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
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
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2) acc[e2] = round_bf16(acc[e2]);  // bf16 latents
    }
    if (p.w_fmt == 1 && tk < p.S) {
      // MXFP4: the block of 32 spans lanes 4g .. 4g + 3 (per half row)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t am = 0;
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) am = max(am, (__float_as_uint(acc[c * 8 + e2]) >> 16) & 0x7FFFu);
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const uint32_t sc = mx_scale_code(am);
        const float scale = e8m0_to_f32(sc), inv = e8m0_inverse(sc);
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) acc[c * 8 + e2] = mx_fake_quant(acc[c * 8 + e2], sc, scale, inv);
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e2 = 0; e2 < 8; ++e2) lrow[256 * c + 8 * lane + e2] = (tk < p.S) ? acc[c * 8 + e2] : 0.0f;
  }
  __syncthreads();

  // ---- thread (token t, row r): four K chains in order, then their sum ----
  const int t = threadIdx.x >> 4, r = threadIdx.x & 15;
  if (t < p.S) {
    float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float *lt = lat + t * kSmallLat;
#pragma unroll 4
    for (int k = 0; k < kD; k += 4) {
#pragma unroll
      for (int c = 0; c < 4; ++c) s4[c] = __fadd_rn(s4[c], __fmul_rn(wt[(k + c) * kSmallVR + r], lt[k + c]));
    }
    const float acc = __fadd_rn(__fadd_rn(s4[0], s4[1]), __fadd_rn(s4[2], s4[3]));
    const long long off = (long long)t * W + h * kV + vb * kSmallVR + r;
    const float g = bf16_lo((uint32_t)p.gate[off]);
    const __nv_bfloat16 y = __float2bfloat16_rn(round_bf16(acc) * g);  // exact product, one rounding
    p.out[off] = *reinterpret_cast<const uint16_t *>(&y);
  }
  // rows S .. S_out - 1 of core are zero (this CTA's slice of them)
  const long long n8 = (long long)(p.S_out - p.S) * W / 8;
  if (n8 > 0) {
    const long long zb = (long long)blockIdx.x * n8 / gridDim.x;
    const long long ze = (long long)(blockIdx.x + 1) * n8 / gridDim.x;
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (long long)p.S * W);
    for (long long k = zb + threadIdx.x; k < ze; k += kSimtThreads) dst[k] = make_uint4(0, 0, 0, 0);
  }
}

bool simt_small_fits(int S, int n_part) { return S >= 1 && S <= kSmallMaxS && n_part <= 32; }
size_t simt_small_smem_bytes() { return (size_t)kD * kSmallVR * 4 + (size_t)kSmallMaxS * kSmallLat * 4; }
int simt_small_grid(int H) { return H * (kV / kSmallVR); }

cudaError_t launch_simt_small(const KParams &p, cudaStream_t stream) {
  const size_t smem = simt_small_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(simt_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)simt_small_grid(p.H), 1, 1);
  cfg.blockDim = dim3(kSimtThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, simt_small_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
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
