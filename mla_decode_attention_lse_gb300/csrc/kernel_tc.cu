// kernel_tc.cu -- fused tensor-core kernel of the MLA decode post-attention
// stage for sm_103a: LSE combine -> (MXFP4) latents in shared memory ->
// tcgen05 W_UV GEMM with the accumulator in TMEM -> gate epilogue.
//
// Work unit: (head h, BN-token tile), head-major, split into one contiguous
// run per CTA (persistent grid of at most one CTA per SM), so a CTA keeps
// W_V[h] resident in shared memory across the token tiles of a head.
//
// GEMM orientation (per unit): D[v, t] = sum_k W_V[h][v][k] * lat[t][k] with
// M = 128 (the V rows), N = BN tokens, K = 512, both operands K-major with
// the 128-byte swizzle.  This keeps M at the tensor core's 128 while the
// token tile stays small enough for decode batches.
//
// Warp roles (288 threads):
//   warps 0-7  combine a unit's tokens (BN/8 each) into the latent buffer,
//              then run the epilogue of the previous unit (TMEM -> registers,
//              bf16(acc) * gate -> core);
//   warp 8     allocates TMEM, loads W_V[h] with TMA (bf16) and issues the
//              32 MMAs of a unit from one thread.
// Latent buffers and TMEM accumulators are double-buffered, so the combine of
// unit i overlaps the MMA of unit i-1 and the epilogue of unit i-2.
//
// Semantics follow the vLLM page "vllm.models.kimi_k3.amd.specialized_decode.
// mono.attention.mla_back": combine_ranks / combine_splits (sane, LSE weights,
// zero-weight partials masked), stage_combine (bf16 latents, passthrough for
// one partial, padded tokens zero), stage_uv (MXFP4 latents, W_UV, bf16(acc)
// * gate), combine_tasks / tasks (a persistent loop over (head, tokens)
// tasks).  Every mbarrier wait is bounded; on timeout the kernel records an
// error, drains its own in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr uint32_t kABytes = 128u * 1024u;  // W_V[h], bf16, 8 K-blocks x 16 KiB

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int *err, int code,
                                              volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitNs) {
      atomicCAS(err, 0, code);
      *abort_flag = 1;
      return false;
    }
  }
}

// Quantise a lane's 8 bf16 latents (one 16-byte chunk) to MXFP4 and return
// the dequantised values as bf16; the 32-element block spans lanes 4g..4g+3.
__device__ __forceinline__ uint4 mx_chunk(uint4 x) {
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
  return make_uint4(u[0], u[1], u[2], u[3]);
}

}  // namespace

template <int BN, int WFMT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tmap_w) {
  constexpr int TPW = BN / 8;                       // tokens per worker warp per unit
  constexpr uint32_t kBBytes = BN * 1024u;          // one latent buffer (BN x 512 bf16)
  constexpr uint32_t kCols = (2 * BN < 32) ? 32u : (uint32_t)(2 * BN);
  constexpr uint32_t kIdesc = idesc_bf16(128, BN);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;    // 1024-byte aligned (swizzle atoms)
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB0 = sbase + kABytes;
  uint8_t *gA = gbase;
  uint8_t *gB0 = gbase + kABytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + kABytes + 2 * kBBytes);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 8);
  volatile int *s_abort = reinterpret_cast<volatile int *>(bars + 8) + 1;
  const uint32_t bar_wv = smem_u32(&bars[0]);
  const uint32_t bar_lat0 = smem_u32(&bars[1]);  // +8*b
  const uint32_t bar_mma0 = smem_u32(&bars[3]);
  const uint32_t bar_acc0 = smem_u32(&bars[5]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar_wv, WFMT == 0 ? 1u : 8u);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_lat0 + 8 * b, 8u);
      mbar_init(bar_mma0 + 8 * b, 1u);
      mbar_init(bar_acc0 + 8 * b, 8u);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_holder), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int tph = p.tiles_per_head;
  const int ub = (int)((long long)blockIdx.x * p.units / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * p.units / gridDim.x);
  const int nu = ue - ub;
  const int Wrow = p.H * kV;

  if (warp == 8) {
    // ---------------- control: W_V loads and MMA issue ----------------
    if (lane == 0) {
      int prev_h = -1, last = -1;
      uint32_t wv_par = 0;
      bool tma_pending = false;
      for (int i = 0; i < nu; ++i) {
        if (*s_abort) break;
        const int u = ub + i, h = u / tph, b = i & 1;
        if (h != prev_h) {
          // every MMA reading the previous head's W_V must be done
          if (i > 0 &&
              !wait_or_abort(bar_mma0 + 8 * ((i - 1) & 1), ((i - 1) >> 1) & 1, p.err, kErrWaitMma, s_abort))
            break;
          if (WFMT == 0) {
            mbar_arrive_expect_tx(bar_wv, kABytes);
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) tma_load_3d(sA + kb * 16384u, &tmap_w, kb * 64, 0, h, bar_wv);
            tma_pending = true;
          }
          if (!wait_or_abort(bar_wv, wv_par, p.err, kErrWaitWv, s_abort)) break;
          tma_pending = false;
          wv_par ^= 1u;
          prev_h = h;
        }
        if (!wait_or_abort(bar_lat0 + 8 * b, (i >> 1) & 1, p.err, kErrWaitLatent, s_abort)) break;
        if (i >= 2 && !wait_or_abort(bar_acc0 + 8 * b, ((i - 2) >> 1) & 1, p.err, kErrWaitAccEmpty, s_abort))
          break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * BN);
        const uint32_t sB = sB0 + (uint32_t)b * kBBytes;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const uint32_t kb = k >> 2, kk = k & 3;
          tc_mma_f16(d, smem_desc_sw128(sA + kb * 16384u + kk * 32u),
                     smem_desc_sw128(sB + kb * (uint32_t)(BN * 128) + kk * 32u), kIdesc, k > 0 ? 1u : 0u);
        }
        tc_commit(bar_mma0 + 8 * b);
        last = i;
      }
      // drain what this thread started: a W_V copy and the last MMAs
      if (tma_pending) mbar_wait(bar_wv, wv_par, p.err, kErrWaitTeardown);
      if (last >= 0) mbar_wait(bar_mma0 + 8 * (last & 1), (last >> 1) & 1, p.err, kErrWaitTeardown);
    }
    __syncwarp();
  } else {
    // ---------------- workers: combine + epilogue ----------------
    const int wq = warp & 3;   // TMEM lane quadrant of this warp
    const int wh = warp >> 2;  // which half of the tile's columns it drains
    const int layout = p.layout, n = p.n_part;

    // Epilogue of local unit j: TMEM accumulator -> bf16 -> * gate -> core.
    auto epilogue = [&](int j) -> bool {
      const int u = ub + j, h = u / tph, t0 = (u - h * tph) * BN, bj = j & 1;
      const int v = wq * 32 + lane;
      const int tb = t0 + wh * (BN / 2);
      uint16_t g[BN / 2];
#pragma unroll
      for (int e = 0; e < BN / 2; ++e) {
        const int t = tb + e;
        g[e] = (t < p.S) ? __ldg(p.gate + (long long)t * Wrow + h * kV + v) : (uint16_t)0;
      }
      bool ok = wait_or_abort(bar_mma0 + 8 * bj, (j >> 1) & 1, p.err, kErrWaitMma, s_abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      tc_fence_after();
#pragma unroll
      for (int c8 = 0; c8 < BN / 16; ++c8) {
        uint32_t r[8];
        tmem_ld_x8(tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(bj * BN + wh * (BN / 2) + c8 * 8), r);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = tb + c8 * 8 + e;
          if (t < p.S) {
            const float a = round_bf16(__uint_as_float(r[e]));
            const float gv = __uint_as_float((uint32_t)g[c8 * 8 + e] << 16);
            const __nv_bfloat16 o = __float2bfloat16_rn(a * gv);
            p.out[(long long)t * Wrow + h * kV + v] = *reinterpret_cast<const uint16_t *>(&o);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc0 + 8 * bj);
      return true;
    };

    // Combine the warp's TPW tokens of a unit into latent buffer b.
    auto combine = [&](int h, int t0, int b) {
      uint8_t *gB = gB0 + (size_t)b * kBBytes;
      int tt[TPW];
      bool valid[TPW];
#pragma unroll
      for (int tk = 0; tk < TPW; ++tk) {
        tt[tk] = t0 + warp * TPW + tk;
        valid[tk] = tt[tk] < p.S;
      }
      uint4 res[TPW][2];
      if (layout == kPassthrough) {
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk) {
          if (valid[tk]) {
            const uint4 *row =
                reinterpret_cast<const uint4 *>(p.o + (long long)tt[tk] * p.o_st + (long long)h * p.o_sh);
            res[tk][0] = __ldcs(row + lane);
            res[tk][1] = __ldcs(row + lane + 32);
          } else {
            res[tk][0] = res[tk][1] = make_uint4(0, 0, 0, 0);
          }
        }
      } else {
        long long rowoff[TPW];  // o element offset of token tk's first partial
        float wgt[TPW];         // this lane's partial's weight, per token
        float lv[TPW];
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk) {
          const int r0 = (layout == kRequestMajor) ? (tt[tk] / p.q) * p.spr : 0;
          rowoff[tk] = (long long)r0 * p.o_sp + (long long)tt[tk] * p.o_st + (long long)h * p.o_sh;
          lv[tk] = (valid[tk] && lane < n)
                       ? sane(__ldg(p.lse + (long long)(r0 + lane) * p.l_sp + (long long)tt[tk] * p.l_st +
                                    (long long)h * p.l_sh))
                       : __int_as_float(0xFF800000);
        }
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk) {
          float m = lv[tk];
#pragma unroll
          for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
          if (m == __int_as_float(0xFF800000)) m = 0.0f;
          const float e = (lane < n) ? exp2f(__fmul_rn(__fsub_rn(lv[tk], m), kLog2e)) : 0.0f;
          float Z = 0.0f;  // in partial order, as a sequential fp32 sum
          for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, j));
          const float inv = (Z == 0.0f) ? 0.0f : __frcp_rn(Z);
          wgt[tk] = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
        }
        float acc[TPW][16];
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk)
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[tk][e] = 0.0f;
        uint4 cur[TPW][2], nxt[TPW][2];
        float cw[TPW], nw[TPW];
        auto load = [&](int j, uint4 (&buf)[TPW][2], float (&w)[TPW]) {
#pragma unroll
          for (int tk = 0; tk < TPW; ++tk) {
            w[tk] = __shfl_sync(0xffffffffu, wgt[tk], j);
            if (w[tk] != 0.0f) {
              const uint4 *row = reinterpret_cast<const uint4 *>(p.o + rowoff[tk] + (long long)j * p.o_sp);
              buf[tk][0] = __ldcs(row + lane);
              buf[tk][1] = __ldcs(row + lane + 32);
            } else {
              buf[tk][0] = buf[tk][1] = make_uint4(0, 0, 0, 0);
            }
          }
        };
        load(0, cur, cw);
        for (int j = 0; j < n; ++j) {
          if (j + 1 < n) load(j + 1, nxt, nw);
#pragma unroll
          for (int tk = 0; tk < TPW; ++tk) {
            if (cw[tk] == 0.0f) continue;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t uu[4] = {cur[tk][c].x, cur[tk][c].y, cur[tk][c].z, cur[tk][c].w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                acc[tk][c * 8 + 2 * q] = __fadd_rn(acc[tk][c * 8 + 2 * q], __fmul_rn(cw[tk], bf16_lo(uu[q])));
                acc[tk][c * 8 + 2 * q + 1] =
                    __fadd_rn(acc[tk][c * 8 + 2 * q + 1], __fmul_rn(cw[tk], bf16_hi(uu[q])));
              }
            }
          }
#pragma unroll
          for (int tk = 0; tk < TPW; ++tk) {
            cur[tk][0] = nxt[tk][0];
            cur[tk][1] = nxt[tk][1];
            cw[tk] = nw[tk];
          }
        }
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            res[tk][c] = make_uint4(pack_bf16(acc[tk][c * 8 + 0], acc[tk][c * 8 + 1]),
                                    pack_bf16(acc[tk][c * 8 + 2], acc[tk][c * 8 + 3]),
                                    pack_bf16(acc[tk][c * 8 + 4], acc[tk][c * 8 + 5]),
                                    pack_bf16(acc[tk][c * 8 + 6], acc[tk][c * 8 + 7]));
      }
#pragma unroll
      for (int tk = 0; tk < TPW; ++tk) {
        const int row = warp * TPW + tk;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint4 x = res[tk][c];
          if (WFMT == 1) x = mx_chunk(x);
          if (!valid[tk]) x = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(gB + sw128_offset(row, lane + 32 * c, BN)) = x;
        }
      }
    };

    // MXFP4: W_V[h] codes + scales -> exact bf16 values in the swizzled A tile.
    auto dequant_wv = [&](int h) {
      const uint8_t *wbase = static_cast<const uint8_t *>(p.w_v) + (long long)h * p.w_sh;
      const uint8_t *sbase_h = p.w_scale + (long long)h * p.s_sh;
      for (int s = threadIdx.x; s < kV * 64; s += 256) {
        const int v = s >> 6, c = s & 63;
        const uint32_t codes = __ldg(reinterpret_cast<const uint32_t *>(wbase + (long long)v * p.w_sv) + c);
        const float scale = e8m0_to_f32(__ldg(sbase_h + (long long)v * p.s_sv + (c >> 2)));
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t c0 = (codes >> (8 * q)) & 0xFu, c1 = (codes >> (8 * q + 4)) & 0xFu;
          float a = e2m1_mag_value(c0 & 7u) * scale, bb = e2m1_mag_value(c1 & 7u) * scale;
          pk[q] = pack_bf16((c0 & 8u) ? -a : a, (c1 & 8u) ? -bb : bb);
        }
        *reinterpret_cast<uint4 *>(gA + sw128_offset(v, c, kV)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    };

    int prev_h = -1;
    bool ok = true;
    for (int i = 0; i < nu && ok; ++i) {
      if (*s_abort) {
        ok = false;
        break;
      }
      const int u = ub + i, h = u / tph, t0 = (u - h * tph) * BN, b = i & 1;
      bool ep_done = false;
      if (WFMT == 1 && h != prev_h) {
        if (i > 0) {
          if (!epilogue(i - 1)) {
            ok = false;
            break;
          }
          ep_done = true;
        }
        dequant_wv(h);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_wv);
        prev_h = h;
      }
      combine(h, t0, b);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_lat0 + 8 * b);
      if (i > 0 && !ep_done) ok = epilogue(i - 1);
    }
    if (ok && nu > 0 && !*s_abort) epilogue(nu - 1);

    // rows S .. S_out-1 of core are zero (this CTA's slice of them)
    const long long n16 = (long long)(p.S_out - p.S) * p.H * (kV * 2 / 16);
    if (n16 > 0) {
      const long long zb = (long long)blockIdx.x * n16 / gridDim.x;
      const long long ze = (long long)(blockIdx.x + 1) * n16 / gridDim.x;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + (long long)p.S * Wrow);
      for (long long k = zb + threadIdx.x; k < ze; k += 256) dst[k] = make_uint4(0, 0, 0, 0);
    }
  }

  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

size_t tc_smem_bytes(int tile) { return 1024 + kABytes + 2u * (size_t)tile * 1024u + 128; }

template <int BN, int WFMT>
static cudaError_t launch_one(const KParams &p, const CUtensorMap *tmap, int grid, cudaStream_t s) {
  static bool attr_set = false;  // per process; the attribute is per function
  const size_t smem = tc_smem_bytes(BN);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc_kernel<BN, WFMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  tc_kernel<BN, WFMT><<<grid, kTcThreads, smem, s>>>(p, *tmap);
  return cudaGetLastError();
}

cudaError_t launch_tc(const KParams &p, const CUtensorMap *tmap_w, int grid, cudaStream_t stream) {
  if (p.tile == 16) return p.w_fmt == 0 ? launch_one<16, 0>(p, tmap_w, grid, stream)
                                        : launch_one<16, 1>(p, tmap_w, grid, stream);
  if (p.tile == 32) return p.w_fmt == 0 ? launch_one<32, 0>(p, tmap_w, grid, stream)
                                        : launch_one<32, 1>(p, tmap_w, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mla
