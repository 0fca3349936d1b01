// kernel_tc.cu -- fused tensor-core kernel of the MLA decode post-attention
// stage for sm_103a: LSE combine -> (MXFP4) latents in shared memory ->
// tcgen05 W_UV GEMM with the accumulator in TMEM -> gate epilogue.
//
// Work unit: (head h, BN-token tile), head-major, split into one contiguous
// run per CTA (persistent grid of at most one CTA per SM), so a CTA keeps
// W_V[h] resident in shared memory across the token tiles of a head.  The
// epilogue stages each warp's bf16 accumulators through shared memory so the
// gate loads and core stores are 16-byte, token-major accesses.
//
// GEMM orientation (per unit): D[v, t] = sum_k W_V[h][v][k] * lat[t][k] with
// M = 128 (the V rows), N = BN tokens, K = 512, both operands K-major with
// the 128-byte swizzle.  This keeps M at the tensor core's 128 while the
// token tile stays small enough for decode batches.
//
// Warp roles (512 threads, 16 warps, all alike): each warp combines BN/16 of
// a unit's tokens into the latent buffer, then runs the epilogue of the
// previous unit (TMEM -> registers, bf16(acc) * gate -> core).  The warp that
// completes a unit's latents last (per-buffer monotonic arrival counters)
// issues that unit's 32 MMAs from one thread and commits them to an
// mbarrier; being last also proves every warp has drained the previous
// accumulator in that TMEM buffer.  At a head change every warp first waits
// for the previous head's MMAs, then copies (bf16) or dequantises (MXFP4)
// W_V[h] into the A tile.  Latent buffers and TMEM accumulators
// are double-buffered, so the combine of unit i overlaps the MMA of unit i-1
// and the epilogue of unit i-2.  A warp issues all of its tokens' partial-row
// loads of a batch at once and prefetches the next unit's LSE values while
// they are in flight.
//
// Semantics follow the vLLM page "vllm.models.kimi_k3.amd.specialized_decode.
// mono.attention.mla_back": combine_ranks / combine_splits (sane, LSE weights,
// zero-weight partials masked), stage_combine (bf16 latents, passthrough for
// one partial, padded tokens zero), stage_uv (MXFP4 latents, W_UV, bf16(acc)
// * gate), combine_tasks / tasks (a persistent loop over (head, tokens)
// tasks).  The merge keeps one rounding per multiply and per add, partials in
// index order (packed f32x2 arithmetic rounds each lane like a scalar op).
// Every mbarrier wait is bounded; on timeout the kernel records an error,
// drains its own in-flight copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr uint32_t kABytes = 128u * 1024u;  // W_V[h], bf16, 8 K-blocks x 16 KiB
constexpr int kWorkers = kTcWarps;           // all warps combine, drain and (one of them) issue
constexpr uint32_t kEpiBytes = kTcWarps * 8u * 32u * 2u;  // epilogue staging, 8 KiB

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

// MXFP4 round trip of a lane's 8 bf16 latents (one 16-byte chunk): the block
// of 32 spans lanes 4g..4g+3.  Scale code from the largest sign-cleared bf16
// pattern; elements scaled by an exact power of two, converted to E2M1 by the
// hardware (nearest even, saturating at 6) and back; the result is the exact
// dequantised value, returned as bf16.
__device__ __forceinline__ uint4 mx_chunk(uint4 x) {
  uint32_t u[4] = {x.x, x.y, x.z, x.w};
  uint32_t am2 = max_u16x2(max_u16x2(u[0] & 0x7FFF7FFFu, u[1] & 0x7FFF7FFFu),
                           max_u16x2(u[2] & 0x7FFF7FFFu, u[3] & 0x7FFF7FFFu));
  uint32_t am = max(am2 & 0xFFFFu, am2 >> 16);
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
  const uint32_t sc = mx_scale_code(am);
  if (sc == 255u) return make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
  const float scale = e8m0_to_f32(sc), inv = e8m0_inverse(sc);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t e = e2m1x2_from_f32(bf16_lo(u[q]) * inv, bf16_hi(u[q]) * inv);
    const uint32_t h2 = f16x2_from_e2m1x2(e);
    u[q] = pack_bf16(f16_lo(h2) * scale, f16_hi(h2) * scale);
  }
  return make_uint4(u[0], u[1], u[2], u[3]);
}

}  // namespace

template <int BN, int WFMT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const __grid_constant__ KParams p) {
  constexpr int TPW = BN / kWorkers;       // tokens per warp per unit
  constexpr int JB = 4 / TPW;              // partials per batch: 4 rows (8 x 16 B per lane)
  constexpr int CPW = BN / 4;              // TMEM columns each warp drains
  constexpr uint32_t kBBytes = BN * 1024u; // one latent buffer (BN x 512 bf16)
  constexpr uint32_t kCols = (2 * BN < 32) ? 32u : (uint32_t)(2 * BN);
  constexpr uint32_t kIdesc = idesc_bf16(128, BN);
  static_assert(TPW >= 1 && BN % kWorkers == 0 && JB >= 1, "tile must split over the warps");
  static_assert(CPW == 4 || CPW == 8, "epilogue drains 4 or 8 columns per warp");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;    // 1024-byte aligned (swizzle atoms)
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB0 = sbase + kABytes;
  uint8_t *gA = gbase;
  uint8_t *gB0 = gbase + kABytes;
  // per-warp epilogue staging: CPW tokens x 32 V rows of bf16
  uint16_t *gE = reinterpret_cast<uint16_t *>(gbase + kABytes + 2 * kBBytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + kABytes + 2 * kBBytes + kEpiBytes);
  uint32_t *misc = reinterpret_cast<uint32_t *>(bars + 4);
  // misc[0] TMEM base, misc[1] abort flag, misc[2..3] arrival counters,
  // misc[4] last unit whose MMAs were issued (+1)
  volatile int *s_abort = reinterpret_cast<volatile int *>(&misc[1]);
  const uint32_t bar_mma0 = smem_u32(&bars[0]);  // +8*b
  const uint32_t cnt0 = smem_u32(&misc[2]);      // +4*b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar_mma0, 1u);
    mbar_init(bar_mma0 + 8, 1u);
    for (int k = 1; k < 6; ++k) misc[k] = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc[0]), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  const int tph = p.tiles_per_head;
  const int ub = (int)((long long)blockIdx.x * p.units / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * p.units / gridDim.x);
  const int nu = ue - ub;
  const int Wrow = p.H * kV;
  const int wq = warp & 3;   // TMEM lane quadrant of this warp
  const int ws = warp >> 2;  // which quarter of the tile's columns it drains
  const int layout = p.layout, n = p.n_part;
  const bool pass = (layout == kPassthrough);
  const float kNegInf = __int_as_float(0xFF800000);
  const int nb = (n + JB - 1) / JB;  // load batches per unit

  // A cursor over the CTA's units: head and token tile, advanced one unit at
  // a time (no division in the loop).
  struct Cur {
    int h, tile;
  };
  const Cur c_first{ub / tph, ub - (ub / tph) * tph};
  auto advance = [&](Cur &c) {
    if (++c.tile == tph) {
      c.tile = 0;
      ++c.h;
    }
  };

  // Epilogue of a unit: TMEM accumulator -> bf16 -> (staged through shared
  // memory, token-major) * gate -> core with 16-byte accesses.
  uint16_t *stage = gE + warp * (CPW * 32);
  auto epilogue = [&](int j, const Cur &c) -> bool {
    const int bj = j & 1;
    // lane -> (token e, 8 consecutive V rows)
    constexpr int kLanes = CPW * 4;
    const int e = lane >> 2, v8 = (lane & 3) * 8;
    const int t = c.tile * BN + ws * CPW + e;
    const bool act = lane < kLanes && t < p.S;
    const long long off = (long long)t * Wrow + c.h * kV + wq * 32 + v8;
    uint4 g = make_uint4(0, 0, 0, 0);
    if (act) g = __ldg(reinterpret_cast<const uint4 *>(p.gate + off));
    bool ok = wait_or_abort(bar_mma0 + 8 * bj, (j >> 1) & 1, p.err, kErrWaitMma, s_abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    tc_fence_after();
    uint32_t r[CPW];
    const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(bj * BN + ws * CPW);
    if constexpr (CPW == 8) {
      tmem_ld_x8(taddr, r);
    } else {
      tmem_ld_x4(taddr, r);
    }
    tc_wait_ld();
    tc_fence_before();
#pragma unroll
    for (int x = 0; x < CPW; ++x) {
      const __nv_bfloat16 a = __float2bfloat16_rn(__uint_as_float(r[x]));
      stage[x * 32 + lane] = *reinterpret_cast<const uint16_t *>(&a);
    }
    __syncwarp();
    if (act) {
      const uint4 a = *reinterpret_cast<const uint4 *>(stage + e * 32 + v8);
      const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, gg[4] = {g.x, g.y, g.z, g.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = pack_bf16(bf16_lo(aa[q]) * bf16_lo(gg[q]), bf16_hi(aa[q]) * bf16_hi(gg[q]));
      *reinterpret_cast<uint4 *>(p.out + off) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncwarp();
    return true;
  };

  // This lane's LSE of partial `lane` for the warp's tokens of a unit (-inf
  // past n or past S; sanitised when used).
  auto load_lse = [&](const Cur &c, float (&lv)[TPW]) {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      const int t = c.tile * BN + warp * TPW + tk;
      lv[tk] = kNegInf;
      if (!pass && t < p.S && lane < n) {
        const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
        lv[tk] = __ldg(p.lse + (long long)(r0 + lane) * p.l_sp + (long long)t * p.l_st + (long long)c.h * p.l_sh);
      }
    }
  };

  // Weight of partial `lane` per token (LSE rule; one partial passes through).
  auto weights_of = [&](const float (&lv)[TPW], float (&wg)[TPW]) {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      if (pass) {
        wg[tk] = (lane == 0) ? 1.0f : 0.0f;
        continue;
      }
      const float l = sane(lv[tk]);
      float m = l;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
      if (m == kNegInf) m = 0.0f;
      const float e = (lane < n) ? exp2f(__fmul_rn(__fsub_rn(l, m), kLog2e)) : 0.0f;
      float Z = 0.0f;  // sequential fp32 sum in partial order
      for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, j));
      const float inv = (Z == 0.0f) ? 0.0f : __frcp_rn(Z);
      wg[tk] = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
    }
  };

  using Buf = uint4[JB][TPW][2];
  using Wts = float[JB][TPW];

  // Issue the loads of one batch: unit at cursor c, partials j0 .. j0+JB-1
  // (rows of zero weight and tokens past S are not read).
  auto issue = [&](const Cur &c, int j0, Buf &buf, Wts &w, const float (&wg)[TPW]) {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      const int t = c.tile * BN + warp * TPW + tk;
      const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
      const uint16_t *base = p.o + (long long)t * p.o_st + (long long)c.h * p.o_sh + (long long)(r0 + j0) * p.o_sp;
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        w[jj][tk] = __shfl_sync(0xffffffffu, wg[tk], (j0 + jj) & 31);  // 0 past n
        if (w[jj][tk] != 0.0f && t < p.S) {
          const uint4 *row = reinterpret_cast<const uint4 *>(base + (long long)jj * p.o_sp);
          buf[jj][tk][0] = __ldcs(row + lane);
          buf[jj][tk][1] = __ldcs(row + lane + 32);
        } else {
          buf[jj][tk][0] = buf[jj][tk][1] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  };

  uint64_t acc[TPW][8];  // fp32 pairs: elements (2q, 2q+1) of chunk q/4
  auto clear_acc = [&]() {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[tk][e] = 0ull;
  };

  // Merge one batch in partial order: acc += w * o, one rounding per op.
  auto consume = [&](const Buf &buf, const Wts &w) {
#pragma unroll
    for (int jj = 0; jj < JB; ++jj) {
#pragma unroll
      for (int tk = 0; tk < TPW; ++tk) {
        if (w[jj][tk] == 0.0f) continue;
        const uint64_t w2 = f2_pack(w[jj][tk], w[jj][tk]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t uu[4] = {buf[jj][tk][c].x, buf[jj][tk][c].y, buf[jj][tk][c].z, buf[jj][tk][c].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint64_t o2 = f2_pack(bf16_lo(uu[q]), bf16_hi(uu[q]));
            acc[tk][c * 4 + q] = f2_add(acc[tk][c * 4 + q], f2_mul(w2, o2));
          }
        }
      }
    }
  };

  // W_V[h] -> the swizzled bf16 A tile: bf16 rows copied, MXFP4 codes +
  // scales turned into their exact bf16 values.
  auto load_wv = [&](int h) {
    if (WFMT == 0) {
      const uint16_t *wb = static_cast<const uint16_t *>(p.w_v) + (long long)h * p.w_sh;
      constexpr int kPer = kV * 64 / kTcThreads;
      uint4 x[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int s = threadIdx.x + i * kTcThreads;
        x[i] = __ldg(reinterpret_cast<const uint4 *>(wb + (long long)(s >> 6) * p.w_sv) + (s & 63));
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int s = threadIdx.x + i * kTcThreads;
        *reinterpret_cast<uint4 *>(gA + sw128_offset(s >> 6, s & 63, kV)) = x[i];
      }
      return;
    }
    const uint8_t *wbase = static_cast<const uint8_t *>(p.w_v) + (long long)h * p.w_sh;
    const uint8_t *sbase_h = p.w_scale + (long long)h * p.s_sh;
    constexpr int kPer = kV * 64 / kTcThreads;  // 16-byte chunks per thread
#pragma unroll 4
    for (int i = 0; i < kPer; ++i) {
      const int s = threadIdx.x + i * kTcThreads;
      const int v = s >> 6, c = s & 63;
      const uint32_t codes = __ldg(reinterpret_cast<const uint32_t *>(wbase + (long long)v * p.w_sv) + c);
      const float scale = e8m0_to_f32(__ldg(sbase_h + (long long)v * p.s_sv + (c >> 2)));
      uint32_t pk[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t h2 = f16x2_from_e2m1x2((codes >> (8 * q)) & 0xFFu);
        pk[q] = pack_bf16(f16_lo(h2) * scale, f16_hi(h2) * scale);
      }
      *reinterpret_cast<uint4 *>(gA + sw128_offset(v, c, kV)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  };

  // The unit's MMAs (one thread): D[v, t] = sum_k W_V[h][v][k] * lat[t][k].
  auto issue_mma = [&](int i) {
    const int b = i & 1;
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
    misc[4] = (uint32_t)(i + 1);
  };

  bool ep_early = false;  // epilogue of the previous unit already done

  // Unit i (cursor c; previous unit at cp) has its latents merged: round /
  // quantise, store, arrive (the last warp issues the MMAs), then drain the
  // previous unit's accumulator.
  auto finish = [&](int i, const Cur &c, const Cur &cp, const Buf &raw_rows) -> bool {
    const int b = i & 1;
    uint8_t *gB = gB0 + (size_t)b * kBBytes;
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      const bool valid = c.tile * BN + warp * TPW + tk < p.S;
      const int row = warp * TPW + tk;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint4 x;
        if (pass) {
          x = raw_rows[0][tk][cc];
        } else {
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float lo, hi;
            f2_unpack(acc[tk][cc * 4 + q], lo, hi);
            pk[q] = pack_bf16(lo, hi);
          }
          x = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        if (WFMT == 1) x = mx_chunk(x);
        if (!valid) x = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(gB + sw128_offset(row, lane + 32 * cc, BN)) = x;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      // arrivals on buffer b are numbered across its uses: use (i >> 1) takes
      // numbers (i >> 1) * kWorkers .. + kWorkers - 1; the last one issues
      const uint32_t prev = atom_add_acq_rel_cta(cnt0 + 4 * b, 1u);
      if (prev == (uint32_t)((i >> 1) + 1) * kWorkers - 1u) issue_mma(i);
    }
    __syncwarp();
    bool ok = true;
    if (i > 0 && !ep_early) ok = epilogue(i - 1, cp);
    ep_early = false;
    clear_acc();
    // next unit on another head: W_V must be replaced once this unit's MMAs
    // are complete
    if (ok && i + 1 < nu && c.tile + 1 == tph) {
      ok = epilogue(i, c);
      ep_early = true;
      if (ok) load_wv(c.h + 1);
    }
    return ok;
  };

  // ---- the pipeline: step k merges batch k while batch k+1 is in flight ----
  bool ok = true;
  clear_acc();
  float lse1[TPW], lse2[TPW];  // LSE of units i+1 and i+2
  float wcur[TPW], wnxt[TPW];  // weights of units i and i+1
  Buf bufA, bufB;
  Wts wA, wB;
  Cur cu = c_first;    // unit i (being merged)
  Cur cprev = c_first; // unit i-1
  Cur cn = c_first;    // unit of the next batch to issue
  Cur cl = c_first;    // next unit whose LSE is loaded (i+3)
  int i = 0, bi = 0;   // unit and batch being merged
  int nbi = 1;         // batch index of the next batch within its unit
  if (nu > 0) {
    float lse0[TPW];
    load_lse(cl, lse0);
    advance(cl);
    if (nu > 1) load_lse(cl, lse1);
    advance(cl);
    if (nu > 2) load_lse(cl, lse2);
    advance(cl);
    load_wv(c_first.h);
    weights_of(lse0, wcur);
    issue(cu, 0, bufA, wA, wcur);
    if (nbi == nb) {
      nbi = 0;
      advance(cn);
    }
  }
  const int total = nu * nb;

  auto step = [&](int k, Buf &cur, Wts &wc, Buf &nxt, Wts &wn) -> bool {
    if (k + 1 < total) {
      if (nbi == 0) {
        // the next batch opens unit i+1
        weights_of(lse1, wnxt);
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk) lse1[tk] = lse2[tk];
        if (i + 3 < nu) load_lse(cl, lse2);
        advance(cl);
        issue(cn, 0, nxt, wn, wnxt);
      } else {
        issue(cn, nbi * JB, nxt, wn, wcur);
      }
      if (++nbi == nb) {
        nbi = 0;
        advance(cn);
      }
    }
    consume(cur, wc);
    if (++bi == nb) {
      if (!finish(i, cu, cprev, cur)) return false;
#pragma unroll
      for (int tk = 0; tk < TPW; ++tk) wcur[tk] = wnxt[tk];
      cprev = cu;
      advance(cu);
      ++i;
      bi = 0;
    }
    return true;
  };

  for (int k = 0; k < total; k += 2) {
    if (*s_abort) {
      ok = false;
      break;
    }
    if (!step(k, bufA, wA, bufB, wB)) {
      ok = false;
      break;
    }
    if (k + 1 < total && !step(k + 1, bufB, wB, bufA, wA)) {
      ok = false;
      break;
    }
  }
  if (ok && nu > 0 && !*s_abort) epilogue(nu - 1, cprev);

  // rows S .. S_out-1 of core are zero (this CTA's slice of them)
  const long long n16 = (long long)(p.S_out - p.S) * p.H * (kV * 2 / 16);
  if (n16 > 0) {
    const long long zb = (long long)blockIdx.x * n16 / gridDim.x;
    const long long ze = (long long)(blockIdx.x + 1) * n16 / gridDim.x;
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (long long)p.S * Wrow);
    for (long long k = zb + threadIdx.x; k < ze; k += kTcThreads) dst[k] = make_uint4(0, 0, 0, 0);
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    // drain what this CTA started (only pending after an abort): the last
    // committed MMAs
    if (misc[4] > 0u) {
      const int last = (int)misc[4] - 1;
      mbar_wait(bar_mma0 + 8 * (last & 1), (last >> 1) & 1, p.err, kErrWaitTeardown);
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

size_t tc_smem_bytes(int tile) { return 1024 + kABytes + 2u * (size_t)tile * 1024u + kEpiBytes + 128; }

template <int BN, int WFMT>
static cudaError_t launch_one(const KParams &p, int grid, cudaStream_t s) {
  const size_t smem = tc_smem_bytes(BN);
  cudaError_t e = cudaFuncSetAttribute(tc_kernel<BN, WFMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_kernel<BN, WFMT><<<grid, kTcThreads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc(const KParams &p, int grid, cudaStream_t stream) {
  if (p.tile == 16) return p.w_fmt == 0 ? launch_one<16, 0>(p, grid, stream) : launch_one<16, 1>(p, grid, stream);
  if (p.tile == 32) return p.w_fmt == 0 ? launch_one<32, 0>(p, grid, stream) : launch_one<32, 1>(p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mla
