// kernel_attn.cu -- the partial producer: split-KV MLA decode attention in
// the absorbed form, writing the (o, lse) partials the combine merges.
//
// The vLLM page "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.
// mla_back" names this producer (M1c, mla_attn: o / lse of dense [splits, S,
// 12, 512] bf16 / [splits, S, 12] f32, a request's splits merged by the
// combine) but does not print it; this kernel follows the plain definition.
// A query row is 576 wide (latent query, W_UK absorbed, then rope query); a
// cached row is the latent (512) then the rope key (64).  Token i of request
// b sees positions j < kv_len[b] - (q - 1 - i); split r covers [r C,
// (r + 1) C) with C = ceil(kv_len[b] / spr).  Per (split, token, head):
// lse = ln sum_j exp(scale q.k_j) and o = sum_j softmax_j * latent_j (bf16);
// a split with no visible position gives lse -inf and o 0.
//
// Work items are (request, split, group of G heads): the N = roundup16(q G)
// query rows of an item share every cached row it reads, so a row is read
// once per group.  A persistent grid walks the items.  Up to 16 query rows
// run two CTAs per SM with tiles of 64 positions, 32 rows one CTA per SM with
// tiles of 128.  Per tile:
//   * TMA brings the tile as four double blocks (latents 128 c .. 128 c +
//     127, two [positions x 64] boxes with the 128-byte swizzle) and one rope
//     block, into rings of shared-memory slots;
//   * one thread issues S^T = K Q^T on the tensor cores (M = the tile's
//     positions, N query rows, K = 576), accumulator in TMEM;
//   * eight softmax warps (two per TMEM lane quadrant, a thread per position,
//     half the query rows each) mask, take the column max, write P^T =
//     exp2(s - reference max) in bf16 to shared memory and, when a column's
//     reference moved, rescale that column of the O accumulator in TMEM;
//   * O^T += V^T P^T (four M = 128 latent chunks, K = the tile's positions),
//     V^T being the tile's latent read MN-major in place: issued by the same
//     thread, or (the attention alone) by a thread of its own, so that the
//     next tile's S^T goes out while this tile's softmax and O^T run.
// At the end of an item the softmax warps divide by the column sums, write o
// (bf16) and lse.  Every wait is bounded; a timeout records an error, the
// roles stop, and the kernel waits (bounded) for its own copies and MMAs
// before it frees TMEM and returns.
//
// The FUSED instance (mla_attn_combine_uv) runs the combine of the same page
// behind the attention in the same launch, as the page's M1c + combine pair
// does.  Its items come from a queue every CTA draws from (a workspace
// counter): the TMA lane draws the next item when it is ready to copy its
// tiles and hands it to the other roles through a small shared ring.  After
// an item's o / lse are written, the softmax warps add one arrival to each
// 8-token tile the request covers.  Behind the attention items the queue
// holds the combine units (8-token tile, head), tile-major: a CTA that draws
// one has finished its own attention items; it waits (bounded) until every
// item of the tile has arrived -- those items were all drawn earlier, by CTAs
// that are running, and none of them waits on a combine unit -- then one
// warp per token merges the token's partials (read back from L2) with the
// combine's LSE weights into bf16 latents in shared memory, W_V[h] arrives by
// TMA, one thread issues the W_UV GEMM (32 kind::f16 MMAs, M = 128 V rows,
// N = 16 with 8 tokens) into TMEM, and the same warps apply the gate and
// store core.  With an o_proj weight, units of (64 outputs, 64 tokens) of
// this rank's o_proj shard follow the combine units in the queue: each waits
// (bounded) until every combine unit has stored its core rows, then runs the
// GEMM the standalone o_proj kernel runs, with the same arithmetic.  The last
// CTA to finish zeroes the workspace again.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kAttnK = kD + 64;     // query / cached row width (576)
constexpr int kAttnSmx = 8;         // softmax warps: two per TMEM lane quadrant, half the query rows each
// warp 0 TMA, warp 1 MMAs, softmax warps 2 .. 1 + kAttnSmx, one query warp,
// and (AttnLayout::kSplitMma) one more warp for the O^T MMAs
constexpr int kPvWarp = 3 + kAttnSmx;
constexpr uint32_t kWvBytes = 128u * 1024u;  // FUSED: W_V[h], [128 x 512] bf16

constexpr int kItemRing = 4;        // FUSED: items handed from the TMA lane to the other roles
constexpr int kCmbTile = 8;         // FUSED: tokens per combine unit (one merging warp each)
constexpr uint32_t kOpBox = 64u * 128u;  // 64 rows x 64 bf16, 128-byte swizzle

// Two tilings.  Up to 16 query rows (N = 16) run two CTAs per SM, each with
// 64-position tiles (a tile's S^T is an M = 64 MMA, D row i in TMEM lane
// 32 (i / 16) + i % 16) and five latent double blocks plus a rope slot: one
// CTA's copies land while the other computes (the fused
// launch's combine units then stream W_V[h] through two 32-KiB slots).
// N = 32 runs one CTA per SM with 128-position tiles and a ring of five
// double blocks (its combine units keep W_V[h] resident).
template <int N, bool FUSED = false>
struct AttnLayout {
  static constexpr int kCtas = (N == 16) ? 2 : 1;             // CTAs per SM
  // The S^T and the O^T MMAs from two threads (one thread issues an MMA about
  // every 55 cycles at these N whatever its size, and the MMAs of two threads
  // overlap): S^T of the next tile then goes out while the softmax and the
  // O^T MMAs of this one run.  Not in the fused step: its 12th warp would cap
  // two CTAs per SM at 80 registers, and the launch measured slower.
  static constexpr bool kSplitMma = !FUSED;
  static constexpr int kThreads = ((kSplitMma ? 4 : 3) + kAttnSmx) * 32;
  static constexpr int kItemTakers = (kSplitMma ? 3 : 2) + kAttnSmx;  // FUSED: MMA lane(s), query warp, softmax warps
  static constexpr int kTile = kCtas == 2 ? 64 : 128;          // positions per tile (MMA M of S^T)
  static constexpr uint32_t kDblBytes = 2u * kTile * 128u;     // latents 128 c .. 128 c + 127 of a tile
  static constexpr uint32_t kRopeBytes = kTile * 128u;         // the tile's rope block
  static constexpr int kDbl = 5;                               // double-block slots (a tile needs 4)
  static constexpr int kRope = 1;                              // rope-block slots
  // FUSED o_proj: stages of a weight box and a core box (16 KiB each) below the barriers
  static constexpr int kOp = kCtas == 2 ? 6 : 10;
  static constexpr uint32_t dbl_off = 0;
  static constexpr uint32_t rope_off = dbl_off + kDbl * kDblBytes;
  static constexpr uint32_t q_off = rope_off + kRope * kRopeBytes;  // 9 K blocks of [N x 128 B]
  static constexpr uint32_t p_off = q_off + 9u * N * 128u;          // kTile / 64 K blocks of [N x 128 B]
  static constexpr uint32_t red_off = p_off + (kTile / 64) * N * 128u;  // float [2][4][N] (by tile parity)
  static constexpr uint32_t lim_off = red_off + 2u * 4u * N * 4u;   // int [N]
  static constexpr uint32_t row_off = (lim_off + N * 4u + 7u) & ~7u;  // long long [N]: o / lse row of a query row
  static constexpr uint32_t bar_off = row_off + N * 8u;
  // barriers: full/empty per double slot, full/empty per rope slot, then
  // s_full, s_free, p_full, o_full, q_full, q_free
  // FUSED adds: item full / empty per ring slot, W_V full, combine MMA done,
  // then the o_proj stages' full / empty, its accumulators' full and a
  // drain barrier per o_proj MMA thread; last, a drain barrier per attention
  // MMA thread (S^T, O^T)
  static constexpr int kBars = 2 * kDbl + 2 * kRope + 6 + (FUSED ? 2 * kItemRing + 5 + 2 * kOp + 3 : 0) + 2;
  // misc: [0] TMEM base, [1] abort flag, [2 .. 2 + kItemRing) item ring,
  // [6] the combine unit drawn last
  static constexpr uint32_t misc_off = bar_off + kBars * 8u;
  static constexpr uint32_t total = misc_off + 32u;
  static constexpr uint32_t tmem_cols = (5 * N <= 128) ? 128u : 256u;  // S^T (N) + O^T (4 N)
};
static_assert(AttnLayout<16, true>::total + 1024 <= 227u * 1024u, "shared memory (N = 16)");
static_assert(AttnLayout<32, true>::total + 1024 <= 227u * 1024u, "shared memory (N = 32)");
// FUSED: W_V[h] (128 KiB) reuses the first four double-block slots, the
// latent tile [16 x 512] bf16 (16 KiB) the first rope slot
static_assert(AttnLayout<16, false>::total + 1024 <= 113u * 1024u && AttnLayout<16, true>::total + 1024 <= 113u * 1024u,
              "shared memory (two CTAs per SM)");
// FUSED combine: W_V[h] resident in the first four double slots (one CTA per
// SM) or streamed in quarters through two 32-KiB slots (two CTAs per SM); the
// latent tile [16 x 512] bf16 in the rope slots
static_assert(4 * AttnLayout<32, true>::kDblBytes == kWvBytes && AttnLayout<32, true>::kRope * AttnLayout<32, true>::kRopeBytes >= 16u * 1024u &&
                  AttnLayout<16, true>::kDbl * AttnLayout<16, true>::kDblBytes >= kWvBytes / 2 &&
                  AttnLayout<16, true>::kRope * AttnLayout<16, true>::kRopeBytes + 9u * 16u * 128u >= 16u * 1024u,
              "combine tiles");
// FUSED o_proj: its stage ring reuses the latent double-block slots, its
// output tile [64 tokens x 64 features] bf16 is staged right after the ring
template <int N>
constexpr uint32_t kOpStgOff = AttnLayout<N, true>::kOp * 2u * kOpBox;
static_assert(kOpStgOff<16> + 64u * 128u <= AttnLayout<16, true>::bar_off &&
                  kOpStgOff<32> + 64u * 128u <= AttnLayout<32, true>::bar_off,
              "o_proj stages and output tile");

// Bounded wait on an mbarrier phase, shared abort flag (as the combine kernels).
__device__ __forceinline__ bool attn_wait(uint32_t bar, uint32_t parity, int *err, volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitNs) {
      atomicCAS(err, 0, kErrWaitAttn);
      *abort_flag = 1;
      return false;
    }
  }
}

// Wait (bounded) until the global counter reaches `target` (acquire).
__device__ __forceinline__ bool wait_count(const int *cnt, int target, unsigned long long limit_ns) {
  if (ld_acquire_gpu(cnt) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    __nanosleep(128);
    if (ld_acquire_gpu(cnt) >= target) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint4 ld_cg_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_cg_f32(const float *p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// The combine units of the fused launch (see the file comment), run by every
// thread of the CTA once its role has finished the attention items.  Shared
// memory: W_V[h] in the first four double-block slots (8 K blocks of [128 x
// 128 B], 128-byte swizzle, as TMA writes them), the unit's latents in the
// first rope slot (8 K blocks of [16 x 128 B]); TMEM columns 0..15 hold the
// accumulator D[v, token].
template <int N>
__device__ __forceinline__ void combine_phase(const AttnParams &p, const CUtensorMap &wv_map, uint32_t sbase,
                                              uint8_t *gbase, uint32_t tmem, uint32_t *misc, volatile int *s_abort,
                                              uint32_t wv_full, uint32_t wv_free, uint32_t cmb_mma, int nitems) {
  using L = AttnLayout<N, true>;
  // W_V[h] resident (one CTA per SM: reloaded only when the head changes), or
  // streamed per unit in quarters (kb 2q, 2q + 1) through two 32-KiB slots
  // (two CTAs per SM): the MMAs of a quarter run while the next one lands
  constexpr bool kStream = L::kCtas == 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.B * p.q, H = p.H, n = p.spr;
  const int nunits = p.ntiles * H;
  const int Wrow = H * kV;
  const uint32_t sA = sbase + L::dbl_off;
  const uint32_t sB = sbase + L::rope_off;
  uint8_t *gB = gbase + L::rope_off;
  const float kNegInf = __int_as_float(0xFF800000);
  constexpr unsigned kFull = 0xffffffffu;

  tc_fence_before();
  __syncthreads();  // every role is done with its attention items (copies landed, MMAs complete)
  tc_fence_after();
  int cur_h = -1, units = 0;
  int wv_issued = 0;   // thread 0: W_V loads issued (resident: whole W_V; streamed: quarters)
  int mma_issued = 0;  // MMA lane: units whose MMAs it committed
  int q_done = 0;      // MMA lane (streamed): quarters whose MMAs it committed
  int wv_seen = 0;     // every thread: W_V loads so far (resident)
  // streamed quarter q of W_V[h] (8 K blocks of 64, boxes [128 x 64]) into slot q % 2
  auto load_quarter = [&](int q, int h) {
    const uint32_t bar = wv_full + 8u * (uint32_t)(q & 1);
    mbar_arrive_expect_tx(bar, kWvBytes / 4);
    for (int j = 0; j < 2; ++j)
      tma_load_3d(sA + (uint32_t)(q & 1) * 32768u + (uint32_t)j * 16384u, &wv_map, 64 * (2 * q + j), 0, h, bar);
    ++wv_issued;
  };
  uint32_t unit = misc[6];
  while (!*s_abort && unit != 0xFFFFFFFFu && (int)unit - nitems < nunits) {
    const int u = (int)unit - nitems;
    const int tile = u / H, h = u - tile * H;
    const bool new_h = h != cur_h;
    if (threadIdx.x == 0) {
      // W_V[h] first (a weight: it does not wait for the attention), so its
      // copy overlaps the wait for the tile's partials
      if constexpr (kStream) {
        load_quarter(0, h);
        load_quarter(1, h);
      } else if (new_h) {
        mbar_arrive_expect_tx(wv_full, kWvBytes);
#pragma unroll 1
        for (int kb = 0; kb < 8; ++kb) tma_load_3d(sA + (uint32_t)kb * 16384u, &wv_map, 64 * kb, 0, h, wv_full);
        ++wv_issued;
      }
      // every (request, split, head group) item of the requests the tile covers
      const int t_lo = tile * kCmbTile, t_hi = min(t_lo + kCmbTile, S) - 1;
      const int target = (t_hi / p.q - t_lo / p.q + 1) * p.spr * p.groups;
      if (!wait_count(p.ws + 2 + tile, target, p.wait_ns)) {
        atomicCAS(p.err, 0, kErrWaitTile);
        *s_abort = 1;
      }
    }
    __syncthreads();
    if (*s_abort) break;
    if (new_h) {
      cur_h = h;
      ++wv_seen;
    }
    const bool merger = warp >= 2 && warp < 2 + kAttnSmx;
    if (merger) {
      // token t: the LSE weights of its spr partials (one per lane), then its
      // rows in partial order, fp32, one rounding per operation (the rule of
      // the combine kernels), rounded to bf16 into row mw of the tile
      const int mw = warp - 2, t = tile * kCmbTile + mw;
      const bool valid = t < S;
      float lv = kNegInf;
      if (valid && lane < n) lv = ld_cg_f32(p.lse + ((long long)lane * S + t) * H + h);
      const float l = sane(lv);
      float m = l;
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, s));
      if (m == kNegInf) m = 0.0f;
      const float e = (lane < n) ? ex2_approx(__fmul_rn(__fsub_rn(l, m), kLog2e)) : 0.0f;
      float Z = 0.0f;
      for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, __shfl_sync(kFull, e, j));
      const float inv = (Z == 0.0f) ? 0.0f : rcp_approx(Z);
      const float wg = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
      uint64_t acc[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] = 0ull;
      const long long pstride = (long long)S * H * kD;
      const uint16_t *row0 = p.o + ((long long)t * H + h) * kD;
      // batches of MB partial rows in flight (fewer with two CTAs per SM, whose
      // threads have 80 registers)
      constexpr int MB = kStream ? 4 : 8;
      for (int j0 = 0; j0 < n; j0 += MB) {
        uint4 buf[MB][2];
        float w[MB];
#pragma unroll
        for (int jj = 0; jj < MB; ++jj) {
          w[jj] = __shfl_sync(kFull, wg, (j0 + jj) & 31);  // 0 for partials past n
          if (w[jj] != 0.0f && valid) {
            const uint16_t *r = row0 + (long long)(j0 + jj) * pstride;
            buf[jj][0] = ld_cg_v4(r + 8 * lane);
            buf[jj][1] = ld_cg_v4(r + 256 + 8 * lane);
          } else {
            buf[jj][0] = buf[jj][1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int jj = 0; jj < MB; ++jj) {
          if (w[jj] == 0.0f) continue;
          const uint64_t w2 = f2_pack(w[jj], w[jj]);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t uu[4] = {buf[jj][c].x, buf[jj][c].y, buf[jj][c].z, buf[jj][c].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[c * 4 + q] = f2_add(acc[c * 4 + q], f2_mul(w2, f2_pack(bf16_lo(uu[q]), bf16_hi(uu[q]))));
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float lo, hi;
          f2_unpack(acc[c * 4 + q], lo, hi);
          pk[q] = pack_bf16(lo, hi);
        }
        const uint4 x = valid ? make_uint4(pk[0], pk[1], pk[2], pk[3]) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(gB + sw128_offset(mw, lane + 32 * c, 16)) = x;
      }
      fence_proxy_async_smem();
    }
    __syncthreads();
    if constexpr (kStream) {
      if (threadIdx.x == 0) {
        // quarters 2 and 3 into the slots quarters 0 and 1 free (each slot's
        // first free of the unit: parity 0)
        for (int q = 2; q < 4; ++q) {
          if (!attn_wait(wv_free + 8u * (uint32_t)(q & 1), 0u, p.err, s_abort)) break;
          load_quarter(q, h);
        }
      } else if (warp == 1 && lane == 0) {
        // D[v, token] = sum_k W_V[h][v][k] lat[token][k]: M = 128, N = 16, K = 512, quarter by quarter
        bool ok = true;
        const uint32_t dB = (uint32_t)smem_desc_sw128(sB);
        constexpr uint32_t kIdesc = idesc_bf16(128, 16);
        for (int q = 0; q < 4 && ok; ++q) {
          ok = attn_wait(wv_full + 8u * (uint32_t)(q & 1), (uint32_t)(q >> 1), p.err, s_abort);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dA = (uint32_t)smem_desc_sw128(sA + (uint32_t)(q & 1) * 32768u);
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            const uint32_t j = (uint32_t)k8 >> 2, kk = (uint32_t)k8 & 3u, kb = 2u * q + j;
            tc_mma_f16(tmem, desc_sw128_at(dA, j * 16384u + kk * 32u), desc_sw128_at(dB, kb * 2048u + kk * 32u), kIdesc,
                       (q | k8) ? 1u : 0u);
          }
          tc_commit(wv_free + 8u * (uint32_t)(q & 1));
          ++q_done;
        }
        if (ok) {
          tc_commit(cmb_mma);
          ++mma_issued;
        }
      }
    } else if (warp == 1 && lane == 0) {
      // D[v, token] = sum_k W_V[h][v][k] lat[token][k]: M = 128, N = 16, K = 512
      const bool ok = !new_h || attn_wait(wv_full, (uint32_t)(wv_seen - 1) & 1u, p.err, s_abort);
      if (ok) {
        tc_fence_after();
        const uint32_t dA = (uint32_t)smem_desc_sw128(sA), dB = (uint32_t)smem_desc_sw128(sB);
        constexpr uint32_t kIdesc = idesc_bf16(128, 16);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const uint32_t kb = (uint32_t)k >> 2, kk = (uint32_t)k & 3u;
          tc_mma_f16(tmem, desc_sw128_at(dA, kb * 16384u + kk * 32u), desc_sw128_at(dB, kb * 2048u + kk * 32u), kIdesc,
                     k > 0 ? 1u : 0u);
        }
        tc_commit(cmb_mma);
        ++mma_issued;
      }
    }
    if (merger) {
      // epilogue: this warp's TMEM lane quadrant (32 V rows) x 4 tokens
      const int qd = warp & 3, hh = (warp - 2) >> 2;
      bool ok = attn_wait(cmb_mma, (uint32_t)units & 1u, p.err, s_abort);
      ok = __all_sync(kFull, ok);
      if (ok) {
        tc_fence_after();
        uint32_t r[4];
        tmem_ld_x4(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(hh * 4), r);
        tc_wait_ld();
        tc_fence_before();
        const int v = qd * 32 + lane;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int t = tile * kCmbTile + hh * 4 + x;
          if (t < S) {
            const long long off = (long long)t * Wrow + h * kV + v;
            const float a = round_bf16(__uint_as_float(r[x]));
            const float g = __uint_as_float((uint32_t)__ldg(p.gate + off) << 16);
            const __nv_bfloat16 y = __float2bfloat16_rn(a * g);  // bf16(acc) * gate, exact in fp32, one rounding
            p.out[off] = *reinterpret_cast<const uint16_t *>(&y);
          }
        }
      }
    }
    ++units;
    __syncthreads();
    if (threadIdx.x == 0) {
      if (p.n_out > 0) {  // this unit's core rows are stored (read by the o_proj units)
        __threadfence();
        atomicAdd(p.ws + 2 + p.ntiles, 1);
      }
      misc[6] = (uint32_t)atomicAdd(p.ws, 1);
    }
    __syncthreads();
    unit = misc[6];
  }
  // after an abort: this CTA's weight copies and MMAs land before it exits
  if constexpr (kStream) {
    if (threadIdx.x == 0)  // quarter g of the CTA went to slot g % 2, the (g / 2)-th use of its barrier
      for (int g = wv_issued - 2 < 0 ? 0 : wv_issued - 2; g < wv_issued; ++g)
        mbar_wait(wv_full + 8u * (uint32_t)(g & 1), (uint32_t)(g >> 1) & 1u, p.err, kErrWaitTeardown);
    if (warp == 1 && lane == 0 && q_done > 0)
      mbar_wait(wv_free + 8u * (uint32_t)((q_done - 1) & 1), (uint32_t)((q_done - 1) >> 1) & 1u, p.err,
                kErrWaitTeardown);
  } else if (threadIdx.x == 0 && wv_issued > 0) {
    mbar_wait(wv_full, (uint32_t)(wv_issued - 1) & 1u, p.err, kErrWaitTeardown);
  }
  if (warp == 1 && lane == 0 && mma_issued > 0)
    mbar_wait(cmb_mma, (uint32_t)(mma_issued - 1) & 1u, p.err, kErrWaitTeardown);
  // rows S .. S_out - 1 of core are zero (this CTA's slice of them)
  const long long n16 = (long long)(p.S_out - S) * Wrow / 8;
  if (n16 > 0) {
    const long long zb = (long long)blockIdx.x * n16 / gridDim.x;
    const long long ze = (long long)(blockIdx.x + 1) * n16 / gridDim.x;
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (long long)S * Wrow);
    for (long long k = zb + threadIdx.x; k < ze; k += blockDim.x) dst[k] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// The o_proj units of the fused launch (n_out > 0), run by every thread of
// the CTA after its combine units: unit u covers outputs 64 (u % MT) .. + 63
// and tokens 64 (u / MT) .. + 63 of y[t][j] = sum_k core[t][k] W_o[j][k]
// (the page's stage ends at "o_proj's input"; this is the shard of o_proj
// that follows it).  Per 64-wide K block a stage holds the weight box and the
// core box (TMA, 128-byte swizzle); one thread issues four kind::f16 MMAs of
// M = 64, N = 64, K = 16 into TMEM columns 0..63 (D row i in lane 32 (i / 16)
// + i % 16), and warps 2..5 store the bf16 rounding of the accumulator.  The
// weight boxes of a CTA's first stages go out at once (a weight no kernel
// writes); its first core copy waits (bounded) until every combine unit has
// stored -- units drawn before any o_proj unit by CTAs that are running and
// never wait on an o_proj unit -- then orders those stores before its TMA
// reads with a proxy fence.
template <int N>
__device__ __forceinline__ void oproj_phase(const AttnParams &p, const CUtensorMap &wo_map, const CUtensorMap &x_map,
                                            uint32_t sbase, uint8_t *gbase, uint32_t tmem, uint32_t *misc,
                                            volatile int *s_abort, uint32_t obar) {
  using L = AttnLayout<N, true>;
  constexpr unsigned kFull = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.B * p.q, K = p.H * kV, KB = K / 64, MT = p.n_out / 64;
  const int base = p.B * p.spr * p.groups + p.ntiles * p.H;  // queue index of o_proj unit 0
  auto full = [&](int s) { return obar + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return obar + 8u * (uint32_t)(L::kOp + s); };
  const uint32_t acc_full = obar + 8u * (uint32_t)(2 * L::kOp);
  auto drain = [&](int w) { return obar + 8u * (uint32_t)(2 * L::kOp + 1 + w); };
  // two accumulators, D0 (even K blocks, issued by warp 1) and D1 (odd K
  // blocks, by the query loader's warp, idle here), summed in fp32 by the
  // epilogue: the arithmetic of the standalone o_proj kernel, so that both
  // give the same bits, with the MMAs of two threads overlapping
  constexpr int kW1 = 2 + kAttnSmx;
  auto sA = [&](int s) { return sbase + L::dbl_off + (uint32_t)s * 2u * kOpBox; };
  auto sB = [&](int s) { return sbase + L::dbl_off + (uint32_t)s * 2u * kOpBox + kOpBox; };

  tc_fence_before();
  __syncthreads();  // the combine units of this CTA are done (their copies landed, MMAs complete)
  tc_fence_after();
  int g = 0;           // stages issued (thread 0) / consumed (MMA lane) over this CTA's units
  int issued = 0;      // thread 0: stages whose copies went out
  int nu = 0;          // units done
  bool ready = false;  // thread 0: every combine unit has stored
  bool issued_mma = false;  // MMA lanes: this thread issued o_proj MMAs
  uint32_t unit = misc[6];
  while (!*s_abort && unit != 0xFFFFFFFFu && (int)unit >= base && (int)unit - base < p.op_units) {
    const int u = (int)unit - base, mt = u % MT, nt = u / MT;
    if (threadIdx.x == 0) {
      bool ok = true;
      int pre = 0;
      if (!ready) {  // the CTA's first unit (g == 0): weight boxes first, then the wait
        pre = KB < L::kOp ? KB : L::kOp;
        for (int kb = 0; kb < pre; ++kb) {
          mbar_arrive_expect_tx(full(kb), 2u * kOpBox);
          tma_load_3d(sA(kb), &wo_map, 64 * kb, mt * 64, 0, full(kb));
        }
        if (!wait_count(p.ws + 2 + p.ntiles, p.ntiles * p.H, p.wait_ns)) {
          atomicCAS(p.err, 0, kErrWaitTile);
          *s_abort = 1;
          ok = false;
        }
        fence_proxy_async_global();
        ready = true;
        // their core boxes (after a failed wait too, so that every stage
        // whose weight went out completes and the teardown can wait for it)
        for (int kb = 0; kb < pre; ++kb) tma_load_3d(sB(kb), &x_map, 64 * kb, nt * 64, 0, full(kb));
        g = pre;
        issued = pre;
      }
      for (int kb = pre; kb < KB && ok; ++kb, ++g) {
        const int s = g % L::kOp;
        if (g >= L::kOp) ok = attn_wait(empty(s), (uint32_t)(g / L::kOp - 1) & 1u, p.err, s_abort);
        if (!ok) break;
        mbar_arrive_expect_tx(full(s), 2u * kOpBox);
        tma_load_3d(sA(s), &wo_map, 64 * kb, mt * 64, 0, full(s));
        tma_load_3d(sB(s), &x_map, 64 * kb, nt * 64, 0, full(s));
        issued = g + 1;
      }
    } else if ((warp == 1 || warp == kW1) && lane == 0) {
      constexpr uint32_t kId = idesc_bf16(64, 64);
      const int w = warp == 1 ? 0 : 1;
      const uint32_t d = tmem + (uint32_t)(64 * w);
      bool ok = true;
      issued_mma = true;
      for (int kb = 0; kb < KB && ok; ++kb, ++g) {
        if ((kb & 1) != w) continue;
        const int s = g % L::kOp;
        ok = attn_wait(full(s), (uint32_t)(g / L::kOp) & 1u, p.err, s_abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dA = (uint32_t)smem_desc_sw128(sA(s)), dB = (uint32_t)smem_desc_sw128(sB(s));
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          tc_mma_f16(d, desc_sw128_at(dA, (uint32_t)k4 * 32u), desc_sw128_at(dB, (uint32_t)k4 * 32u), kId,
                     (kb >= 2 || k4) ? 1u : 0u);
        tc_commit(empty(s));
      }
      if (ok) tc_commit(acc_full);  // with no K block of this parity (K = 64) it arrives at once
    } else if (warp >= 2 && warp < 6) {
      // quadrant warp % 4: rows 16 qd .. 16 qd + 15 of the M = 64 accumulator
      // in lanes 0..15; D0 + D1 rounded to bf16 into a staging tile in shared
      // memory, then copied out row by row with coalesced stores (per-element
      // stores from the accumulator's layout cost ~2 us per unit)
      const int qd = warp & 3, et = threadIdx.x - 64;  // et: 0 .. 127
      bool ok = attn_wait(acc_full, (uint32_t)nu & 1u, p.err, s_abort);
      ok = named_barrier_and(2, 128, ok);  // the four warps decide together
      if (ok) {
        tc_fence_after();
        const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
        uint16_t *stg = reinterpret_cast<uint16_t *>(gbase + kOpStgOff<N>);  // [64][64]
#pragma unroll 1
        for (int c = 0; c < 64; c += 16) {
          uint32_t r[16], r1[16];
          tmem_ld_x16(trow + (uint32_t)c, r);
          if (KB > 1) tmem_ld_x16(trow + 64u + (uint32_t)c, r1);
          tc_wait_ld();
          // lanes l and l + 16 write the even and odd tokens of feature 16 qd + l
          uint16_t *srow = stg + (c + (lane >> 4)) * 64 + qd * 16 + (lane & 15);
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const float e =
                KB > 1 ? __fadd_rn(__uint_as_float(r[x]), __uint_as_float(r1[x])) : __uint_as_float(r[x]);
            const float o =
                KB > 1 ? __fadd_rn(__uint_as_float(r[x + 1]), __uint_as_float(r1[x + 1])) : __uint_as_float(r[x + 1]);
            const float o_hi = __shfl_xor_sync(kFull, o, 16);
            const __nv_bfloat16 hv = __float2bfloat16_rn(lane < 16 ? e : o_hi);
            srow[x * 64] = *reinterpret_cast<const uint16_t *>(&hv);
          }
        }
        named_barrier(2, 128);  // the tile is staged
        const int rows = min(64, S - nt * 64);
        uint16_t *ybase = p.y + (long long)nt * 64 * p.y_st + mt * 64;
        if ((reinterpret_cast<uintptr_t>(p.y) & 15u) == 0 && (p.y_st & 7) == 0) {
          for (int ch = et; ch < rows * 8; ch += 128) {
            const int row = ch >> 3, c16 = ch & 7;
            *reinterpret_cast<uint4 *>(ybase + (long long)row * p.y_st + c16 * 8) =
                *reinterpret_cast<const uint4 *>(stg + row * 64 + c16 * 8);
          }
        } else {
          for (int e = et; e < rows * 64; e += 128) ybase[(long long)(e >> 6) * p.y_st + (e & 63)] = stg[e];
        }
      }
    }
    ++nu;
    tc_fence_before();
    __syncthreads();  // the accumulator is drained before the next unit's MMAs overwrite it
    tc_fence_after();
    if (threadIdx.x == 0) misc[6] = (uint32_t)atomicAdd(p.ws, 1);
    __syncthreads();
    unit = misc[6];
  }
  // after an abort: this CTA's copies land and its committed MMAs complete
  if (threadIdx.x == 0)
    for (int q = issued - L::kOp < 0 ? 0 : issued - L::kOp; q < issued; ++q)
      mbar_wait(full(q % L::kOp), (uint32_t)(q / L::kOp) & 1u, p.err, kErrWaitTeardown);
  if (issued_mma) {  // every o_proj MMA of this thread completes before TMEM is freed
    const int w = warp == 1 ? 0 : 1;
    tc_commit(drain(w));
    mbar_wait(drain(w), 0u, p.err, kErrWaitTeardown);
  }
}

// The last CTA of the fused launch to finish leaves the workspace zeroed for
// the next call.
__device__ __forceinline__ void finish_workspace(const AttnParams &p) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.ws + 1, 1) == (int)gridDim.x - 1) {
      __threadfence();
      for (int k = 0; k <= p.ntiles; ++k) p.ws[2 + k] = 0;
      p.ws[0] = 0;
      p.ws[1] = 0;
      __threadfence();
    }
  }
}

}  // namespace

template <int N, bool FUSED>
__global__ void __launch_bounds__(AttnLayout<N, FUSED>::kThreads, AttnLayout<N, FUSED>::kCtas)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap kv_map,
                const __grid_constant__ CUtensorMap wv_map, const __grid_constant__ CUtensorMap wo_map,
                const __grid_constant__ CUtensorMap x_map) {
  using L = AttnLayout<N, FUSED>;
  constexpr int NR = L::kRope;
  constexpr int kAttnDbl = L::kDbl;
  constexpr int kAttnTile = L::kTile;
  constexpr uint32_t kDblBytes = L::kDblBytes, kRopeBytes = L::kRopeBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // swizzle atoms: 1024-byte aligned
  uint8_t *gbase = smem_raw + (sbase - raw);
  float *red = reinterpret_cast<float *>(gbase + L::red_off);
  int *lim_s = reinterpret_cast<int *>(gbase + L::lim_off);
  long long *orow_s = reinterpret_cast<long long *>(gbase + L::row_off);
  uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + L::misc_off);
  volatile int *s_abort = reinterpret_cast<volatile int *>(&misc[1]);
  const uint32_t bar0 = sbase + L::bar_off;
  auto full_db = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_db = [&](int s) { return bar0 + 8u * (uint32_t)(kAttnDbl + s); };
  auto full_r = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kAttnDbl + s); };
  auto empty_r = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kAttnDbl + NR + s); };
  const uint32_t s_full = bar0 + 8u * (uint32_t)(2 * kAttnDbl + 2 * NR);  // S^T of a tile is in TMEM
  const uint32_t s_free = s_full + 8u;   // the softmax warps have read it (one arrival per warp)
  const uint32_t p_full = s_full + 16u;  // P^T written, O rescaled (one arrival per softmax warp)
  const uint32_t o_full = s_full + 24u;  // a tile's O^T MMAs are complete
  const uint32_t q_full = s_full + 32u;  // an item's query rows are in shared memory
  const uint32_t q_free = s_full + 40u;  // the item's last S^T MMAs are done: Q may be replaced
  // every MMA of the S^T / O^T thread is complete (its teardown, once)
  const uint32_t drain_s = bar0 + 8u * (uint32_t)(L::kBars - 2), drain_pv = drain_s + 8u;
  // FUSED: item ring slots (full: published by the TMA lane; empty: every
  // taker has read it), W_V of a combine unit in shared memory, its MMAs done
  auto item_full = [&](int s) { return s_full + 48u + 8u * (uint32_t)s; };
  auto item_empty = [&](int s) { return s_full + 48u + 8u * (uint32_t)(kItemRing + s); };
  // W_V slots: full / free (a streamed quarter's MMAs are done), two each
  const uint32_t wv_full = s_full + 48u + 8u * (uint32_t)(2 * kItemRing);
  const uint32_t wv_free = wv_full + 16u;
  const uint32_t cmb_mma = wv_free + 16u;
  const uint32_t op_bar = cmb_mma + 8u;  // FUSED o_proj: full / empty per stage, accumulators full, drain[2]
  volatile uint32_t *ring = misc + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnDbl; ++s) {
      mbar_init(full_db(s), 1u);
      mbar_init(empty_db(s), 1u);
    }
    for (int s = 0; s < NR; ++s) {
      mbar_init(full_r(s), 1u);
      mbar_init(empty_r(s), 1u);
    }
    mbar_init(s_full, 1u);
    mbar_init(s_free, (uint32_t)kAttnSmx);
    mbar_init(p_full, (uint32_t)kAttnSmx);
    mbar_init(o_full, 1u);
    mbar_init(q_full, 1u);
    mbar_init(q_free, 1u);
    mbar_init(drain_s, 1u);
    mbar_init(drain_pv, 1u);
    if constexpr (FUSED) {
      for (int s = 0; s < kItemRing; ++s) {
        mbar_init(item_full(s), 1u);
        mbar_init(item_empty(s), (uint32_t)L::kItemTakers);
      }
      for (int b = 0; b < 4; ++b) mbar_init(wv_full + 8u * (uint32_t)b, 1u);  // wv_full[2], wv_free[2]
      mbar_init(cmb_mma, 1u);
      for (int s = 0; s < 2 * L::kOp + 3; ++s)  // the accumulators' full: both MMA threads commit
        mbar_init(op_bar + 8u * (uint32_t)s, s == 2 * L::kOp ? 2u : 1u);
    }
    misc[1] = 0u;
    misc[6] = 0xFFFFFFFFu;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc[0]), L::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  // Work items (request b, split r, head group g), the groups of one (b, r)
  // adjacent so that they read its cached rows from L2 together; CTA c takes
  // items c, c + grid, ...  Every role walks the same items and numbers the
  // tiles globally, so the rings and barriers run on across items.
  const int nitems = p.B * p.spr * p.groups;
  struct Item {
    int b, r, g, Lb, j0, jend, ntiles;
  };
  auto item_of = [&](int it) {
    Item I;
    I.g = it % p.groups;
    const int br = it / p.groups;
    I.r = br % p.spr;
    I.b = br / p.spr;
    int Lb = __ldg(p.kv_len + I.b);
    if (Lb < 0 || Lb > p.Lmax) {  // outside the cache tensor: recorded, clamped
      atomicCAS(p.err, 0, kErrKvLen);
      Lb = Lb < 0 ? 0 : p.Lmax;
    }
    I.Lb = Lb;
    const int C = (Lb + p.spr - 1) / p.spr;
    I.j0 = I.r * C;
    I.jend = min(I.j0 + C, Lb);
    I.ntiles = I.jend > I.j0 ? (I.jend - I.j0 + kAttnTile - 1) / kAttnTile : 0;
    return I;
  };
  // the query rows, the lengths and the cache come from earlier kernels
  // (and, FUSED, the workspace's last user)
  grid_dependency_wait();

  // The k-th item of this CTA: a fixed stride over the grid, or (FUSED) the
  // queue: the TMA lane draws it and publishes it in ring slot k % kItemRing,
  // the other roles read it there and release the slot.  An index >= nitems
  // ends the attention items.
  auto draw = [&](int k, bool &ok) -> int {  // TMA lane
    if constexpr (!FUSED) {
      return blockIdx.x + k * gridDim.x;
    } else {
      const int s = k % kItemRing;
      if (k >= kItemRing) ok = attn_wait(item_empty(s), (uint32_t)(k / kItemRing - 1) & 1u, p.err, s_abort);
      if (!ok) return nitems;
      const int it = atomicAdd(p.ws, 1);
      ring[s] = (uint32_t)it;
      mbar_arrive(item_full(s));
      return it;
    }
  };
  auto take = [&](int k, bool &ok) -> int {  // the other roles
    if constexpr (!FUSED) {
      return blockIdx.x + k * gridDim.x;
    } else {
      const int s = k % kItemRing;
      ok = ok && attn_wait(item_full(s), (uint32_t)(k / kItemRing) & 1u, p.err, s_abort);
      return ok ? (int)ring[s] : nitems;
    }
  };
  auto release = [&](int k) {  // once per taker
    if constexpr (FUSED) mbar_arrive(item_empty(k % kItemRing));
  };

  if (warp == 0) {
    // ---- TMA producer: per tile four double blocks, then the rope block ----
    if (lane == 0) {
      bool ok = true;
      int T = 0;                        // tiles started
      int issued_db = 0, issued_r = 0;  // double blocks / rope blocks whose copies were issued
      for (int k = 0; ok; ++k) {
        const int it = draw(k, ok);
        if (!ok) break;
        if (it >= nitems) {
          if constexpr (FUSED) misc[6] = (uint32_t)it;  // this CTA's first combine unit
          break;
        }
        const Item I = item_of(it);
        for (int t = 0; t < I.ntiles && ok; ++t, ++T) {
          const int y = I.j0 + t * kAttnTile;
          for (int c = 0; c < 4 && ok; ++c) {
            const int gb = 4 * T + c, s = gb % kAttnDbl;
            if (gb >= kAttnDbl) ok = attn_wait(empty_db(s), (uint32_t)(gb / kAttnDbl - 1) & 1u, p.err, s_abort);
            if (!ok) break;
            const uint32_t dst = sbase + L::dbl_off + (uint32_t)s * kDblBytes;
            mbar_arrive_expect_tx(full_db(s), kDblBytes);
            tma_load_3d(dst, &kv_map, 128 * c, y, I.b, full_db(s));
            tma_load_3d(dst + kDblBytes / 2, &kv_map, 128 * c + 64, y, I.b, full_db(s));
            issued_db = gb + 1;
          }
          if (!ok) break;
          const int s = T % NR;
          if (T >= NR) ok = attn_wait(empty_r(s), (uint32_t)(T / NR - 1) & 1u, p.err, s_abort);
          if (!ok) break;
          mbar_arrive_expect_tx(full_r(s), kRopeBytes);
          tma_load_3d(sbase + L::rope_off + (uint32_t)s * kRopeBytes, &kv_map, kD, y, I.b, full_r(s));
          issued_r = T + 1;
        }
      }
      // after an abort: every copy still in flight lands before the CTA exits
      // (bounded waits; on the normal path these phases are complete)
      for (int gb = issued_db - kAttnDbl < 0 ? 0 : issued_db - kAttnDbl; gb < issued_db; ++gb)
        mbar_wait(full_db(gb % kAttnDbl), (uint32_t)(gb / kAttnDbl) & 1u, p.err, kErrWaitTeardown);
      for (int t = issued_r - NR < 0 ? 0 : issued_r - NR; t < issued_r; ++t)
        mbar_wait(full_r(t % NR), (uint32_t)(t / NR) & 1u, p.err, kErrWaitTeardown);
    }
  } else if (warp == 1 || (L::kSplitMma && warp == kPvWarp)) {
    // ---- MMA issuers: warp 1 the S^T MMAs (and, one thread for both, the
    // O^T MMAs), warp kPvWarp the O^T MMAs when they have a thread of their
    // own ----
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kAttnTile, N);         // M = the tile's positions
      constexpr uint32_t kIdO = idesc_bf16(128, N) | (1u << 15);  // A = V^T, MN-major
      const uint32_t tS = tmem, tO = tmem + (uint32_t)N;
      const uint32_t dQ = (uint32_t)smem_desc_sw128(sbase + L::q_off);
      const uint32_t dP = (uint32_t)smem_desc_sw128(sbase + L::p_off);
      // S^T[j, m] = sum_k K[j][k] Q[m][k] of tile T (the t-th of item I)
      auto s_tile = [&](int T, int t, int ntiles) -> bool {
        if (T > 0 && !attn_wait(s_free, (uint32_t)(T - 1) & 1u, p.err, s_abort)) return false;
        // the four latent double blocks ...
        for (int c = 0; c < 4; ++c) {
          const int gb = 4 * T + c, s = gb % kAttnDbl;
          if (!attn_wait(full_db(s), (uint32_t)(gb / kAttnDbl) & 1u, p.err, s_abort)) return false;
          tc_fence_after();
          const uint32_t dK = (uint32_t)smem_desc_sw128(sbase + L::dbl_off + (uint32_t)s * kDblBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t box = (uint32_t)kk >> 2, k4 = (uint32_t)kk & 3u;
            tc_mma_f16(tS, desc_sw128_at(dK, box * (kDblBytes / 2) + k4 * 32u),
                       desc_sw128_at(dQ, (2u * c + box) * (N * 128u) + k4 * 32u), kIdS, (c | kk) ? 1u : 0u);
          }
        }
        // ... and the rope block
        const int sr = T % NR;
        if (!attn_wait(full_r(sr), (uint32_t)(T / NR) & 1u, p.err, s_abort)) return false;
        tc_fence_after();
        const uint32_t dR = (uint32_t)smem_desc_sw128(sbase + L::rope_off + (uint32_t)sr * kRopeBytes);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          tc_mma_f16(tS, desc_sw128_at(dR, (uint32_t)k4 * 32u),
                     desc_sw128_at(dQ, 8u * (N * 128u) + (uint32_t)k4 * 32u), kIdS, 1u);
        tc_commit(s_full);
        tc_commit(empty_r(sr));
        if (t == ntiles - 1) tc_commit(q_free);  // the next item's queries may replace these
        return true;
      };
      // O^T[d, m] += sum_j V^T[d][j] P^T[j, m] of tile T, once P(T) is
      // written and O rescaled (which also orders it after the previous
      // item's epilogue).  The double-block slots it frees were read by the
      // tile's S^T MMAs too, which completed before the softmax wrote P(T).
      auto pv_tile = [&](int T, int t) -> bool {
        if (!attn_wait(p_full, (uint32_t)T & 1u, p.err, s_abort)) return false;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t vbase = sbase + L::dbl_off + (uint32_t)((4 * T + c) % kAttnDbl) * kDblBytes;
#pragma unroll
          for (int ks = 0; ks < kAttnTile / 16; ++ks)  // 16 positions per step
            tc_mma_f16(tO + (uint32_t)(c * N), smem_desc_mn_sw128(vbase + (uint32_t)ks * 2048u, kDblBytes / 2),
                       desc_sw128_at(dP, ((uint32_t)ks >> 2) * (N * 128u) + ((uint32_t)ks & 3u) * 32u), kIdO,
                       (t | ks) ? 1u : 0u);
          tc_commit(empty_db((4 * T + c) % kAttnDbl));  // this latent chunk's slot is free once its MMAs are
        }
        tc_commit(o_full);
        return true;
      };
      bool ok = true;
      int T = 0, kq = 0;  // tiles, non-empty items
      if (!L::kSplitMma || warp == 1) {
        for (int k = 0; ok; ++k) {
          const int it = take(k, ok);
          if (!ok) break;
          release(k);
          if (it >= nitems) break;
          const Item I = item_of(it);
          if (I.ntiles == 0) continue;
          ok = attn_wait(q_full, (uint32_t)kq & 1u, p.err, s_abort);
          for (int t = 0; t < I.ntiles && ok; ++t, ++T) {
            ok = s_tile(T, t, I.ntiles);
            if constexpr (!L::kSplitMma) {
              if (ok) ok = pv_tile(T, t);
            }
          }
          ++kq;
        }
        // every MMA this thread issued completes before TMEM is freed (after
        // an abort too)
        tc_commit(drain_s);
        mbar_wait(drain_s, 0u, p.err, kErrWaitTeardown);
      } else {
        for (int k = 0; ok; ++k) {
          const int it = take(k, ok);
          if (!ok) break;
          release(k);
          if (it >= nitems) break;
          const Item I = item_of(it);
          for (int t = 0; t < I.ntiles && ok; ++t, ++T) ok = pv_tile(T, t);
        }
        tc_commit(drain_pv);
        mbar_wait(drain_pv, 0u, p.err, kErrWaitTeardown);
      }
    }
  } else if (warp == 2 + kAttnSmx) {
    // ---- query loader: an item's N rows (row m: token m / G, head g G + m % G;
    // padded rows zero) into the K-major swizzled Q tile, by cp.async ----
    bool ok = true;
    int kq = 0;
    const int qG = p.q * p.G;
    for (int k = 0; ok; ++k) {
      const int it = take(k, ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) release(k);
      if (it >= nitems) break;
      const Item I = item_of(it);
      if (I.ntiles == 0) continue;
      if (kq > 0) ok = attn_wait(q_free, (uint32_t)(kq - 1) & 1u, p.err, s_abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // row by row (token i, head g G + hh of the row kept incrementally: no
      // division per chunk), a lane per 16-byte chunk
      int i = 0, hh = 0;
      for (int m = 0; m < N; ++m) {
        const int h = I.g * p.G + hh;
        const bool live = m < qG && h < p.H;
        const uint4 *src = reinterpret_cast<const uint4 *>(p.qv + (long long)(I.b * p.q + i) * p.q_st +
                                                           (long long)h * p.q_sh);
        for (int ch = lane; ch < kAttnK / 8; ch += 32) {
          const uint32_t dst = sbase + L::q_off + (uint32_t)((ch >> 3) * (N * 128) + m * 128 + (((ch & 7) ^ (m & 7)) << 4));
          if (live)
            cp_async_16(dst, src + ch);
          else
            *reinterpret_cast<uint4 *>(gbase + (dst - sbase)) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (++hh == p.G) {
          hh = 0;
          ++i;
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
      ++kq;
    }
  } else {
    // ---- softmax warps 2 .. 2 + kAttnSmx - 1: TMEM lane quadrant warp % 4 (a
    // thread per position), query rows c0 .. c0 + NC - 1 of the N ----
    constexpr int NC = N / 2;                     // query rows per softmax warp
    constexpr uint32_t kSmxThreads = kAttnSmx * 32;
    const int qd = warp & 3;                      // TMEM lane quadrant
    const int c0 = ((warp - 2) >> 2) * NC;        // this warp's first query row
    // S^T holds position 32 qd + lane of a 128-position tile, or (M = 64)
    // position 16 qd + lane of a 64-position tile in lanes 0 .. 15; O^T row 32 qd + lane
    const bool has_pos = kAttnTile == 128 || lane < 16;
    const int pos = kAttnTile == 128 ? qd * 32 + lane : qd * 16 + (lane & 15);  // position within a tile
    const int dv = qd * 32 + lane;                // O^T row within a latent chunk
    const int ts = threadIdx.x - 64;              // 0 .. kSmxThreads - 1
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const int qG = p.q * p.G;
    const int S = p.B * p.q;
    const float kNegInf = __int_as_float(0xFF800000);
    constexpr float kLn2 = 0.6931471805599453f;
    // a column's reference max moves only when a tile's max exceeds it by more
    // than 2^8 (the weights then stay below 256): O is rescaled rarely
    constexpr float kSlack = 8.0f;
    // Every exit decision is taken by all softmax warps together (an AND over
    // the named barrier), so that no warp waits at a barrier another left.
    bool ok = true;
    int T = 0;  // tiles
    // FUSED: one arrival per 8-token tile the item's request covers, once
    // every softmax warp has written the item's o / lse
    auto arrive_tiles = [&](const Item &I) {
      if constexpr (FUSED) {
        named_barrier(1, kSmxThreads);
        if (ts == 0) {
          __threadfence();
          for (int k = (I.b * p.q) / kCmbTile; k <= (I.b * p.q + p.q - 1) / kCmbTile; ++k) atomicAdd(p.ws + 2 + k, 1);
        }
      }
    };
    for (int k = 0; ok; ++k) {
      bool got = true;
      const int it = take(k, got);
      __syncwarp();
      if (lane == 0 && got) release(k);
      // (also: the previous item's readers of lim_s / orow_s are done)
      ok = named_barrier_and(1, kSmxThreads, got);
      if (!ok || it >= nitems) break;
      const Item I = item_of(it);
      // per query row: the positions of this split it sees (counted from j0)
      // and its o / lse row (-1: a padded row)
      if (ts < N) {
        const int m = ts, i = m / p.G, h = I.g * p.G + (m - i * p.G);
        int lim = 0;
        long long row = -1;
        if (m < qG && h < p.H) {
          lim = min(I.jend, I.Lb - (p.q - 1 - i)) - I.j0;
          row = ((long long)I.r * S + (I.b * p.q + i)) * p.H + h;
        }
        lim_s[m] = lim < 0 ? 0 : lim;
        orow_s[m] = row;
      }
      named_barrier(1, kSmxThreads);
      if (I.ntiles == 0) {  // the split holds no position: lse -inf, o 0
        if (ts < N && orow_s[ts] >= 0) p.lse[orow_s[ts]] = kNegInf;
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          const long long row = orow_s[c0 + x];
          if (row >= 0)
#pragma unroll
            for (int c = 0; c < 4; ++c) p.o[row * kD + 128 * c + dv] = 0;
        }
        arrive_tiles(I);
        continue;
      }
      int lim[NC];
      float m_ref[NC], l_part[NC];  // reference max (log2 units), this position's share of the sums
#pragma unroll
      for (int x = 0; x < NC; ++x) {
        lim[x] = lim_s[c0 + x];
        m_ref[x] = kNegInf;
        l_part[x] = 0.0f;
      }
      for (int t = 0; t < I.ntiles; ++t, ++T) {
        bool got = ok && attn_wait(s_full, (uint32_t)T & 1u, p.err, s_abort);
        got = __all_sync(0xffffffffu, got);
        uint32_t sr[NC];
#pragma unroll
        for (int x = 0; x < NC; ++x) sr[x] = 0u;
        if (got) {
          tc_fence_after();
          if constexpr (NC == 16)
            tmem_ld_x16(trow + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[16]>(&sr[0]));
          else
            tmem_ld_x8(trow + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[8]>(&sr[0]));
          tc_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
        }
        // scores in log2 units, masked
        const int jr = t * kAttnTile + pos;
        float sc[NC];
        bool up = false;  // a score of this thread exceeds its column's reference by more than the slack
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          sc[x] = (has_pos && jr < lim[x]) ? __uint_as_float(sr[x]) * p.scale_log2 : kNegInf;
          up |= sc[x] > m_ref[x] + kSlack;
        }
        // After an item's first tile a column's reference rarely moves: one
        // barrier vote (every wait succeeded, no score above its reference +
        // slack) lets the warps take P = exp2(s - reference) at once -- the same
        // values the exchange below gives when no column moves
        const bool fast = t > 0 && named_barrier_and(1, kSmxThreads, got && !up);
        float alpha[NC];
        bool moved = false;
        if (fast) {
#pragma unroll
          for (int x = 0; x < NC; ++x) {
            alpha[x] = 1.0f;
            sc[x] = (sc[x] == kNegInf) ? 0.0f : ex2_approx(sc[x] - m_ref[x]);  // P
            l_part[x] = __fmaf_rn(l_part[x], 1.0f, sc[x]);
          }
        } else {
          // the tile's column max over its positions, exchanged through shared memory
          float *rd = red + (T & 1) * 4 * N;
#pragma unroll
          for (int x = 0; x < NC; ++x) {
            float mx = sc[x];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == x) rd[qd * N + c0 + x] = mx;
          }
          ok = named_barrier_and(1, kSmxThreads, got);
          if (!ok) break;
#pragma unroll
          for (int x = 0; x < NC; ++x) {
            const int m = c0 + x;
            const float tmax = fmaxf(fmaxf(rd[m], rd[N + m]), fmaxf(rd[2 * N + m], rd[3 * N + m]));
            const float mn = (tmax > m_ref[x] + kSlack) ? tmax : m_ref[x];
            alpha[x] = (mn == m_ref[x]) ? 1.0f : ex2_approx(m_ref[x] - mn);  // 0 when m_ref was -inf
            moved |= (alpha[x] != 1.0f) && (m_ref[x] != kNegInf);
            m_ref[x] = mn;
            sc[x] = (sc[x] == kNegInf) ? 0.0f : ex2_approx(sc[x] - mn);  // P
            l_part[x] = __fmaf_rn(l_part[x], alpha[x], sc[x]);
          }
          moved = __any_sync(0xffffffffu, moved);
        }
        // the previous tile's O^T MMAs are done before P and O are touched (a
        // failed wait is shared at the next barrier)
        if (T > 0) {
          ok = attn_wait(o_full, (uint32_t)(T - 1) & 1u, p.err, s_abort);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) continue;
          tc_fence_after();
        }
        // P^T row m, column pos (K-major, 128-byte swizzle, K blocks of 64 positions)
        if (has_pos) {
          uint8_t *pb = gbase + L::p_off + (pos >> 6) * (N * 128);
          const int x2 = (pos & 63) * 2;
#pragma unroll
          for (int x = 0; x < NC; ++x) {
            const int m = c0 + x;
            const __nv_bfloat16 v = __float2bfloat16_rn(sc[x]);
            *reinterpret_cast<__nv_bfloat16 *>(pb + m * 128 + (((x2 >> 4) ^ (m & 7)) << 4) + (x2 & 15)) = v;
          }
        }
        // a cached row past kv_len (inside the cache tensor) may hold anything:
        // its latent is zeroed (by one warp of the quadrant) so that 0 * it
        // stays 0 in O
        if (c0 == 0 && has_pos && I.j0 + jr >= I.Lb && I.j0 + jr < p.Lmax) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint8_t *rowp = gbase + L::dbl_off + (size_t)((4 * T + c) % kAttnDbl) * kDblBytes + pos * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              reinterpret_cast<uint4 *>(rowp)[k] = make_uint4(0u, 0u, 0u, 0u);
              reinterpret_cast<uint4 *>(rowp + kDblBytes / 2)[k] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        // a column whose reference max moved: its accumulated O^T scaled by alpha
        if (t > 0 && moved) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t ta = trow + (uint32_t)(N + c * N + c0);
            uint32_t ov[NC];
            if constexpr (NC == 16)
              tmem_ld_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
            else
              tmem_ld_x8(ta, *reinterpret_cast<uint32_t(*)[8]>(&ov[0]));
            tc_wait_ld();
#pragma unroll
            for (int x = 0; x < NC; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * alpha[x]);
            if constexpr (NC == 16)
              tmem_st_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
            else
              tmem_st_x8(ta, *reinterpret_cast<uint32_t(*)[8]>(&ov[0]));
          }
          tc_wait_st();
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) {  // left the tile loop early (or a late wait failed): shared, then stop
        named_barrier_and(1, kSmxThreads, false);
        break;
      }
      // the item's last O^T MMAs, then the column sums over the positions (fixed order)
      bool fin = attn_wait(o_full, (uint32_t)(T - 1) & 1u, p.err, s_abort);
      fin = __all_sync(0xffffffffu, fin);
      if (fin) tc_fence_after();
      float *rd = red + (T & 1) * 4 * N;
#pragma unroll
      for (int x = 0; x < NC; ++x) {
        float l = l_part[x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == x) rd[qd * N + c0 + x] = l;
      }
      ok = named_barrier_and(1, kSmxThreads, fin);
      if (!ok) break;
      float inv[NC];  // 1 / column sum; 0 where the row sees nothing
#pragma unroll
      for (int x = 0; x < NC; ++x) {
        const int m = c0 + x;
        const float l = (rd[m] + rd[N + m]) + (rd[2 * N + m] + rd[3 * N + m]);
        inv[x] = l > 0.0f ? rcp_approx(l) : 0.0f;  // rcp.approx.f32: a correctly rounded reciprocal costs ~0.4 us per item here
        if (qd == 0 && lane == x && orow_s[m] >= 0)
          p.lse[orow_s[m]] = l > 0.0f ? (m_ref[x] + lg2_approx(l)) * kLn2 : kNegInf;
      }
      // o[row][128 c + pos] for this warp's query rows: a warp writes 64 contiguous bytes
      // (the rows' addresses read from shared memory once, not after every TMEM load)
      uint16_t *orow[NC];
#pragma unroll
      for (int x = 0; x < NC; ++x) {
        const long long row = orow_s[c0 + x];
        orow[x] = row >= 0 ? p.o + row * kD + dv : nullptr;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[NC];
        const uint32_t ta = trow + (uint32_t)(N + c * N + c0);
        if constexpr (NC == 16)
          tmem_ld_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
        else
          tmem_ld_x8(ta, *reinterpret_cast<uint32_t(*)[8]>(&ov[0]));
        tc_wait_ld();
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          if (orow[x]) {
            const float v = (inv[x] != 0.0f) ? __uint_as_float(ov[x]) * inv[x] : 0.0f;
            const __nv_bfloat16 hv = __float2bfloat16_rn(v);
            orow[x][128 * c] = *reinterpret_cast<const uint16_t *>(&hv);
          }
        }
      }
      tc_fence_before();
      arrive_tiles(I);
    }
    // the next kernel on the stream may start its prologue
    grid_launch_dependents();
  }
  if constexpr (FUSED) {
    combine_phase<N>(p, wv_map, sbase, gbase, tmem, misc, s_abort, wv_full, wv_free, cmb_mma, nitems);
    if (p.n_out > 0) oproj_phase<N>(p, wo_map, x_map, sbase, gbase, tmem, misc, s_abort, op_bar);
    finish_workspace(p);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

// Query rows per CTA: every head when q H <= 32, else groups of 32 / q heads;
// the MMA's N is that rounded up to 16.
int attn_heads_per_cta(int q, int H) { return q * H <= 32 ? H : (32 / q > 0 ? 32 / q : 1); }
int attn_rows(int q, int H) { return ((q * attn_heads_per_cta(q, H) + 15) / 16) * 16; }
size_t attn_smem_bytes(int rows) { return 1024 + (rows <= 16 ? AttnLayout<16>::total : AttnLayout<32>::total); }
int attn_tile_positions(int rows, bool fused) {
  if (fused) return rows <= 16 ? AttnLayout<16, true>::kTile : AttnLayout<32, true>::kTile;
  return rows <= 16 ? AttnLayout<16, false>::kTile : AttnLayout<32, false>::kTile;
}
int attn_combine_tiles(int S) { return (S + kCmbTile - 1) / kCmbTile; }

template <int N, bool FUSED>
static cudaError_t launch_attn_n(const AttnParams &p, const CUtensorMap &map, const CUtensorMap &wv_map,
                                 const CUtensorMap &wo_map, const CUtensorMap &x_map, unsigned grid,
                                 cudaStream_t stream) {
  const size_t smem = 1024 + AttnLayout<N, FUSED>::total;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<N, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(AttnLayout<N, FUSED>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_kernel<N, FUSED>, p, map, wv_map, wo_map, x_map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Persistent: one or two CTAs per SM (the shared-memory plan fills an SM or
// half of one), at most one per work item.
cudaError_t launch_attn(const AttnParams &p, const CUtensorMap &map, int num_sms, cudaStream_t stream) {
  const long long items = (long long)p.B * p.spr * p.groups;
  if (items <= 0 || items >= (1LL << 31) || num_sms < 1) return cudaErrorInvalidValue;
  const int rows = ((p.q * p.G + 15) / 16) * 16;  // the host keeps q G <= 32
  if (rows > 32) return cudaErrorInvalidValue;
  const long long slots = (long long)num_sms * (rows <= 16 ? AttnLayout<16, false>::kCtas : AttnLayout<32, false>::kCtas);
  const unsigned grid = (unsigned)(items < slots ? items : slots);
  CUtensorMap none;
  std::memset(&none, 0, sizeof none);
  return rows <= 16 ? launch_attn_n<16, false>(p, map, none, none, none, grid, stream)
                    : launch_attn_n<32, false>(p, map, none, none, none, grid, stream);
}

// The fused attention + combine (+ o_proj): a persistent grid (two CTAs per SM
// for up to 16 query rows, else one) over the attention items, then the
// combine units (ntiles * H), then the o_proj units, all drawn from the
// workspace queue.
cudaError_t launch_attn_combine(const AttnParams &p, const CUtensorMap &map, const CUtensorMap &wv_map,
                                const CUtensorMap &wo_map, const CUtensorMap &x_map, int num_sms, cudaStream_t stream) {
  const long long work =
      (long long)p.B * p.spr * p.groups + (long long)p.ntiles * p.H + (p.n_out > 0 ? (long long)p.op_units : 0);
  if (work <= 0 || work >= (1LL << 31) || num_sms < 1 || !p.ws) return cudaErrorInvalidValue;
  if (p.n_out > 0 && (p.n_out % 64 || (p.H * kV) % 64 || !p.y)) return cudaErrorInvalidValue;
  const int rows = ((p.q * p.G + 15) / 16) * 16;
  if (rows > 32 || p.spr > 32) return cudaErrorInvalidValue;
  const long long slots = (long long)num_sms * (rows <= 16 ? AttnLayout<16, true>::kCtas : AttnLayout<32, true>::kCtas);
  const unsigned grid = (unsigned)(work < slots ? work : slots);
  return rows <= 16 ? launch_attn_n<16, true>(p, map, wv_map, wo_map, x_map, grid, stream)
                    : launch_attn_n<32, true>(p, map, wv_map, wo_map, x_map, grid, stream);
}

}  // namespace mla
