// kernel_attn_pair.cu -- the partial producer on 2-CTA clusters: the split-KV
// MLA decode attention of kernel_attn.cu with every cached row's 512 latents
// split over the two CTAs of a cluster.
//
// The definition is the one of kernel_attn.cu (the vLLM page
// "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back" names
// the producer, M1c, but does not print it): per (split, token, head)
// lse = ln sum_j exp(scale q.k_j) over the positions of the split the token
// sees, o = sum_j softmax_j latent_j in bf16; an empty split gives lse -inf,
// o 0.
//
// Why two CTAs: a 128-position tile is 144 KiB (576 bf16 per position), so one
// CTA holds barely more than one tile and its chain -- copies, S^T MMAs,
// softmax, PV MMAs -- runs in series.  Here CTA r of a cluster holds latents
// [256 r, 256 r + 256) of every tile (two double blocks, 64 KiB) and rank 1
// also the rope block: two to three tiles fit, and each CTA issues half of
// the MMAs.
//   * S^T: each CTA accumulates its part of the scores over its own
//     dimensions into one of two TMEM buffers; the softmax warps read it,
//     send it to the peer by st.async into a receive buffer (two slots,
//     completing on an mbarrier there) and add the peer's part: both CTAs
//     hold the same fp32 scores (one addition, commutative) and so compute
//     the same softmax, the same P^T and the same column sums.
//   * PV: each CTA accumulates O^T for its own 256 latents.  The MMA thread
//     issues the next tile's S^T before the previous tile's PV (the S buffer
//     is double), so the tensor core works on the next scores while the
//     softmax of the current tile runs.
//   * Each CTA writes its half of every o row; rank 0 writes lse.
// A receive slot is rewritten two tiles later, and the peer sends those
// bytes only after it has received all of this CTA's scores of the tile in
// between, which this CTA sends only after reading the slot -- so the slots
// need no release signal; the next phase of a slot's mbarrier is armed one
// tile ahead, before this CTA's sends that the peer's next send waits for.
// Every wait is bounded; a timeout records an error, the roles stop, the
// peer times out on its next exchange, and both meet at the closing cluster
// barrier before TMEM is freed.
//
// Measured on the 16-split decode step (64 requests x 12 heads, up to 4096
// positions): 135.9 us against 87.6 us for one CTA per item.  A tile here
// takes about 5.4 us against about 7 us, but every SM pair walks twice the
// tiles: the per-tile chain (scores, exchange, softmax, PV) is bound by its
// latencies, not by the bytes the split halves.  The library runs it on
// request only.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kPrTile = 128;      // positions per tile
constexpr int kPrSmx = 8;         // softmax warps: two per TMEM lane quadrant
constexpr int kPrThreads = (3 + kPrSmx) * 32;  // warp 0 TMA, warp 1 MMA, softmax warps, one query warp
constexpr uint32_t kPrDbl = 2u * kPrTile * 128u;  // 32 KiB: 128 positions x 128 latents
constexpr uint32_t kPrRope = kPrTile * 128u;      // 16 KiB
constexpr int kPrQBlocks = 5;     // a CTA's query K blocks: 4 of latents (+ the rope block on rank 1)

template <int N>
struct PairLayout {
  static constexpr int kSlots = (N == 16) ? 5 : 4;  // double-block slots (a tile needs 2)
  static constexpr int kRope = 2;
  static constexpr uint32_t dbl_off = 0;
  static constexpr uint32_t rope_off = dbl_off + kSlots * kPrDbl;
  static constexpr uint32_t q_off = rope_off + kRope * kPrRope;              // kPrQBlocks x [N x 128 B]
  static constexpr uint32_t p_off = q_off + kPrQBlocks * N * 128u;            // 2 K blocks of [N x 128 B]
  static constexpr uint32_t recv_off = p_off + 2u * N * 128u;                 // float [2][128][N]
  static constexpr uint32_t red_off = recv_off + 2u * kPrTile * N * 4u;       // float [2][4][N]
  static constexpr uint32_t lim_off = red_off + 2u * 4u * N * 4u;             // int [N]
  static constexpr uint32_t row_off = (lim_off + N * 4u + 7u) & ~7u;         // long long [N]
  static constexpr uint32_t bar_off = row_off + N * 8u;
  // full / empty per slot, full / empty per rope slot, then s_full[2],
  // s_free[2], p_full, o_full, q_full, q_free, x_full[2]
  static constexpr int kBars = 2 * kSlots + 2 * kRope + 10;
  static constexpr uint32_t misc_off = bar_off + kBars * 8u;  // TMEM base, abort flag
  static constexpr uint32_t total = misc_off + 16u;
  static constexpr uint32_t tmem_cols = (4 * N <= 64) ? 64u : 128u;  // S (2 N, double) + O (2 N)
  static constexpr uint32_t xbytes = kPrTile * N * 4u;               // one tile's partial scores
};
static_assert(PairLayout<16>::total + 1024 <= 227u * 1024u, "shared memory (N = 16)");
static_assert(PairLayout<32>::total + 1024 <= 227u * 1024u, "shared memory (N = 32)");

__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, int *err, volatile int *abort_flag) {
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

}  // namespace

template <int N>
__global__ void __launch_bounds__(kPrThreads, 1)
    attn_pair_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap kv_map) {
  using L = PairLayout<N>;
  constexpr int NS = L::kSlots, NR = L::kRope;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  float *red = reinterpret_cast<float *>(gbase + L::red_off);
  const float *recv = reinterpret_cast<const float *>(gbase + L::recv_off);
  int *lim_s = reinterpret_cast<int *>(gbase + L::lim_off);
  long long *orow_s = reinterpret_cast<long long *>(gbase + L::row_off);
  uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + L::misc_off);
  volatile int *s_abort = reinterpret_cast<volatile int *>(&misc[1]);
  const uint32_t bar0 = sbase + L::bar_off;
  auto full_db = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_db = [&](int s) { return bar0 + 8u * (uint32_t)(NS + s); };
  auto full_r = [&](int s) { return bar0 + 8u * (uint32_t)(2 * NS + s); };
  auto empty_r = [&](int s) { return bar0 + 8u * (uint32_t)(2 * NS + NR + s); };
  const uint32_t b2 = bar0 + 8u * (uint32_t)(2 * NS + 2 * NR);
  auto s_full = [&](int b) { return b2 + 8u * (uint32_t)b; };        // S^T part of a tile in TMEM buffer b
  auto s_free = [&](int b) { return b2 + 16u + 8u * (uint32_t)b; };  // buffer b read (one arrival per softmax warp)
  const uint32_t p_full = b2 + 32u;  // P^T written, O rescaled
  const uint32_t o_full = b2 + 40u;  // a tile's PV MMAs are complete
  const uint32_t q_full = b2 + 48u;  // an item's query dims are in shared memory
  const uint32_t q_free = b2 + 56u;  // the item's last S^T MMAs are done
  auto x_full = [&](int b) { return b2 + 64u + 8u * (uint32_t)b; };  // the peer's scores of a tile, receive slot b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full_db(s), 1u);
      mbar_init(empty_db(s), 1u);
    }
    for (int s = 0; s < NR; ++s) {
      mbar_init(full_r(s), 1u);
      mbar_init(empty_r(s), 1u);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1u);
      mbar_init(s_free(b), (uint32_t)kPrSmx);
      mbar_init(x_full(b), 1u);
    }
    mbar_init(p_full, (uint32_t)kPrSmx);
    mbar_init(o_full, 1u);
    mbar_init(q_full, 1u);
    mbar_init(q_free, 1u);
    mbar_arrive_expect_tx(x_full(0), L::xbytes);  // the first tile's scores from the peer
    misc[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc[0]), L::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before either signals the other's
  tc_fence_after();
  const uint32_t tmem = misc[0];

  // Work items (request b, split r, head group g), the groups of one (b, r)
  // adjacent; cluster c takes items c, c + clusters, ...; both CTAs walk the
  // same items and number the tiles globally.
  const int nitems = p.B * p.spr * p.groups;
  const int cid = (int)cluster_id_x(), ncl = (int)(gridDim.x >> 1);
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
    I.ntiles = I.jend > I.j0 ? (I.jend - I.j0 + kPrTile - 1) / kPrTile : 0;
    return I;
  };
  grid_dependency_wait();

  if (warp == 0) {
    // ---- TMA: this CTA's two latent double blocks of every tile (latents
    // 256 rank .. + 255), and on rank 1 the rope block ----
    if (lane == 0) {
      bool ok = true;
      int T = 0, issued_db = 0, issued_r = 0;
      for (int it = cid; it < nitems && ok; it += ncl) {
        const Item I = item_of(it);
        for (int t = 0; t < I.ntiles && ok; ++t, ++T) {
          const int y = I.j0 + t * kPrTile;
          for (int c = 0; c < 2 && ok; ++c) {
            const int gb = 2 * T + c, s = gb % NS;
            if (gb >= NS) ok = pair_wait(empty_db(s), (uint32_t)(gb / NS - 1) & 1u, p.err, s_abort);
            if (!ok) break;
            const uint32_t dst = sbase + L::dbl_off + (uint32_t)s * kPrDbl;
            const int x = 128 * (2 * (int)rank + c);
            mbar_arrive_expect_tx(full_db(s), kPrDbl);
            tma_load_3d(dst, &kv_map, x, y, I.b, full_db(s));
            tma_load_3d(dst + kPrDbl / 2, &kv_map, x + 64, y, I.b, full_db(s));
            issued_db = gb + 1;
          }
          if (!ok || rank == 0) continue;
          const int s = T % NR;
          if (T >= NR) ok = pair_wait(empty_r(s), (uint32_t)(T / NR - 1) & 1u, p.err, s_abort);
          if (!ok) break;
          mbar_arrive_expect_tx(full_r(s), kPrRope);
          tma_load_3d(sbase + L::rope_off + (uint32_t)s * kPrRope, &kv_map, kD, y, I.b, full_r(s));
          issued_r = T + 1;
        }
      }
      // after an abort: every copy still in flight lands before the CTA exits
      for (int gb = issued_db - NS < 0 ? 0 : issued_db - NS; gb < issued_db; ++gb)
        mbar_wait(full_db(gb % NS), (uint32_t)(gb / NS) & 1u, p.err, kErrWaitTeardown);
      for (int t = issued_r - NR < 0 ? 0 : issued_r - NR; t < issued_r; ++t)
        mbar_wait(full_r(t % NR), (uint32_t)(t / NR) & 1u, p.err, kErrWaitTeardown);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: S^T part of tile T, then the PV of tile T - 1 ----
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, N);
      constexpr uint32_t kIdO = idesc_bf16(128, N) | (1u << 15);  // A = V^T, MN-major
      const uint32_t tO = tmem + 2u * (uint32_t)N;
      const uint32_t dQ = (uint32_t)smem_desc_sw128(sbase + L::q_off);
      const uint32_t dP = (uint32_t)smem_desc_sw128(sbase + L::p_off);
      int last_s = -1, last_o = -1, last_q = -1;
      bool ok = true;
      int T = 0, kq = 0;
      int prev = -1;           // the tile whose PV is still to issue
      bool prev_first = false; // ... the first tile of its item (the accumulator restarts)
      auto pv = [&](int Tp, bool first) {
        ok = pair_wait(p_full, (uint32_t)Tp & 1u, p.err, s_abort);
        if (!ok) return;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int s = (2 * Tp + c) % NS;
          const uint32_t vbase = sbase + L::dbl_off + (uint32_t)s * kPrDbl;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // 16 positions per step
            tc_mma_f16(tO + (uint32_t)(c * N), smem_desc_mn_sw128(vbase + (uint32_t)ks * 2048u, kPrDbl / 2),
                       desc_sw128_at(dP, ((uint32_t)ks >> 2) * (N * 128u) + ((uint32_t)ks & 3u) * 32u), kIdO,
                       (!first || ks > 0) ? 1u : 0u);
          tc_commit(empty_db(s));  // this chunk's slot is free once its MMAs are
        }
        tc_commit(o_full);
        last_o = Tp;
      };
      for (int it = cid; it < nitems && ok; it += ncl) {
        const Item I = item_of(it);
        if (I.ntiles == 0) continue;
        ok = pair_wait(q_full, (uint32_t)kq & 1u, p.err, s_abort);
        for (int t = 0; t < I.ntiles && ok; ++t, ++T) {
          const int b = T & 1;
          if (T >= 2) ok = pair_wait(s_free(b), (uint32_t)((T >> 1) - 1) & 1u, p.err, s_abort);
          // S^T[j, m] over this CTA's dimensions: its two latent double blocks ...
          for (int c = 0; c < 2 && ok; ++c) {
            const int gb = 2 * T + c, s = gb % NS;
            ok = pair_wait(full_db(s), (uint32_t)(gb / NS) & 1u, p.err, s_abort);
            if (!ok) break;
            tc_fence_after();
            const uint32_t dK = (uint32_t)smem_desc_sw128(sbase + L::dbl_off + (uint32_t)s * kPrDbl);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t box = (uint32_t)kk >> 2, k4 = (uint32_t)kk & 3u;
              tc_mma_f16(tmem + (uint32_t)(b * N), desc_sw128_at(dK, box * (kPrDbl / 2) + k4 * 32u),
                         desc_sw128_at(dQ, (2u * c + box) * (N * 128u) + k4 * 32u), kIdS, (c | kk) ? 1u : 0u);
            }
          }
          if (!ok) break;
          // ... and on rank 1 the rope block
          if (rank == 1) {
            const int sr = T % NR;
            ok = pair_wait(full_r(sr), (uint32_t)(T / NR) & 1u, p.err, s_abort);
            if (!ok) break;
            tc_fence_after();
            const uint32_t dR = (uint32_t)smem_desc_sw128(sbase + L::rope_off + (uint32_t)sr * kPrRope);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              tc_mma_f16(tmem + (uint32_t)(b * N), desc_sw128_at(dR, (uint32_t)k4 * 32u),
                         desc_sw128_at(dQ, 4u * (N * 128u) + (uint32_t)k4 * 32u), kIdS, 1u);
            tc_commit(empty_r(sr));
          }
          tc_commit(s_full(b));
          last_s = T;
          if (t == I.ntiles - 1) {
            tc_commit(q_free);  // the next item's queries may replace these
            last_q = kq;
          }
          // the previous tile's PV (this item's or the last item's), once its
          // P^T is written and O rescaled
          if (prev >= 0) pv(prev, prev_first);
          prev = T;
          prev_first = (t == 0);
        }
        ++kq;
      }
      if (ok && prev >= 0) pv(prev, prev_first);
      // after an abort: the committed MMAs finish before TMEM is freed
      if (last_s >= 0) mbar_wait(s_full(last_s & 1), (uint32_t)(last_s >> 1) & 1u, p.err, kErrWaitTeardown);
      if (last_o >= 0) mbar_wait(o_full, (uint32_t)last_o & 1u, p.err, kErrWaitTeardown);
      if (last_q >= 0) mbar_wait(q_free, (uint32_t)last_q & 1u, p.err, kErrWaitTeardown);
    }
  } else if (warp == 2 + kPrSmx) {
    // ---- query loader: an item's N rows, this CTA's dimensions only (rank 0
    // latents 0..255: 4 K blocks; rank 1 latents 256..511 and the rope: 5) ----
    bool ok = true;
    int kq = 0;
    const int qG = p.q * p.G;
    const int nch = rank ? 40 : 32;  // 16-byte chunks of a row this CTA holds
    const int ch0 = rank ? 32 : 0;   // the first one's index in the 576-wide row
    for (int it = cid; it < nitems && ok; it += ncl) {
      const Item I = item_of(it);
      if (I.ntiles == 0) continue;
      if (kq > 0) ok = pair_wait(q_free, (uint32_t)(kq - 1) & 1u, p.err, s_abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      for (int e = lane; e < N * nch; e += 32) {
        const int m = e / nch, ch = e - m * nch;
        const int i = m / p.G, h = I.g * p.G + (m - i * p.G);
        const uint32_t dst = sbase + L::q_off + (uint32_t)((ch >> 3) * (N * 128) + m * 128 + (((ch & 7) ^ (m & 7)) << 4));
        if (m < qG && h < p.H)
          cp_async_16(dst, reinterpret_cast<const uint4 *>(p.qv + (long long)(I.b * p.q + i) * p.q_st +
                                                           (long long)h * p.q_sh) + ch0 + ch);
        else
          *reinterpret_cast<uint4 *>(gbase + (dst - sbase)) = make_uint4(0u, 0u, 0u, 0u);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
      ++kq;
    }
  } else {
    // ---- softmax warps 2 .. 9: TMEM lane quadrant warp % 4 (a thread per
    // position), query rows c0 .. c0 + NC - 1 ----
    constexpr int NC = N / 2;
    constexpr uint32_t kSmxThreads = kPrSmx * 32;
    const int qd = warp & 3;
    const int c0 = ((warp - 2) >> 2) * NC;
    const int pos = qd * 32 + lane;
    const int ts = threadIdx.x - 64;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const int qG = p.q * p.G;
    const int S = p.B * p.q;
    const float kNegInf = __int_as_float(0xFF800000);
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kSlack = 8.0f;
    // this thread's slot in a receive buffer, here and in the peer
    const uint32_t my_recv = sbase + L::recv_off + (uint32_t)(pos * N + c0) * 4u;
    const uint32_t peer_recv = mapa_shared(my_recv, peer);
    const uint32_t peer_x0 = mapa_shared(x_full(0), peer);
    bool ok = true;
    int T = 0;
    for (int it = cid; it < nitems && ok; it += ncl) {
      const Item I = item_of(it);
      named_barrier(1, kSmxThreads);  // the previous item's readers of lim_s / orow_s are done
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
      if (I.ntiles == 0) {  // the split holds no position: lse -inf, o 0 (this CTA's half)
        if (rank == 0 && ts < N && orow_s[ts] >= 0) p.lse[orow_s[ts]] = kNegInf;
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          const long long row = orow_s[c0 + x];
          if (row >= 0)
#pragma unroll
            for (int c = 0; c < 2; ++c) p.o[row * kD + 256 * (int)rank + 128 * c + pos] = 0;
        }
        continue;
      }
      int lim[NC];
      float m_ref[NC], l_part[NC];
#pragma unroll
      for (int x = 0; x < NC; ++x) {
        lim[x] = lim_s[c0 + x];
        m_ref[x] = kNegInf;
        l_part[x] = 0.0f;
      }
      for (int t = 0; t < I.ntiles; ++t, ++T) {
        const int b = T & 1;
        bool got = ok && pair_wait(s_full(b), (uint32_t)(T >> 1) & 1u, p.err, s_abort);
        got = __all_sync(0xffffffffu, got);
        uint32_t sr[NC];
#pragma unroll
        for (int x = 0; x < NC; ++x) sr[x] = 0u;
        if (got) {
          tc_fence_after();
          if constexpr (NC == 16)
            tmem_ld_x16(trow + (uint32_t)(b * N + c0), *reinterpret_cast<uint32_t(*)[16]>(&sr[0]));
          else
            tmem_ld_x8(trow + (uint32_t)(b * N + c0), *reinterpret_cast<uint32_t(*)[8]>(&sr[0]));
          tc_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free(b));
        }
        // exchange the partial scores: arm the other receive slot's next
        // phase (the next tile), then -- after every softmax thread of this
        // CTA has passed that point -- send this tile's part to the peer
        if (ts == 0) mbar_arrive_expect_tx(x_full(b ^ 1), L::xbytes);
        named_barrier(1, kSmxThreads);
        if (got) {
          const uint32_t dst = peer_recv + (uint32_t)b * (kPrTile * N * 4u);
          const uint32_t rb = peer_x0 + 8u * (uint32_t)b;
#pragma unroll
          for (int x = 0; x < NC; x += 4)
            st_async_v4(dst + 4u * (uint32_t)x, __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]),
                        __uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3]), rb);
        }
        got = got && pair_wait(x_full(b), (uint32_t)(T >> 1) & 1u, p.err, s_abort);
        got = __all_sync(0xffffffffu, got);
        // scores in log2 units, masked; the tile's column max over 128 positions
        const int jr = t * kPrTile + pos;
        float sc[NC];
        float *rd = red + (T & 1) * 4 * N;
        const float *pr = recv + b * (kPrTile * N) + pos * N + c0;
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          const float s_tot = __fadd_rn(__uint_as_float(sr[x]), got ? pr[x] : 0.0f);
          sc[x] = (jr < lim[x]) ? s_tot * p.scale_log2 : kNegInf;
          float mx = sc[x];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == x) rd[qd * N + c0 + x] = mx;
        }
        ok = named_barrier_and(1, kSmxThreads, got);
        if (!ok) break;
        float alpha[NC];
        bool moved = false;
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          const int m = c0 + x;
          const float tmax = fmaxf(fmaxf(rd[m], rd[N + m]), fmaxf(rd[2 * N + m], rd[3 * N + m]));
          const float mn = (tmax > m_ref[x] + kSlack) ? tmax : m_ref[x];
          alpha[x] = (mn == m_ref[x]) ? 1.0f : ex2_approx(m_ref[x] - mn);
          moved |= (alpha[x] != 1.0f) && (m_ref[x] != kNegInf);
          m_ref[x] = mn;
          sc[x] = (sc[x] == kNegInf) ? 0.0f : ex2_approx(sc[x] - mn);
          l_part[x] = __fmaf_rn(l_part[x], alpha[x], sc[x]);
        }
        moved = __any_sync(0xffffffffu, moved);
        // the previous tile's PV MMAs are done before P and O are touched
        if (T > 0) {
          ok = pair_wait(o_full, (uint32_t)(T - 1) & 1u, p.err, s_abort);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) continue;
          tc_fence_after();
        }
        {
          uint8_t *pb = gbase + L::p_off + (pos >> 6) * (N * 128);
          const int x2 = (pos & 63) * 2;
#pragma unroll
          for (int x = 0; x < NC; ++x) {
            const int m = c0 + x;
            const __nv_bfloat16 v = __float2bfloat16_rn(sc[x]);
            *reinterpret_cast<__nv_bfloat16 *>(pb + m * 128 + (((x2 >> 4) ^ (m & 7)) << 4) + (x2 & 15)) = v;
          }
        }
        // a cached row past kv_len may hold anything: this CTA's latents of it
        // are zeroed so that 0 * it stays 0 in O
        if (c0 == 0 && I.j0 + jr >= I.Lb && I.j0 + jr < p.Lmax) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint8_t *rowp = gbase + L::dbl_off + (size_t)((2 * T + c) % NS) * kPrDbl + pos * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              reinterpret_cast<uint4 *>(rowp)[k] = make_uint4(0u, 0u, 0u, 0u);
              reinterpret_cast<uint4 *>(rowp + kPrDbl / 2)[k] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        if (t > 0 && moved) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t ta = trow + (uint32_t)(2 * N + c * N + c0);
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
      if (!ok) {
        named_barrier_and(1, kSmxThreads, false);
        break;
      }
      // the item's last PV MMAs, then the column sums (fixed order)
      bool fin = pair_wait(o_full, (uint32_t)(T - 1) & 1u, p.err, s_abort);
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
      float inv[NC];
#pragma unroll
      for (int x = 0; x < NC; ++x) {
        const int m = c0 + x;
        const float l = (rd[m] + rd[N + m]) + (rd[2 * N + m] + rd[3 * N + m]);
        inv[x] = l > 0.0f ? rcp_approx(l) : 0.0f;
        if (rank == 0 && qd == 0 && lane == x && orow_s[m] >= 0)
          p.lse[orow_s[m]] = l > 0.0f ? (m_ref[x] + lg2_approx(l)) * kLn2 : kNegInf;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ov[NC];
        const uint32_t ta = trow + (uint32_t)(2 * N + c * N + c0);
        if constexpr (NC == 16)
          tmem_ld_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(&ov[0]));
        else
          tmem_ld_x8(ta, *reinterpret_cast<uint32_t(*)[8]>(&ov[0]));
        tc_wait_ld();
#pragma unroll
        for (int x = 0; x < NC; ++x) {
          const long long row = orow_s[c0 + x];
          if (row >= 0) {
            const float v = (inv[x] != 0.0f) ? __uint_as_float(ov[x]) * inv[x] : 0.0f;
            const __nv_bfloat16 hv = __float2bfloat16_rn(v);
            p.o[row * kD + 256 * (int)rank + 128 * c + pos] = *reinterpret_cast<const uint16_t *>(&hv);
          }
        }
      }
      tc_fence_before();
    }
    grid_launch_dependents();
  }
  // both CTAs are done with each other's shared memory before either exits
  tc_fence_before();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

template <int N>
static cudaError_t launch_pair_n(const AttnParams &p, const CUtensorMap &map, int num_sms, cudaStream_t stream) {
  const size_t smem = 1024 + PairLayout<N>::total;
  cudaError_t e = cudaFuncSetAttribute(attn_pair_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPrThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // as many clusters as can be resident at once (an SM pair each), at most
  // one per work item
  cfg.gridDim = dim3((unsigned)(2 * (num_sms / 2)), 1, 1);
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, attn_pair_kernel<N>, &cfg) != cudaSuccess || max_clusters < 1)
    max_clusters = num_sms / 2;
  const long long items = (long long)p.B * p.spr * p.groups;
  const long long clusters = items < max_clusters ? items : max_clusters;
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  e = cudaLaunchKernelEx(&cfg, attn_pair_kernel<N>, p, map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_pair(const AttnParams &p, const CUtensorMap &map, int num_sms, cudaStream_t stream) {
  const long long items = (long long)p.B * p.spr * p.groups;
  if (items <= 0 || items >= (1LL << 31) || num_sms < 2) return cudaErrorInvalidValue;
  const int rows = ((p.q * p.G + 15) / 16) * 16;
  if (rows > 32) return cudaErrorInvalidValue;
  return rows <= 16 ? launch_pair_n<16>(p, map, num_sms, stream) : launch_pair_n<32>(p, map, num_sms, stream);
}

}  // namespace mla
