// kernel_tc.cu -- fused tensor-core kernel of the MLA decode post-attention
// stage for sm_103a: LSE combine -> bf16 (or MXFP4) latents in shared memory
// -> tcgen05 W_UV GEMM with the accumulator in TMEM -> gate epilogue.
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
// token tile stays small enough for decode batches.  bf16 W_V: 32 MMAs of
// kind::f16 (K = 16).  MXFP4 W_V: W_V stays as packed E2M1 codes (32 KiB),
// the latents are quantised straight to E2M1 codes + E8M0 block scales, and
// 8 MMAs of kind::mxf4.block_scale (K = 64) read both operands' scales from
// TMEM, where tcgen05.cp puts them: for V row m, lane m, column
// (group base + m / 32); for token n, lane 32q + n in every lane quadrant q;
// each 32-bit word holds the scales of four consecutive 32-wide K blocks.
//
// Warp roles (16 warps, all alike; 8 for MXFP4 with 16-token tiles): each
// warp combines its tokens of a unit into the latent buffer, then runs the
// epilogue of the unit two back (TMEM -> registers, bf16(acc) * gate ->
// core).  The warp that completes a unit's latents last (per-stage monotonic
// arrival counters) issues that unit's MMAs from one thread and commits them
// to an mbarrier -- or, unless every warp drains the unit at once (the last
// of a head or of the CTA), only marks it pending, and the first warp to
// reach its next finish claims and issues it, off the slowest warp's path;
// either way the issue follows every warp's drain of that TMEM buffer's
// previous use.  At a head change every warp first waits for the
// previous head's MMAs, then copies W_V[h] (and, for MXFP4, its scales) into
// shared memory.  Latent buffers and TMEM accumulators have three stages, so
// the combine of unit i overlaps the MMA of unit i-1 and the epilogue of
// unit i-2.  A warp issues a batch of partial-row loads before merging the
// previous one, loads LSE values three units ahead, and prefetches into L2
// the gate lines of the unit it drains next.  Launched with programmatic
// stream serialization: set-up and the first head's W_V copy overlap the
// previous kernel's tail; everything that reads o, lse or gate, or writes,
// follows griddepcontrol.wait.  Offsets are 32-bit when the host found every
// dereferenced offset below 2^32 (the O32 instances), else 64-bit.
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


// Shared memory and TMEM plan of one CTA.
struct TcLayout {
  uint32_t a_bytes, b_off, b_bytes, sfa_off, sfb_off, epi_off, bar_off, total;
  uint32_t tmem_cols, sfa_col, sfb_col;
};
// Pipeline stages (latent buffers, TMEM accumulators, latent scale buffers):
// the epilogue of unit i - (stages - 1) runs after unit i is merged, giving
// the MMAs of a unit a full unit of slack.
__host__ __device__ constexpr int tc_stages(int, int) { return 3; }
// bf16 W_V with 32-token tiles has no room for the 8 KiB epilogue staging
// area: its epilogue stages in the warp's own rows of the latent buffer of
// the unit being drained (that unit's MMAs are complete, and only this warp
// rewrites those rows, at its next finish of that stage).
__host__ __device__ constexpr bool tc_epi_in_latents(int BN, int WFMT) { return WFMT == 0 && BN == 32; }
__host__ __device__ constexpr TcLayout tc_layout(int BN, int WFMT, int NW) {
  TcLayout L{};
  const uint32_t st = (uint32_t)tc_stages(BN, WFMT);
  L.a_bytes = WFMT ? 128u * 256u : 128u * 1024u;           // W_V[h]: E2M1 codes or bf16
  L.b_off = L.a_bytes;
  L.b_bytes = WFMT ? (uint32_t)BN * 256u : (uint32_t)BN * 1024u;  // one latent buffer
  L.sfa_off = L.b_off + st * L.b_bytes;
  L.sfb_off = L.sfa_off + (WFMT ? 2048u : 0u);
  L.epi_off = L.sfb_off + (WFMT ? st * 2048u : 0u);
  L.bar_off = L.epi_off + (tc_epi_in_latents(BN, WFMT) ? 0u : (uint32_t)NW * (4u * (uint32_t)BN / (uint32_t)NW) * 64u);
  L.total = L.bar_off + 128u;
  // TMEM: `st` fp32 accumulators of BN columns; MXFP4 adds a 16-column region
  // for W_V's scales and one per stage for the latents' scales
  const uint32_t acc = st * (uint32_t)BN;
  L.sfa_col = (acc + 15u) & ~15u;
  L.sfb_col = L.sfa_col + 16u;
  const uint32_t need = WFMT ? L.sfb_col + 16u * st : acc;
  uint32_t cols = 32u;
  while (cols < need) cols *= 2u;
  L.tmem_cols = cols;
  return L;
}
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int *err, int code,
                                              volatile int *abort_flag, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      atomicCAS(err, 0, code);
      *abort_flag = 1;
      return false;
    }
  }
}

}  // namespace

template <int BN, int WFMT, int NW, bool O32, bool HR, bool RT>
__global__ void __launch_bounds__(NW * 32, 16 / NW)
    tc_kernel(const __grid_constant__ KParams p) {
  constexpr int kWorkers = NW;             // all warps combine, drain and (one of them) issue
  constexpr int NT = NW * 32;              // threads
  // HR (half rows; 8-token tiles for split-KV decode steps with few units): a
  // unit is BN / 2 tokens and two warps share a token, each merging one half
  // of its 512 latents, so twice as many CTAs share the partial rows.  The
  // MMA keeps N = BN: the latent rows of the absent tokens are never written,
  // and their accumulator columns are computed from whatever those rows hold
  // and never stored.  (The HR branches below are `if constexpr`, so the
  // other instances compile exactly as without them: this kernel's speed was
  // measured to depend on the code generated for its loop.)
  constexpr int UT = HR ? BN / 2 : BN;     // tokens per unit
  constexpr int TPW = HR ? 1 : BN / NW;    // tokens per warp per unit
  constexpr int NCH = HR ? 1 : 2;          // 16-byte chunks per lane and partial row
  constexpr int JB = HR ? 8 : 4 / TPW;     // partials per batch (8 x 16 B per lane)
  constexpr int CPW = 4 * BN / NW;         // TMEM columns each warp drains
  constexpr TcLayout L = tc_layout(BN, WFMT, NW);
  constexpr uint32_t kCols = L.tmem_cols;
  constexpr int ST = tc_stages(BN, WFMT);
  static_assert(TPW >= 1 && BN % NW == 0 && JB >= 1 && NW % 4 == 0, "tile must split over the warps");
  static_assert(!HR || NW == 2 * UT, "half rows: two warps per token");
  static_assert(CPW == 4 || CPW == 8 || CPW == 16, "epilogue drains 4, 8 or 16 columns per warp");
  static_assert(!(RT && HR), "runtime tiles use whole rows");
  // RT (runtime tile): a unit is p.tile <= BN tokens; the MMA keeps N = BN and
  // the slots past p.tile are empty (their latent rows zero, their columns
  // never stored): a slot index past the unit gets a token index no token
  // has, so every `t < p.S` test below leaves it out.  Decode batches use it
  // to give every SM one unit.  Other instances: tile * BN + slot.
  auto tok = [&](int tile, int slot) -> int {
    if constexpr (RT)
      return slot < p.tile ? tile * p.tile + slot : 0x7FFFFFFF;
    else
      return tile * BN + slot;
  };

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;    // 1024-byte aligned (swizzle atoms)
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t sA = sbase;
  const uint32_t sB0 = sbase + L.b_off;
  uint8_t *gA = gbase;
  uint8_t *gB0 = gbase + L.b_off;
  uint8_t *gSFA = gbase + L.sfa_off;   // MXFP4: W_V scale atoms (4 x 512 B)
  uint8_t *gSFB0 = gbase + L.sfb_off;  // MXFP4: latent scale atoms, per buffer
  // per-warp epilogue staging: CPW tokens x 32 V rows of bf16
  uint16_t *gE = reinterpret_cast<uint16_t *>(gbase + L.epi_off);
  uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + L.bar_off);
  uint32_t *misc = reinterpret_cast<uint32_t *>(bars + 4);
  // misc[0] TMEM base, misc[1] abort flag, misc[4..4+ST) arrival counters,
  // misc[8..8+ST) pending issues (unit + 1 of a complete unit whose MMAs wait
  // for a claim; 0 none), misc[12..12+ST) last unit issued on each stage (+1)
  volatile int *s_abort = reinterpret_cast<volatile int *>(&misc[1]);
  const uint32_t bar_mma0 = smem_u32(&bars[0]);  // +8*b, one per stage
  const uint32_t cnt0 = smem_u32(&misc[4]);      // +4*b
  const uint32_t pend0 = smem_u32(&misc[8]);     // +4*b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < ST; ++b) mbar_init(bar_mma0 + 8 * b, 1u);
    for (int k = 1; k < 12 + ST; ++k) misc[k] = 0u;
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
  // the next launch on the stream may begin its prologue as this grid's CTAs
  // finish (its dependent work waits for this grid's completion)
  grid_launch_dependents();
  constexpr bool kGatePrefetch = true;
  constexpr bool kTwoBatchLoop = true;
  // deferred MMA issue (see finish): off the slowest warp's path (large
  // batch bf16 358 -> 342 us, MXFP4 309 -> 304 us)
  constexpr bool kDeferIssue = true;

  // Element offset a * sa + b * sb + c * sc: unsigned 32-bit arithmetic when
  // the host found every dereferenced offset below 2^32 (O32; addresses formed
  // for tokens past S may wrap but are never dereferenced), else 64-bit.
  auto off3 = [](int a, long long sa, int b, long long sb, int c, long long sc) -> unsigned long long {
    if constexpr (O32)
      return (uint32_t)((uint32_t)a * (uint32_t)sa + (uint32_t)b * (uint32_t)sb + (uint32_t)c * (uint32_t)sc);
    else
      return (unsigned long long)((long long)a * sa + (long long)b * sb + (long long)c * sc);
  };
  auto off1 = [](int a, long long sa) -> unsigned long long {
    if constexpr (O32)
      return (uint32_t)((uint32_t)a * (uint32_t)sa);
    else
      return (unsigned long long)((long long)a * sa);
  };

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
  int np2 = 1;                       // n rounded up to a power of two (<= SEG)
  while (np2 < n) np2 <<= 1;

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
  // L2 prefetch of the gate lines a later epilogue of unit c reads (one
  // 128-byte-aligned line per 64-byte token segment of this warp)
  auto prefetch_gate = [&](const Cur &c) {
    constexpr int kRounds = (CPW + 7) / 8;
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      const int e = rd * 8 + (lane >> 2);
      if constexpr (HR) {
        const int t = c.tile * UT + ws * CPW + e;
        if ((lane & 3) == 0 && e < CPW && ws * CPW + e < UT && t < p.S)
          prefetch_l2_line(p.gate + off3(t, Wrow, c.h, kV, 1, wq * 32));
      } else {
        const int t = tok(c.tile, ws * CPW + e);
        if ((lane & 3) == 0 && e < CPW && t < p.S) prefetch_l2_line(p.gate + off3(t, Wrow, c.h, kV, 1, wq * 32));
      }
    }
  };

  auto epilogue = [&](int j, const Cur &c) -> bool {
    const int bj = j % ST;
    // staging: CPW tokens x 32 V rows of bf16 (512 bytes), addressed in
    // 128-byte pieces: the warp's own area, or (see tc_epi_in_latents) the
    // K blocks 0..3 of the warp's first latent row in stage bj
    uint8_t *const st_base = tc_epi_in_latents(BN, WFMT)
                                 ? gB0 + (size_t)bj * L.b_bytes + (size_t)(warp * TPW) * 128u
                                 : reinterpret_cast<uint8_t *>(gE + warp * (CPW * 32));
    constexpr uint32_t kPiece = tc_epi_in_latents(BN, WFMT) ? (uint32_t)BN * 128u : 128u;
    auto stg = [&](uint32_t o) { return st_base + (o >> 7) * kPiece + (o & 127u); };
    // lane -> (token e0 + lane/4, 8 consecutive V rows)
    constexpr int kRounds = (CPW + 7) / 8;
    const int v8 = (lane & 3) * 8;
    uint4 g[kRounds];
    long long off[kRounds];
    bool act[kRounds];
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      const int e = rd * 8 + (lane >> 2);
      const int t = HR ? c.tile * UT + ws * CPW + e : tok(c.tile, ws * CPW + e);
      if constexpr (HR)
        act[rd] = e < CPW && ws * CPW + e < UT && t < p.S;
      else
        act[rd] = e < CPW && t < p.S;
      off[rd] = (long long)off3(t, Wrow, c.h, kV, 1, wq * 32 + v8);
      g[rd] = act[rd] ? __ldg(reinterpret_cast<const uint4 *>(p.gate + off[rd])) : make_uint4(0, 0, 0, 0);
    }
    bool ok = wait_or_abort(bar_mma0 + 8 * bj, (uint32_t)(j / ST) & 1u, p.err, kErrWaitMma, s_abort, p.wait_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    tc_fence_after();
    uint32_t r[CPW];
    const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(bj * BN + ws * CPW);
    if constexpr (CPW == 16) {
      tmem_ld_x16(taddr, r);
    } else if constexpr (CPW == 8) {
      tmem_ld_x8(taddr, r);
    } else {
      tmem_ld_x4(taddr, r);
    }
    tc_wait_ld();
    tc_fence_before();
#pragma unroll
    for (int x = 0; x < CPW; ++x) {
      const __nv_bfloat16 a = __float2bfloat16_rn(__uint_as_float(r[x]));
      *reinterpret_cast<uint16_t *>(stg((uint32_t)(x * 64 + 2 * lane))) = *reinterpret_cast<const uint16_t *>(&a);
    }
    __syncwarp();
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      if (act[rd]) {
        const int e = rd * 8 + (lane >> 2);
        const uint4 a = *reinterpret_cast<const uint4 *>(stg((uint32_t)(e * 64 + 2 * v8)));
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, gg[4] = {g[rd].x, g[rd].y, g[rd].z, g[rd].w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = mul_bf16x2(aa[q], gg[q]);  // bf16(acc) * gate, one rounding
        *reinterpret_cast<uint4 *>(p.out + off[rd]) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncwarp();
    return true;
  };

  // LSE values and weights are packed one (token, partial) per lane: the
  // warp's TPW tokens take SEG = 32 / TPW lanes each, lane tk * SEG + j holding
  // partial j of token tk (n <= SEG), so one warp-wide pass serves all of them.
  constexpr int SEG = 32 / TPW;
  const int my_tk = lane / SEG, my_j = lane % SEG;

  // This lane's LSE (-inf past n or past S; sanitised when used).
  auto load_lse = [&](const Cur &c, float &lv) {
    const int t = HR ? c.tile * UT + (warp >> 1) + my_tk : tok(c.tile, warp * TPW + my_tk);
    lv = kNegInf;
    if (!pass && t < p.S && my_j < n) {
      const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
      lv = __ldg(p.lse + off3(r0 + my_j, p.l_sp, t, p.l_st, c.h, p.l_sh));
    }
  };

  // L2 prefetch of a unit's live partial rows: each lane prefetches its
  // partial's 1-KiB row when its LSE is finite (the rows the merge will
  // read), so the merge's own loads hit L2.  Used with bf16 W_V, where the
  // merge is latency-bound; with MXFP4 W_V (more arithmetic per row between
  // loads) it measured slower and is left out.
  auto prefetch_rows = [&](const Cur &c, float lv) {
    if (WFMT != 0) return;
    const int t = HR ? c.tile * UT + (warp >> 1) + my_tk : tok(c.tile, warp * TPW + my_tk);
    const bool live = pass ? (my_j == 0 && t < p.S) : isfinite(lv);
    if (live) {
      const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
      if constexpr (HR)  // this warp's half of the row
        prefetch_l2_bulk(p.o + off3(t, p.o_st, c.h, p.o_sh, r0 + my_j, p.o_sp) + (warp & 1) * (kD / 2), kD);
      else
        prefetch_l2_bulk(p.o + off3(t, p.o_st, c.h, p.o_sh, r0 + my_j, p.o_sp),
                         kD * 2);
    }
  };

  // This lane's weight (LSE rule; one partial passes through).
  auto weights_of = [&](float lv, float &wg) {
    if (pass) {
      wg = (my_j == 0) ? 1.0f : 0.0f;
      return;
    }
    const float l = sane(lv);
    float m = l;  // max over the token's lanes (np2 <= SEG; lanes past n hold -inf)
    for (int s = 1; s < np2; s <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    if (m == kNegInf) m = 0.0f;
    const float e = (my_j < n) ? ex2_approx(__fmul_rn(__fsub_rn(l, m), kLog2e)) : 0.0f;
    float Z = 0.0f;  // sequential fp32 sum in partial order
    const int seg0 = my_tk * SEG;
    for (int j = 0; j < n; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, seg0 + j));
    const float inv = (Z == 0.0f) ? 0.0f : rcp_approx(Z);
    wg = (e == 0.0f) ? 0.0f : __fmul_rn(e, inv);
  };

  using Buf = uint4[JB][TPW][NCH];
  using Wts = float[JB][TPW];

  // Issue the loads of one batch: unit at cursor c, partials j0 .. j0+JB-1
  // (rows of zero weight and tokens past S are not read).
  auto issue = [&](const Cur &c, int j0, Buf &buf, Wts &w, float wg) {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      const int t = HR ? c.tile * UT + (warp >> 1) + tk : tok(c.tile, warp * TPW + tk);
      const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
      const uint16_t *base = p.o + off3(t, p.o_st, c.h, p.o_sh, r0 + j0, p.o_sp);
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        w[jj][tk] = __shfl_sync(0xffffffffu, wg, tk * SEG + j0 + jj);  // 0 past n
        if (w[jj][tk] != 0.0f && t < p.S) {
          const uint4 *row = reinterpret_cast<const uint4 *>(base + off1(jj, p.o_sp));
          if constexpr (HR) {
            buf[jj][tk][0] = __ldcs(row + (warp & 1) * 32 + lane);
          } else {
            buf[jj][tk][0] = __ldcs(row + lane);
            buf[jj][tk][1] = __ldcs(row + lane + 32);
          }
        } else {
          if constexpr (HR)
            buf[jj][tk][0] = make_uint4(0, 0, 0, 0);
          else
            buf[jj][tk][0] = buf[jj][tk][1] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  };

  // Partials j0 .. j0+JB-1 of a unit, for every valid token, without weights.
  auto issue_blind = [&](const Cur &c, int j0, Buf &buf) {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      const int t = HR ? c.tile * UT + (warp >> 1) + tk : tok(c.tile, warp * TPW + tk);
      const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
      const uint16_t *base = p.o + off3(t, p.o_st, c.h, p.o_sh, r0 + j0, p.o_sp);
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        if (j0 + jj < n && t < p.S) {
          const uint4 *row = reinterpret_cast<const uint4 *>(base + off1(jj, p.o_sp));
          if constexpr (HR) {
            buf[jj][tk][0] = __ldcs(row + (warp & 1) * 32 + lane);
          } else {
            buf[jj][tk][0] = __ldcs(row + lane);
            buf[jj][tk][1] = __ldcs(row + lane + 32);
          }
        } else {
          if constexpr (HR)
            buf[jj][tk][0] = make_uint4(0, 0, 0, 0);
          else
            buf[jj][tk][0] = buf[jj][tk][1] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  };

  uint64_t acc[TPW][4 * NCH];  // fp32 pairs: elements (2q, 2q+1) of chunk q/4
  auto clear_acc = [&]() {
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk)
#pragma unroll
      for (int e = 0; e < 4 * NCH; ++e) acc[tk][e] = 0ull;
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
        for (int c = 0; c < NCH; ++c) {
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

  // W_V[h] -> shared memory: bf16 rows into the swizzled bf16 A tile, or
  // MXFP4 code rows into the swizzled E2M1 A tile plus the scale atoms (atom
  // g, line r: the scales of K blocks 4g..4g+3 of rows r, r+32, r+64, r+96).
  auto load_wv = [&](int h) {
    if (WFMT == 0) {
      // bf16 (128 KiB): through registers, 16 chunks per thread and pass
      // (measured faster here than asynchronous copies)
      const uint16_t *wb = static_cast<const uint16_t *>(p.w_v) + (long long)h * p.w_sh;
      constexpr int kPer = 16;
#pragma unroll 1
      for (int s0 = 0; s0 < kV * 64; s0 += kPer * NT) {
        uint4 x[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int s = s0 + threadIdx.x + i * NT;
          x[i] = __ldg(reinterpret_cast<const uint4 *>(wb + (long long)(s >> 6) * p.w_sv) + (s & 63));
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int s = s0 + threadIdx.x + i * NT;
          *reinterpret_cast<uint4 *>(gA + sw128_offset(s >> 6, s & 63, kV)) = x[i];
        }
      }
    } else {
      // MXFP4 (34 KiB): asynchronous copies (cp.async), no registers held,
      // overlapped with the loads that follow; each thread waits for its own
      // copies before it next arrives on a latent buffer
      const uint8_t *wb = static_cast<const uint8_t *>(p.w_v) + (long long)h * p.w_sh;
      for (int s = threadIdx.x; s < kV * 16; s += NT) {
        const int v = s >> 4, c = s & 15;  // row, 16-byte chunk (32 codes)
        cp_async_16(smem_u32(gA + (c >> 3) * (kV * 128) + v * 128 + (((c & 7) ^ (v & 7)) << 4)),
                    reinterpret_cast<const uint4 *>(wb + (long long)v * p.w_sv) + c);
      }
      // scales: (row v, group g) -> the 4 scales of K blocks 4g..4g+3
      const uint8_t *sb = p.w_scale + (long long)h * p.s_sh;
      const bool al4 = ((reinterpret_cast<uintptr_t>(sb) | (uintptr_t)p.s_sv) & 3u) == 0;
      for (int s = threadIdx.x; s < kV * 4; s += NT) {
        const int v = s >> 2, g = s & 3;
        const uint8_t *sr = sb + (long long)v * p.s_sv + 4 * g;
        uint8_t *dst = gSFA + g * 512 + (v & 31) * 16 + (v >> 5) * 4;
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

  // The unit's MMAs (one thread): D[v, t] = sum_k W_V[h][v][k] * lat[t][k].
  // `first` marks the first unit of a head in this CTA: W_V's scales go to
  // TMEM then (every earlier MMA is complete by that time).
  auto issue_mma = [&](int i, bool first) {
    const int b = i % ST;
    tc_fence_after();
    const uint32_t d = tmem + (uint32_t)(b * BN);
    const uint32_t sB = sB0 + (uint32_t)b * L.b_bytes;
    const uint32_t dA = (uint32_t)smem_desc_sw128(sA), dB = (uint32_t)smem_desc_sw128(sB);
    if (WFMT == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, BN);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const uint32_t kb = k >> 2, kk = k & 3;
        tc_mma_f16(d, desc_sw128_at(dA, kb * 16384u + kk * 32u), desc_sw128_at(dB, kb * (uint32_t)(BN * 128) + kk * 32u),
                   kIdesc, k > 0 ? 1u : 0u);
      }
    } else {
      constexpr uint32_t kIdesc = idesc_mxf4(128, BN);
      const uint32_t sfa = tmem + L.sfa_col, sfb = tmem + L.sfb_col + 16u * (uint32_t)b;
      const uint32_t sSFA = smem_u32(gSFA), sSFB = smem_u32(gSFB0) + (uint32_t)b * 2048u;
      if (first) {
#pragma unroll
        for (int g = 0; g < 4; ++g) tc_cp_32x128b_warpx4(sfa + 4u * g, smem_desc_rows16(sSFA + 512u * g));
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) tc_cp_32x128b_warpx4(sfb + 4u * g, smem_desc_rows16(sSFB + 512u * g));
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // K = 64 per step: two 32-blocks, scale word k/2, bytes 2(k%2)..
        const uint32_t kb = k >> 2, kk = k & 3;
        tc_mma_mxf4(d, desc_sw128_at(dA, kb * (uint32_t)(kV * 128) + kk * 32u),
                    desc_sw128_at(dB, kb * (uint32_t)(BN * 128) + kk * 32u),
                    kIdesc | idesc_sf_ids(2u * (k & 1)), sfa + 4u * (k >> 1), sfb + 4u * (k >> 1), k > 0 ? 1u : 0u);
      }
    }
    tc_commit(bar_mma0 + 8 * b);
    misc[12 + b] = (uint32_t)(i + 1);
  };

  int drained = 0;        // next unit whose accumulator is drained
  Cur cdr = c_first;      // its cursor
  auto drain_to = [&](int last) -> bool {  // epilogues of units drained .. last
    while (drained <= last) {
      if (!epilogue(drained, cdr)) return false;
      ++drained;
      advance(cdr);
    }
    return true;
  };

  // Unit i (cursor c; previous unit at cp) has its latents merged: round /
  // quantise, store, arrive (the last warp issues the MMAs), then drain the
  // previous unit's accumulator.
  auto finish = [&](int i, const Cur &c, const Buf &raw_rows) -> bool {
    const int b = i % ST;
    uint8_t *gB = gB0 + (size_t)b * L.b_bytes;
#pragma unroll
    for (int tk = 0; tk < TPW; ++tk) {
      const bool valid = HR ? c.tile * UT + (warp >> 1) + tk < p.S : tok(c.tile, warp * TPW + tk) < p.S;
      const int row = HR ? (warp >> 1) + tk : warp * TPW + tk;
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        // HR: this warp's half of the row (a 256-latent K block of MXFP4 codes)
        const int kh = HR ? (warp & 1) : cc;
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
        if (WFMT == 0) {
          if (!valid) x = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(gB + sw128_offset(row, lane + 32 * kh, BN)) = x;
        } else {
          // codes of elements 256kh + 8 lane .. +7: K block kh of the row,
          // bytes 4 lane .. 4 lane + 3; the scale of block 8kh + lane/4
          uint32_t sc;
          uint32_t w = mx_codes(x, sc);
          if (!valid) {
            w = 0u;
            sc = 127u;
          }
          *reinterpret_cast<uint32_t *>(gB + kh * (BN * 128) + row * 128 + ((((lane >> 2) ^ (row & 7))) << 4) +
                                        4 * (lane & 3)) = w;
          if ((lane & 3) == 0) {
            const int blk = 8 * kh + (lane >> 2);
            gSFB0[(size_t)b * 2048 + (blk >> 2) * 512 + row * 16 + (blk & 3)] = (uint8_t)sc;
          }
        }
      }
    }
    cp_async_wait<0>();  // this thread's W_V copies, if any, have landed
    fence_proxy_async_smem();
    __syncwarp();
    // Arrivals on stage b are numbered across its uses: use i / ST takes
    // numbers (i / ST) * kWorkers .. + kWorkers - 1.  The last arriver, the
    // unit's slowest warp, would issue the MMAs on the unit's critical path;
    // instead it marks the unit pending, and the first warp to reach its next
    // finish claims and issues it (at the latest the last arriver itself, one
    // unit on).  A unit every warp drains right away (the last of a head, the
    // CTA's last) is issued at once.  The claim comes before the own arrival,
    // so the MMAs of consecutive units are issued in order.
    const uint32_t last_no = (uint32_t)(i / ST + 1) * kWorkers - 1u;
    const bool defer = kDeferIssue && i + 1 < nu && c.tile + 1 != tph;
    auto arrive = [&]() {  // one lane
      if (kDeferIssue && i > 0 &&
          atom_cas_acq_rel_cta(pend0 + 4 * ((i - 1) % ST), (uint32_t)i, 0u) == (uint32_t)i)
        issue_mma(i - 1, i == 1 || c.tile == 1);  // unit i-1 is of the same head (else it was not deferred)
      if (atom_add_acq_rel_cta(cnt0 + 4 * b, 1u) == last_no) {
        if (defer)
          st_release_cta(pend0 + 4 * b, (uint32_t)(i + 1));
        else
          issue_mma(i, i == 0 || c.tile == 0);
      }
    };
    if (WFMT != 0 && TPW == 2) {
      // MXFP4, two tokens per warp: an elected lane of the converged warp
      // (measured faster than a divergent lane 0; with one token per warp it
      // costs registers)
      uint32_t leader;
      if (elect_one(leader)) arrive();
    } else if (lane == 0) {
      arrive();
    }
    __syncwarp();
    // drain the accumulator of unit i - (ST - 1); before the next unit of
    // another head, drain everything (W_V is replaced once those MMAs are done)
    const bool head_change = i + 1 < nu && c.tile + 1 == tph;
    bool ok = drain_to(head_change ? i : i - (ST - 1));
    // the gate of the unit the next finish drains, into L2 a unit ahead (large
    // batch 315 -> 309 us MXFP4, 344 -> 327 us bf16; at a CTA's last finish
    // the drain follows at once, so it is skipped)
    if (kGatePrefetch && i + 1 < nu && drained < nu) prefetch_gate(cdr);
    clear_acc();
    if (ok && head_change) load_wv(c.h + 1);
    return ok;
  };

  // ---- the pipeline: step k merges batch k while batch k+1 is in flight ----
  bool ok = true;
  clear_acc();
  float lse1 = kNegInf, lse2 = kNegInf;  // LSE of units i+1 and i+2
  float wcur = 0.0f, wnxt = 0.0f;       // weights of units i and i+1
  Buf bufA, bufB;
  Wts wA, wB;
  // MXFP4, 32-token tiles, two batches per unit (the large batch): the first
  // unit's second batch is issued blind with the first, so both register
  // buffers load during the LSE round trip.  Measured 291 -> 282 us per
  // launch, more than one unit of ~80 per CTA can save: the gain is in the
  // code generated for the loop.  bf16 (319 -> 322 us) and the decode-size
  // instances (stacked MXFP4 8.24 -> 8.78 us in the even-batch loop) measured
  // slower with it, so their code stays without it.
  const bool pair_loop = kTwoBatchLoop && (nb == 2 || (!(WFMT != 0 && BN == 16 && NW == 16) && nb % 2 == 0));
  const bool blind2 = kTwoBatchLoop && WFMT != 0 && BN == 32 && nb == 2;
  Cur cu = c_first;    // unit i (being merged)
  Cur cn = c_first;    // unit of the next batch to issue
  Cur cl = c_first;    // next unit whose LSE is loaded (i+3)
  int i = 0, bi = 0;   // unit and batch being merged
  int nbi = 1;         // batch index of the next batch within its unit
  // W_V of the first head is a weight (no earlier kernel writes it): copied
  // before waiting for the previous grid on the stream, so that with a
  // programmatic dependent launch it overlaps that grid's tail; every read
  // of o, lse and gate and every write comes after the wait
  if (nu > 0) load_wv(c_first.h);
  grid_dependency_wait();
  if (p.ready_flag) {
    // the producer's completion flag (optional): no input is read before it
    // is raised; a flag still down at the wait limit ends the call
    if (threadIdx.x == 0) {
      const unsigned long long t0 = globaltimer();
      while (ld_acquire_gpu(p.ready_flag) == 0) {
        if (globaltimer() - t0 > p.wait_ns) {
          atomicCAS(p.err, 0, kErrWaitFlag);
          *s_abort = 1;
          break;
        }
        __nanosleep(256);
      }
    }
    __syncthreads();
  }
  // (after a flag timeout the loops below stop at once: they test the abort flag)
  if (nu > 0 && !(p.ready_flag && *s_abort)) {
    float lse0;
    load_lse(cl, lse0);
    advance(cl);
    if (nu > 1) load_lse(cl, lse1);
    advance(cl);
    if (nu > 2) load_lse(cl, lse2);
    advance(cl);
    {
      Cur c1 = c_first;
      advance(c1);
      if (nu > 1) prefetch_rows(c1, lse1);
    }
    // the first batch is issued before its weights are known (all partials
    // of the range; rows that turn out dead are loaded but never merged), so
    // its loads overlap the LSE round trip
    issue_blind(cu, 0, bufA);
    if (blind2) issue_blind(cu, JB, bufB);
    weights_of(lse0, wcur);
#pragma unroll
    for (int jj = 0; jj < JB; ++jj)
#pragma unroll
      for (int tk = 0; tk < TPW; ++tk) wA[jj][tk] = __shfl_sync(0xffffffffu, wcur, tk * SEG + jj);
    if (blind2) {
#pragma unroll
      for (int jj = 0; jj < JB; ++jj)
#pragma unroll
        for (int tk = 0; tk < TPW; ++tk) wB[jj][tk] = __shfl_sync(0xffffffffu, wcur, tk * SEG + JB + jj);
    }
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
        lse1 = lse2;
        if (i + 2 < nu) {
          Cur c2 = cn;  // unit i+1; lse1 now holds unit i+2's LSE
          advance(c2);
          prefetch_rows(c2, lse1);
        }
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
      if (!finish(i, cu, cur)) return false;
      wcur = wnxt;
      advance(cu);
      ++i;
      bi = 0;
    }
    return true;
  };

  // Exactly two batches per unit (the large batch): batch 0 of a unit never
  // opens a unit and never finishes one, so each copy of the loop body holds
  // only its own half (one copy of the finish and epilogue in the hot loop).
  auto opens_next = [&](Buf &nxt, Wts &wn) {  // batch 0 of unit i+1 (cursor cn)
    weights_of(lse1, wnxt);
    lse1 = lse2;
    if (i + 2 < nu) {
      Cur c2 = cn;
      advance(c2);
      prefetch_rows(c2, lse1);
    }
    if (i + 3 < nu) load_lse(cl, lse2);
    advance(cl);
    issue(cn, 0, nxt, wn, wnxt);
    if (WFMT != 0) {
      // the new unit's second batch into L2 (live rows): it is merged only
      // one batch after it is issued (large MXFP4 batch 291.4 -> 289.4 us;
      // bf16 prefetches whole units ahead instead)
      const int t = HR ? cn.tile * UT + (warp >> 1) + my_tk : tok(cn.tile, warp * TPW + my_tk);
      if (my_j >= JB && my_j < 2 * JB && wnxt != 0.0f && t < p.S) {
        const int r0 = (layout == kRequestMajor) ? (t / p.q) * p.spr : 0;
        if constexpr (HR)  // this warp's half of the row
          prefetch_l2_bulk(p.o + off3(t, p.o_st, cn.h, p.o_sh, r0 + my_j, p.o_sp) + (warp & 1) * (kD / 2), kD);
        else
          prefetch_l2_bulk(p.o + off3(t, p.o_st, cn.h, p.o_sh, r0 + my_j, p.o_sp), kD * 2);
      }
    }
  };
  if (kTwoBatchLoop && nb == 2) {
    for (int k = 0; k < total; k += 2) {
      if (*s_abort) {
        ok = false;
        break;
      }
      // batch 0 of unit i is in bufA: send batch 1 of unit i (the first
      // unit's went out blind), merge batch 0
      if (!(blind2 && k == 0)) issue(cn, JB, bufB, wB, wcur);
      advance(cn);
      consume(bufA, wA);
      // batch 1 in bufB: send batch 0 of unit i+1, merge batch 1, finish unit i
      if (k + 2 < total) opens_next(bufA, wA);
      consume(bufB, wB);
      if (!finish(i, cu, bufB)) {
        ok = false;
        break;
      }
      wcur = wnxt;
      advance(cu);
      ++i;
    }
  } else if (pair_loop) {
    // an even number of batches per unit (decode sizes with more partials):
    // batch pairs, the unit's finish once after its last pair (decode 2%
    // faster; not for the one-token-per-warp MXFP4 instance, where it spills)
    for (int k = 0; k < total; k += nb) {
      if (*s_abort) {
        ok = false;
        break;
      }
      for (int b = 0; b < nb; b += 2) {
        // batch b in bufA: send batch b+1, merge batch b
        issue(cn, (b + 1) * JB, bufB, wB, wcur);
        consume(bufA, wA);
        // batch b+1 in bufB: send the next batch (b+2, or batch 0 of unit i+1)
        if (b + 2 < nb) {
          issue(cn, (b + 2) * JB, bufA, wA, wcur);
        } else {
          advance(cn);
          if (k + nb < total) opens_next(bufA, wA);
        }
        consume(bufB, wB);
      }
      if (!finish(i, cu, bufB)) {
        ok = false;
        break;
      }
      wcur = wnxt;
      advance(cu);
      ++i;
    }
  } else {
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
  }
  if (ok && nu > 0 && !*s_abort) drain_to(nu - 1);

  // rows S .. S_out-1 of core are zero (this CTA's slice of them)
  const long long n16 = (long long)(p.S_out - p.S) * p.H * (kV * 2 / 16);
  if (n16 > 0) {
    const long long zb = (long long)blockIdx.x * n16 / gridDim.x;
    const long long ze = (long long)(blockIdx.x + 1) * n16 / gridDim.x;
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (long long)p.S * Wrow);
    for (long long k = zb + threadIdx.x; k < ze; k += NT) dst[k] = make_uint4(0, 0, 0, 0);
  }

  cp_async_wait<0>();
  __syncthreads();
  if (threadIdx.x == 0) {
    // drain what this CTA started (only pending after an abort): the last
    // committed MMAs
    for (int b = 0; b < ST; ++b) {  // MMAs may come from different threads: every stage's last use
      if (misc[12 + b] > 0u) {
        const int last = (int)misc[12 + b] - 1;
        mbar_wait(bar_mma0 + 8 * b, (uint32_t)(last / ST) & 1u, p.err, kErrWaitTeardown);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// Warps per CTA: 16, except MXFP4 W_V with 16-token tiles and at most 16
// partials per token, which runs two 8-warp CTAs per SM (about 60 KiB of
// shared memory each, independent pipelines).  A warp owns BN / warps tokens;
// with two tokens a warp holds at most 16 partials per token.  8-token tiles
// are the half-row instance of the 16-token kernel: 16 warps, two per token.
int tc_warps(int tile, int w_fmt, int n_part) { return (w_fmt && tile == 16 && n_part <= 16) ? 8 : 16; }
int tc_ctas_per_sm(int tile, int w_fmt, int n_part) { return tc_warps(tile, w_fmt, n_part) == 8 ? 2 : 1; }
// 17..31-token tiles are the 32-token kernel with that many tokens per unit.
int tc_max_part(int tile, int /*w_fmt*/) { return tile > 16 ? 16 : 32; }

size_t tc_smem_bytes(int tile, int w_fmt, int n_part) {
  const int bn = tile == 8 ? 16 : (tile > 16 ? 32 : tile);
  return 1024 + tc_layout(bn, w_fmt, tc_warps(tile, w_fmt, n_part)).total;
}

template <int BN, int WFMT, int NW, bool O32, bool HR = false, bool RT = false>
static cudaError_t launch_one(const KParams &p, int grid, cudaStream_t s) {
  const size_t smem = 1024 + tc_layout(BN, WFMT, NW).total;
  cudaError_t e = cudaFuncSetAttribute(tc_kernel<BN, WFMT, NW, O32, HR, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch (see the prologue)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_kernel<BN, WFMT, NW, O32, HR, RT>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool O32>
static cudaError_t launch_tc_off(const KParams &p, int grid, cudaStream_t stream) {
  const int nw = tc_warps(p.tile, p.w_fmt, p.n_part);
  if (p.tile == 8)
    return p.w_fmt == 0 ? launch_one<16, 0, 16, O32, true>(p, grid, stream)
                        : launch_one<16, 1, 16, O32, true>(p, grid, stream);
  if (p.tile == 16 && p.w_fmt == 0) return launch_one<16, 0, 16, O32>(p, grid, stream);
  if (p.tile == 16 && p.w_fmt == 1)
    return nw == 8 ? launch_one<16, 1, 8, O32>(p, grid, stream) : launch_one<16, 1, 16, O32>(p, grid, stream);
  if (p.tile == 32 && p.n_part <= 16)
    return p.w_fmt == 0 ? launch_one<32, 0, 16, O32>(p, grid, stream) : launch_one<32, 1, 16, O32>(p, grid, stream);
  if (p.tile > 16 && p.tile < 32 && p.n_part <= 16)
    return p.w_fmt == 0 ? launch_one<32, 0, 16, O32, false, true>(p, grid, stream)
                        : launch_one<32, 1, 16, O32, false, true>(p, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc(const KParams &p, int grid, cudaStream_t stream) {
  return p.off32 ? launch_tc_off<true>(p, grid, stream) : launch_tc_off<false>(p, grid, stream);
}

}  // namespace mla
