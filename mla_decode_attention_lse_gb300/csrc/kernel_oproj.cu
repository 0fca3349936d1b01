// kernel_oproj.cu -- downstream of the stage: this rank's o_proj shard.
//
// The vLLM page "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.
// mla_back" ends its stage at "o_proj's input" (core, [S, H*128]).  o_proj is
// a row-parallel linear layer: the rank multiplies its core rows by its slice
// of the weight, out[t][j] = sum_k core[t][k] W[j][k], and the tensor-parallel
// all-reduce (multi-GPU) sums the ranks' outputs.  At decode sizes (64 tokens,
// K = 1536, 7168 outputs) the shard streams 22 MB of weight for 64 tokens: an
// HBM-bound GEMM.
//
// Work units are (64 output features, NT tokens); a persistent grid of one
// CTA per SM walks them.  Warp 0 (one lane) brings, per 64-wide K block, the
// W box [64 rows x 64] and the core box [NT rows x 64] by TMA into a ring of
// stages; two MMA warps (one lane each) issue D[j, t] += W x^T as four
// kind::f16 MMAs of M = 64, N = NT, K = 16 per stage -- warp 1 the even K
// blocks into accumulator D0, warp 6 the odd ones into D1 (one thread issues
// an MMA about every 55 cycles whatever its size at these N, and two threads'
// MMAs overlap) -- with D0 / D1 double-buffered over units where TMEM allows
// (D row i of an M = 64 MMA sits in TMEM lane 32 (i / 16) + i % 16); warps
// 2..5 read both (lanes 0..15 of their quadrant), add them in fp32
// (D = D0 + D1), round to bf16 into a staging tile in shared memory, and copy
// the tile out row by row with coalesced 16-byte stores (per-element stores
// straight from the accumulator's layout took ~2.2 us per unit).  The W copies of the first stages go out before the wait for
// the previous kernel (a weight no earlier kernel writes); the core rows and
// every store come after it.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernel_oproj.h"
#include "kparams.h"

namespace mla {

namespace {

constexpr int kOpM = 64;       // output features per unit (MMA M)
constexpr int kOpThreads = 224;  // warp 0 TMA, warps 1 and 6 MMA, warps 2..5 epilogue
constexpr uint32_t kOpABytes = kOpM * 128u;  // a W box: 64 rows x 128 B

template <int NT>
struct OpLayout {
  static constexpr uint32_t stage = kOpABytes + (uint32_t)NT * 128u;
  static constexpr int kStages = (NT == 64) ? 12 : (NT == 128) ? 8 : 4;
  // the output tile [NT tokens x 64 features] bf16, staged for the copy out
  static constexpr uint32_t stg_off = kStages * stage;
  // full[ST], empty[ST], acc_full[2], acc_empty[2], drain[2] (one per MMA warp)
  static constexpr uint32_t bar_off = stg_off + (uint32_t)NT * 128u;
  static constexpr uint32_t misc_off = bar_off + (2 * kStages + 6) * 8u;
  static constexpr uint32_t total = misc_off + 16u;
  static constexpr int kBufs = NT <= 128 ? 2 : 1;  // accumulator pairs (D0, D1) in TMEM
  static constexpr uint32_t tmem_cols = (uint32_t)(kBufs * 2 * NT);
};
static_assert(OpLayout<64>::tmem_cols == 256 && OpLayout<128>::tmem_cols == 512 && OpLayout<256>::tmem_cols == 512,
              "TMEM columns");
static_assert(OpLayout<64>::total + 1024 <= 227u * 1024u, "shared memory (NT = 64)");
static_assert(OpLayout<128>::total + 1024 <= 227u * 1024u, "shared memory (NT = 128)");
static_assert(OpLayout<256>::total + 1024 <= 227u * 1024u, "shared memory (NT = 256)");

__device__ __forceinline__ bool op_wait(uint32_t bar, uint32_t parity, int *err, volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitNs) {
      atomicCAS(err, 0, kErrWaitMma);
      *abort_flag = 1;
      return false;
    }
  }
}

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kOpThreads, 1)
    oproj_kernel(const __grid_constant__ OprojParams p, const __grid_constant__ CUtensorMap wmap,
                 const __grid_constant__ CUtensorMap xmap) {
  using L = OpLayout<NT>;
  constexpr int ST = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // swizzle atoms: 1024-byte aligned
  uint8_t *gbase = smem_raw + (sbase - raw);
  uint32_t *misc = reinterpret_cast<uint32_t *>(gbase + L::misc_off);
  volatile int *s_abort = reinterpret_cast<volatile int *>(&misc[1]);
  const uint32_t bar0 = sbase + L::bar_off;
  auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(ST + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (uint32_t)(2 * ST + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (uint32_t)(2 * ST + 2 + b); };
  auto drain = [&](int w) { return bar0 + 8u * (uint32_t)(2 * ST + 4 + w); };
  constexpr int NB = L::kBufs;
  // accumulator Dw (w = 0: even K blocks, 1: odd) of buffer b
  auto acc = [&](uint32_t tmem, int b, int w) { return tmem + (uint32_t)((2 * b + w) * NT); };
  auto sA = [&](int s) { return sbase + (uint32_t)s * L::stage; };
  auto sB = [&](int s) { return sbase + (uint32_t)s * L::stage + kOpABytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full(s), 1u);
      mbar_init(empty(s), 1u);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 2u);  // both MMA warps commit
      mbar_init(acc_empty(b), 4u);
      mbar_init(drain(b), 1u);
    }
    misc[1] = 0u;
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
  // the next launch on the stream may begin its prologue while this grid
  // runs (its dependent work waits for this grid's completion)
  grid_launch_dependents();
  // unit u: output features 64 (u % MT) .., tokens NT (u / MT) ..
  const int MT = p.Nout / kOpM, units = MT * ((p.S + NT - 1) / NT), KB = p.K / 64;

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      bool ok = true;
      int issued = 0;  // stages whose copies were issued
      const int u0 = blockIdx.x;
      // the first stages' weight boxes go out before the wait for the previous
      // kernel (no earlier kernel writes the weight); their core boxes after it
      const int pre = u0 < units ? min(ST, KB) : 0;
      for (int g = 0; g < pre; ++g) {
        mbar_arrive_expect_tx(full(g), L::stage);
        tma_load_3d(sA(g), &wmap, 64 * g, (u0 % MT) * kOpM, 0, full(g));
      }
      grid_dependency_wait();
      for (int g = 0; g < pre; ++g) tma_load_3d(sB(g), &xmap, 64 * g, (u0 / MT) * NT, 0, full(g));
      issued = pre;
      int g = 0;
      for (int u = u0; u < units && ok; u += gridDim.x) {
        const int mt = u % MT, nt = u / MT;
        for (int kb = 0; kb < KB; ++kb, ++g) {
          if (g < pre) continue;  // issued above
          const int s = g % ST;
          if (g >= ST) ok = op_wait(empty(s), (uint32_t)(g / ST - 1) & 1u, p.err, s_abort);
          if (!ok) break;
          mbar_arrive_expect_tx(full(s), L::stage);
          tma_load_3d(sA(s), &wmap, 64 * kb, mt * kOpM, 0, full(s));
          tma_load_3d(sB(s), &xmap, 64 * kb, nt * NT, 0, full(s));
          issued = g + 1;
        }
      }
      // after an abort: the copies still in flight land before the CTA exits
      for (int q = issued - ST < 0 ? 0 : issued - ST; q < issued; ++q)
        mbar_wait(full(q % ST), (uint32_t)(q / ST) & 1u, p.err, kErrWaitTeardown);
    }
  } else if (warp == 1 || warp == 6) {
    // ---- MMA issuers: Dw[j, t] += W[j, k] x[t, k] over the K blocks of
    // parity w; both commit a unit's acc_full ----
    if (lane == 0) {
      constexpr uint32_t kId = idesc_bf16(kOpM, NT);
      const int w = warp == 1 ? 0 : 1;
      bool ok = true;
      int g = 0, i = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
        const int b = i % NB;
        if (i >= NB) ok = op_wait(acc_empty(b), (uint32_t)(i / NB - 1) & 1u, p.err, s_abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = acc(tmem, b, w);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          if ((kb & 1) != w) continue;
          const int s = g % ST;
          ok = op_wait(full(s), (uint32_t)(g / ST) & 1u, p.err, s_abort);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dA = (uint32_t)smem_desc_sw128(sA(s)), dB = (uint32_t)smem_desc_sw128(sB(s));
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            tc_mma_f16(d, desc_sw128_at(dA, (uint32_t)k4 * 32u), desc_sw128_at(dB, (uint32_t)k4 * 32u), kId,
                       (kb >= 2 || k4) ? 1u : 0u);
          tc_commit(empty(s));
        }
        if (!ok) break;
        tc_commit(acc_full(b));  // with no K block of this parity (K = 64) it arrives at once
      }
      // every MMA this thread issued completes before TMEM is freed (after an
      // abort too)
      tc_commit(drain(w));
      mbar_wait(drain(w), 0u, p.err, kErrWaitTeardown);
    }
  } else {
    // ---- epilogue warps 2..5: quadrant warp % 4; an M = 64 accumulator has
    // row 16 q + l in lane l < 16 of quadrant q ----
    const int qd = warp & 3, et = threadIdx.x - 64;  // et: 0 .. 127
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    uint16_t *stg = reinterpret_cast<uint16_t *>(gbase + L::stg_off);  // [NT][64]
    // 16-byte stores when every row of out starts on a 16-byte boundary
    const bool vec = (reinterpret_cast<uintptr_t>(p.out) & 15u) == 0 && (p.out_st & 7) == 0;
    grid_dependency_wait();  // out may still be read by the kernel before
    int i = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
      const int b = i % NB, mt = u % MT, nt = u / MT;
      bool ok = op_wait(acc_full(b), (uint32_t)(i / NB) & 1u, p.err, s_abort);
      // the four warps take the exit decision together (a warp that left
      // would leave the others at the staging barriers)
      ok = named_barrier_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < NT; c += 16) {
        uint32_t r[16], r1[16];
        tmem_ld_x16(acc(trow, b, 0) + (uint32_t)c, r);
        if (KB > 1) tmem_ld_x16(acc(trow, b, 1) + (uint32_t)c, r1);
        tc_wait_ld();
        // lane l < 16 holds feature 16 qd + l for tokens c .. c + 15; lanes l
        // and l + 16 write its even and odd tokens (the odd values by one
        // shuffle), so the whole warp stores
        uint16_t *srow = stg + (c + (lane >> 4)) * 64 + qd * 16 + (lane & 15);
#pragma unroll
        for (int x = 0; x < 16; x += 2) {
          const float e = KB > 1 ? __fadd_rn(__uint_as_float(r[x]), __uint_as_float(r1[x])) : __uint_as_float(r[x]);
          const float o =
              KB > 1 ? __fadd_rn(__uint_as_float(r[x + 1]), __uint_as_float(r1[x + 1])) : __uint_as_float(r[x + 1]);
          const float o_hi = __shfl_xor_sync(0xffffffffu, o, 16);
          const __nv_bfloat16 h = __float2bfloat16_rn(lane < 16 ? e : o_hi);
          srow[x * 64] = *reinterpret_cast<const uint16_t *>(&h);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
      named_barrier(1, 128);  // the tile is staged
      const int rows = min(NT, p.S - nt * NT);
      uint16_t *obase = p.out + (long long)nt * NT * p.out_st + mt * kOpM;
      if (vec) {
        for (int ch = et; ch < rows * 8; ch += 128) {
          const int row = ch >> 3, c16 = ch & 7;
          *reinterpret_cast<uint4 *>(obase + (long long)row * p.out_st + c16 * 8) =
              *reinterpret_cast<const uint4 *>(stg + row * 64 + c16 * 8);
        }
      } else {
        for (int e = et; e < rows * 64; e += 128) obase[(long long)(e >> 6) * p.out_st + (e & 63)] = stg[e];
      }
      named_barrier(1, 128);  // the staging tile may be written again
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

int oproj_tokens_per_unit(int S) { return S <= 64 ? 64 : S <= 128 ? 128 : 256; }
size_t oproj_smem_bytes(int nt) {
  return 1024 + (nt == 64 ? OpLayout<64>::total : nt == 128 ? OpLayout<128>::total : OpLayout<256>::total);
}

template <int NT>
static cudaError_t launch_oproj_n(const OprojParams &p, const CUtensorMap &wmap, const CUtensorMap &xmap,
                                  unsigned grid, cudaStream_t stream) {
  const size_t smem = 1024 + OpLayout<NT>::total;
  cudaError_t e = cudaFuncSetAttribute(oproj_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kOpThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, oproj_kernel<NT>, p, wmap, xmap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Persistent: one CTA per SM (the stage ring fills an SM), at most one per unit.
cudaError_t launch_oproj(const OprojParams &p, const CUtensorMap &wmap, const CUtensorMap &xmap, int num_sms,
                         cudaStream_t stream) {
  if (p.S < 1 || p.K < 64 || p.K % 64 || p.Nout < kOpM || p.Nout % kOpM || num_sms < 1) return cudaErrorInvalidValue;
  if (p.nt != oproj_tokens_per_unit(p.S)) return cudaErrorInvalidValue;
  const long long units = (long long)(p.Nout / kOpM) * ((p.S + p.nt - 1) / p.nt);
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(units < num_sms ? units : num_sms);
  if (p.nt == 64) return launch_oproj_n<64>(p, wmap, xmap, grid, stream);
  if (p.nt == 128) return launch_oproj_n<128>(p, wmap, xmap, grid, stream);
  return launch_oproj_n<256>(p, wmap, xmap, grid, stream);
}

}  // namespace mla
