// device_common.cuh -- shared device helpers of the sm_103a kernels: number
// formats (bf16, E2M1, E8M0), the LSE weight rule, bounded mbarrier waits and
// thin inline-PTX wrappers for TMA and tcgen05.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kparams.h"

namespace mla {

constexpr int kD = 512;    // latent width
constexpr int kV = 128;    // V head dim
constexpr int kBlk = 32;   // MX block along K
constexpr float kLog2e = 1.4426950408889634f;

// Bounded waits give up after this long and report MLA_ERR_TIMEOUT through
// the error word; a healthy wait here lasts microseconds.  (The combine's
// tensor-core kernel takes its pipeline limit from its launch parameters.)
constexpr unsigned long long kWaitNs = kDefaultWaitNs;

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- number formats ------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> packed bf16 pair (round to nearest even).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// E8M0 code -> 2^(code - 127) as fp32 (code 255 -> NaN; code 0 -> 2^-127, a
// subnormal).
__device__ __forceinline__ float e8m0_to_f32(uint32_t code) {
  if (code == 255u) return __uint_as_float(0x7FC00000u);
  if (code == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(code << 23);
}

// Shared MX scale code from the largest sign-cleared bf16 pattern of a block:
// floor(log2 amax) - 2 + 127 is the exponent field minus 2 for normal values;
// clamped below at 1 (zero and subnormal blocks); 255 (NaN) when the block
// holds an Inf or NaN.
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t amax_bits) {
  uint32_t ef = (amax_bits >> 7) & 0xFFu;
  if (ef == 0xFFu) return 255u;
  int c = (int)ef - 2;
  return c < 1 ? 1u : (uint32_t)c;
}

// Magnitude code (0..7) of E2M1 for an already-scaled magnitude a >= 0:
// round to nearest, ties to the even code, saturate at 6.  The decision
// points are the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5 and 5; at a tie
// the even code wins, so the comparison is strict where the lower neighbour
// is even and inclusive where the upper one is.
__device__ __forceinline__ uint32_t e2m1_mag_code(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
         (uint32_t)(a > 5.0f);
}

__device__ __forceinline__ float e2m1_mag_value(uint32_t c) {
  // 0, .5, 1, 1.5, 2, 3, 4, 6
  const float m = (c < 4u) ? 0.5f * (float)c : (float)(2u << ((c - 4u) >> 1)) * (1.0f + 0.5f * (float)(c & 1u));
  return m;
}

// Quantise one bf16 value x (given as fp32) with block scale code sc and
// return the dequantised value: +-E2M1(x / 2^(sc-127)) * 2^(sc-127).
// The scaling by a power of two is exact (no flush-to-zero in this build).
__device__ __forceinline__ float mx_fake_quant(float x, uint32_t sc, float scale, float inv_scale) {
  if (sc == 255u) return __uint_as_float(0x7FC00000u);
  float a = fabsf(x) * inv_scale;
  uint32_t c = e2m1_mag_code(a);
  float v = e2m1_mag_value(c) * scale;
  return (c != 0u && signbit(x)) ? -v : v;
}

// 2^(127 - sc) for a scale code 1..254, exact (2^-127 is a subnormal).
__device__ __forceinline__ float e8m0_inverse(uint32_t sc) {
  int e = 127 - (int)sc;  // -127 .. 126
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  return __uint_as_float(0x00400000u);
}

// The hardware's base-2 exponential and reciprocal (the approximations the
// page's combine uses; exact at 0 -> 1 and for powers of two, ex2(-inf) = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sanitise an LSE: NaN and +inf become -inf.
__device__ __forceinline__ float sane(float x) {
  return (x != x || x == __int_as_float(0x7F800000)) ? __int_as_float(0xFF800000) : x;
}

// Packed bf16 product, rounded once to nearest even: the same bits as the
// fp32 product of the two bf16 values (exact) rounded to bf16.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One elected lane of a converged warp: returns true in that lane and sets
// `leader` to its lane id in every lane.
__device__ __forceinline__ bool elect_one(uint32_t &leader) {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync %0|p, 0xffffffff;\n\tselp.u32 %1, 1, 0, p;\n\t}"
               : "=r"(leader), "=r"(e));
  return e != 0;
}

// Per-half unsigned maximum of two packed 16-bit pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---- packed fp32 pairs and hardware E2M1 conversions (sm_100 family) -----

// Round-to-nearest packed fp32 arithmetic on (lo, hi) pairs: one rounding
// per lane of the pair, exactly like two scalar operations.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two fp32 values -> an E2M1 pair (round to nearest even, saturating at +-6),
// `hi` in the upper nibble.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Eight bf16 values (four packed pairs) times an exact power of two -> eight
// E2M1 codes (nearest even, saturating at 6), element 2i in the low nibble of
// byte i.
__device__ __forceinline__ uint32_t e2m1x8_from_bf16x8(const uint32_t (&u)[4], float scale) {
  uint32_t r;
  asm("{\n\t"
      ".reg .b8 c0, c1, c2, c3;\n\t"
      ".reg .f32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      ".reg .b64 p, s;\n\t"
      "shl.b32 l0, %1, 16;\n\tand.b32 h0, %1, 0xffff0000;\n\t"
      "shl.b32 l1, %2, 16;\n\tand.b32 h1, %2, 0xffff0000;\n\t"
      "shl.b32 l2, %3, 16;\n\tand.b32 h2, %3, 0xffff0000;\n\t"
      "shl.b32 l3, %4, 16;\n\tand.b32 h3, %4, 0xffff0000;\n\t"
      "mov.b64 s, {%5, %5};\n\t"
      "mov.b64 p, {l0, h0};\n\tmul.rn.f32x2 p, p, s;\n\tmov.b64 {l0, h0}, p;\n\t"
      "mov.b64 p, {l1, h1};\n\tmul.rn.f32x2 p, p, s;\n\tmov.b64 {l1, h1}, p;\n\t"
      "mov.b64 p, {l2, h2};\n\tmul.rn.f32x2 p, p, s;\n\tmov.b64 {l2, h2}, p;\n\t"
      "mov.b64 p, {l3, h3};\n\tmul.rn.f32x2 p, p, s;\n\tmov.b64 {l3, h3}, p;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, h0, l0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, h1, l1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, h2, l2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, h3, l3;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t"
      "}"
      : "=r"(r)
      : "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "f"(scale));
  return r;
}

// MXFP4 quantisation of a lane's 8 bf16 latents (one 16-byte chunk; the
// block of 32 spans lanes 4g..4g+3).  Scale code from the largest
// sign-cleared bf16 pattern; elements scaled by an exact power of two and
// converted to E2M1 by the hardware (nearest even, saturating at 6).  Returns
// the 8 codes packed (element 2i in the low nibble of byte i) and the scale.
__device__ __forceinline__ uint32_t mx_codes(uint4 x, uint32_t &sc) {
  const uint32_t u[4] = {x.x, x.y, x.z, x.w};
  const uint32_t am2 = max_u16x2(max_u16x2(u[0] & 0x7FFF7FFFu, u[1] & 0x7FFF7FFFu),
                                 max_u16x2(u[2] & 0x7FFF7FFFu, u[3] & 0x7FFF7FFFu));
  uint32_t am = max(am2 & 0xFFFFu, am2 >> 16);
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
  // exponent field ef of the block maximum: scale code max(ef, 3) - 2 (zero
  // and tiny blocks clamp to 1; a finite block never exceeds 252), its
  // inverse 2^(127 - code) has exponent field 256 - max(ef, 3); ef = 255
  // (Inf / NaN in the block) gives the NaN code, which carries it, and zero
  // codes
  const uint32_t ef = am >> 7, e3 = max(ef, 3u);
  sc = (ef == 255u) ? 255u : e3 - 2u;
  const uint32_t w = e2m1x8_from_bf16x8(u, __uint_as_float((256u - e3) << 23));
  return (ef == 255u) ? 0u : w;
}

// An E2M1 pair (low nibble -> lo) -> two fp16 values packed as (lo, hi).
__device__ __forceinline__ uint32_t f16x2_from_e2m1x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

__device__ __forceinline__ float f16_lo(uint32_t h2) {
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t h2) {
  return __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// ---- mbarrier ----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most kWaitNs.
// Returns false (and records `code` in the error word) on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *err, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitNs) {
      if (err) atomicCAS(err, 0, code);
      return false;
    }
  }
}

// Global 32-bit load with acquire semantics at GPU scope (a flag another
// kernel or CTA raises after writing the data it guards).
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory atomic add with acquire-release semantics at CTA scope;
// returns the previous value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_cta(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// Shared-memory compare-and-swap with acquire-release semantics at CTA
// scope; returns the previous value.
__device__ __forceinline__ uint32_t atom_cas_acq_rel_cta(uint32_t addr, uint32_t cmp, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.cas.b32 %0, [%1], %2, %3;" : "=r"(old) : "r"(addr), "r"(cmp), "r"(v)
               : "memory");
  return old;
}
// Shared-memory store with release semantics at CTA scope.
__device__ __forceinline__ void st_release_cta(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Bulk prefetch of a global range into L2 (size a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Prefetch of the 128-byte line holding `src` into L2 (a load-path request).
__device__ __forceinline__ void prefetch_l2_line(const void *src) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
}

// ---- cp.async (per-thread asynchronous copies into shared memory) ----------

__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst_smem, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- proxies, TMA, tcgen05 --------------------------------------------

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order global-memory writes this thread has observed (through an acquire)
// before its later async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// 3-D tiled TMA load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// ---- programmatic dependent launch ---------------------------------------

// Block until every grid this one depends on (the previous kernel on the
// stream, when launched with programmatic stream serialization) has completed
// and its memory is visible; returns at once otherwise.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next dependent launch to begin (its own wait still orders it
// after this grid's completion).
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---- thread-block clusters and distributed shared memory ----------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster; release / acquire ordering of
// shared-memory (and mbarrier) state across the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// 16-byte asynchronous store into another CTA's shared memory, counted as
// transaction bytes on that CTA's mbarrier `rbar` (both shared::cluster).
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float a, float b, float c, float d, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::mxf4 with E8M0 block-32 scales
// (two scales per row per K=64 step, taken from TMEM at sfa / sfb).
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copy a 32-row x 16-byte shared-memory matrix into TMEM lanes 0..31 of four
// columns, replicated into all four lane quadrants.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is
// complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 4 consecutive columns.
__device__ __forceinline__ void tmem_ld_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 columns of fp32 back into TMEM (warp-wide), and the wait for it.
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Barrier over `count` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The same barrier, returning whether `pred` holds in every participating thread.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 lanes x 32 bit, 8 consecutive columns.
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand with the
// 128-byte swizzle, rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address, 16-byte units
  d |= (uint64_t)(16u >> 4) << 16;                  // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                           // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                           // swizzle mode: 128 B
  return d;
}

// The same descriptor at `off` bytes past the one whose lower word is `lo`:
// the start address is the low 14 bits of the lower word (shared memory is
// below 256 KiB), so a 16-byte-unit offset adds to the lower word alone.
constexpr uint32_t kDescSw128Hi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint64_t desc_sw128_at(uint32_t lo, uint32_t off) {
  return ((uint64_t)kDescSw128Hi << 32) | (uint64_t)(lo + (off >> 4));
}

// Descriptor of an MN-major operand with the 128-byte swizzle, as a TMA box of
// [rows x 64 elements] writes it: 64 MN elements per 128-byte row, 8-row K
// groups 1024 bytes apart (stride byte offset), the next 64 MN elements
// `mn_stride` bytes further (leading byte offset).
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Shared-memory descriptor without swizzle: 16-byte rows, 8-row groups 128
// bytes apart (the source layout of a 32x128b tcgen05.cp).
__device__ __forceinline__ uint64_t smem_desc_rows16(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor, kind::mxf4 block-scaled: E2M1 A and B, E8M0 scales,
// fp32 D, both K-major.  The scale-factor ids (byte offset of the two scales
// in each 32-bit TMEM word: 0 or 2) are or-ed in per K step.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7)                      // A format: E2M1
         | (1u << 10)                   // B format: E2M1
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | (1u << 23)                   // scale format: UE8M0
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}
__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t id) { return (id << 4) | (id << 29); }

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// Byte offset of 16-byte chunk `c` (0..63) of row `r` in a K-major bf16 tile
// of `rows` rows stored as 8 K-blocks of [rows x 128 B] with the 128-byte
// swizzle (chunk j of a row lives at j ^ (r % 8)).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c, int rows) {
  const int kb = c >> 3, j = c & 7;
  return (uint32_t)(kb * rows * 128 + r * 128 + ((j ^ (r & 7)) << 4));
}

}  // namespace mla
