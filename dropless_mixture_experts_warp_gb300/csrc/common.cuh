// Shared device helpers: status words, bf16 packing, and the sm_103a PTX wrappers
// (mbarrier, TMA, tcgen05) used by the grouped GEMM.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------ status words

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ bf16 helpers

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&p);
}

// ------------------------------------------------------------------ shared memory

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// A wait that cannot hang: gives up after `limit` clock cycles, records
// MOE_ERR_TIMEOUT in the status word, raises the CTA's abort flag and returns
// false.  It also returns false as soon as another role raised the abort flag.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, int32_t* status,
                                                  long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      set_status(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// Same bound, ignoring the abort flag: used only to drain work already in flight.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes on `bar`.
// x is the innermost (contiguous) coordinate, in elements.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Tensor store of a shared-memory box (bulk-group completion), its commit, and the
// wait until at most N of this thread's bulk groups still read shared memory.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr)
               : "memory");
  return r;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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

// D[tmem] (+)= A[smem] * B[smem]^T for one K=16 slice, kind::f16 (bf16 in, fp32 acc).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane (base+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 32 columns from registers into TMEM (this warp's lane quarter).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bits 46-47, and the
// swizzle mode at bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major-ness (1 = MN), bit 16 B major-ness, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ MXFP8 quantisation
// Scale rule: e = floor(log2(amax)) - 8 clamped to [-127, 127] (byte e + 127; 0 for an
// all-zero block); codes = E4M3(x * 2^-e), round to nearest even, saturating (cvt).
// Scale tiles: tile (r/128, k/128) of 512 bytes; word (r%32)*4 + (r%128)/32 holds the
// four 32-element block scales of row r in that K range.

__device__ __forceinline__ size_t sf_byte_offset(long long r, long long k, long long k_tiles) {
  const long long tile = (r >> 7) * k_tiles + (k >> 7);
  const int word = static_cast<int>((r & 31) * 4 + ((r & 127) >> 5));
  return static_cast<size_t>(tile) * 512 + word * 4 + static_cast<int>((k & 127) >> 5);
}

// floor(log2(a)) - EMAX clamped to [-127, 127] for a finite a >= 0 (-127 for a = 0);
// EMAX is the element format's largest exponent (8 for E4M3, 2 for E2M1).
template <int EMAX>
__device__ __forceinline__ int mx_scale_exp_t(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ef = static_cast<int>((b >> 23) & 0xFF);
  int fl;
  if (ef > 0) {
    fl = ef - 127;
  } else {
    const uint32_t m = b & 0x7FFFFF;
    if (m == 0) return -127;
    fl = (31 - __clz(m)) - 149;
  }
  return max(-127, min(127, fl - EMAX));
}
__device__ __forceinline__ int mx_scale_exp(float a) { return mx_scale_exp_t<8>(a); }

// 2^-e as an fp32 for e in [-127, 127] (2^-127 .. 2^127; 2^-127 is subnormal).
__device__ __forceinline__ float exp2_neg(int e) {
  const int f = 127 - e;  // biased exponent of 2^-e
  return f > 0 ? __uint_as_float(static_cast<uint32_t>(f) << 23) : __uint_as_float(0x00400000u);
}

// Four fp32 -> four E4M3 bytes in one word (x0 in the lowest byte), RNE, saturating; the
// two halves are joined inside the asm (as one packing move, not a widen, shift and or).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\tcvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\tmov.b32 %0, {l, h};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}

// a *= s, b *= s in one packed fp32 multiply (round to nearest even, no flush: the
// same result as two scalar multiplies)
__device__ __forceinline__ void mul_f32x2(float& a, float& b, uint64_t ss) {
  asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%0, %1};\n\tmul.rn.f32x2 x, x, %2;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a), "+f"(b)
      : "l"(ss));
}

// max(|a|, |b|, |c|) in one three-input instruction.
__device__ __forceinline__ float absmax3(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Quantise 32 fp32 values (one block) into 8 words of codes; returns the scale byte.
__device__ __forceinline__ uint32_t quant_block32(const float (&v)[32], uint32_t (&codes)[8]) {
  float m[11];  // a tree of three-input maxima: 11 + 4 + 2 instructions
#pragma unroll
  for (int j = 0; j < 10; ++j) m[j] = absmax3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
  m[10] = absmax3(v[30], v[31], v[31]);
  const float n0 = absmax3(m[0], m[1], m[2]), n1 = absmax3(m[3], m[4], m[5]);
  const float n2 = absmax3(m[6], m[7], m[8]), n3 = absmax3(m[9], m[10], m[10]);
  const float amax = absmax3(absmax3(n0, n1, n2), n3, n3);
  const int e = mx_scale_exp(amax);
  const uint32_t sb = __float_as_uint(exp2_neg(e));
  const uint64_t ss = (static_cast<uint64_t>(sb) << 32) | sb;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    float x0 = v[4 * w + 0], x1 = v[4 * w + 1], x2 = v[4 * w + 2], x3 = v[4 * w + 3];
    mul_f32x2(x0, x1, ss);
    mul_f32x2(x2, x3, ss);
    codes[w] = cvt_e4m3x4(x0, x1, x2, x3);
  }
  return static_cast<uint32_t>(e + 127);
}

// Eight fp32 -> eight E2M1 (FP4) codes in one word, element i in bits 4i..4i+3: round to
// nearest even, saturating at +-6 (hardware cvt; the first source of each cvt goes to
// the upper four bits of its byte).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float x0, float x1, float x2, float x3, float x4, float x5,
                                               float x6, float x7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(x4), "f"(x5), "f"(x6), "f"(x7));
  return r;
}

// One 32-element block as E2M1 codes (16 bytes, two codes a byte, the lower element in
// the lower four bits) with its E8M0 scale byte, returned: the OCP MX rule with E2M1's
// largest exponent, e = floor(log2(amax)) - 2.
__device__ __forceinline__ uint32_t quant_block32_e2m1(const float (&v)[32], uint32_t (&codes)[4]) {
  float m[11];
#pragma unroll
  for (int j = 0; j < 10; ++j) m[j] = absmax3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
  m[10] = absmax3(v[30], v[31], v[31]);
  const float n0 = absmax3(m[0], m[1], m[2]), n1 = absmax3(m[3], m[4], m[5]);
  const float n2 = absmax3(m[6], m[7], m[8]), n3 = absmax3(m[9], m[10], m[10]);
  const float amax = absmax3(absmax3(n0, n1, n2), n3, n3);
  const int e = mx_scale_exp_t<2>(amax);
  const uint32_t sb = __float_as_uint(exp2_neg(e));
  const uint64_t ss = (static_cast<uint64_t>(sb) << 32) | sb;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = v[8 * w + i];
#pragma unroll
    for (int i = 0; i < 8; i += 2) mul_f32x2(x[i], x[i + 1], ss);
    codes[w] = cvt_e2m1x8(x[0], x[1], x[2], x[3], x[4], x[5], x[6], x[7]);
  }
  return static_cast<uint32_t>(e + 127);
}

// ------------------------------------------------------------------ CTA pairs (cta_group::2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the cluster: arrive, then wait for all of them.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on a barrier of either CTA of the pair (a shared::cluster address) with the default
// semantics (release at CTA scope).  The epilogue's arrive that frees an accumulator needs
// no more: its tensor-memory loads have completed (tcgen05.wait::ld) and been fenced
// (tcgen05.fence::before_thread_sync) before it; a cluster-scope release here cost the
// epilogue warps a memory barrier on every tile.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an mbarrier
// of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, uint32_t mbar_cluster, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(mbar_cluster), "r"(x), "r"(y)
      : "memory");
}

// TMEM allocation shared by the CTA pair: one warp of EACH CTA executes these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// M=256 MMA across the pair: A rows 0..127 and the first half of B's rows from this
// (leader) CTA's shared memory, A rows 128..255 and B's second half from the peer's,
// at the same offsets; each CTA's TMEM receives its 128 rows of D.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this shared-memory offset in every CTA of `mask` once the
// pair's prior tcgen05 operations are done.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------ block-scaled (MXFP8)

// Contiguous bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory descriptor without swizzling (descriptor version 1, layout type 0).
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  return d;
}

// 32 rows x 128 bits from shared memory into TMEM lanes 0..31 of every lane quarter
// (4 columns from `taddr`).
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}

// D[tmem] (+)= A * B^T for one K=32 slice of E4M3 codes, each operand scaled per
// 32-element block by its E8M0 factors held in TMEM.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// CTA-pair forms (issued by the leader): the copy runs in both CTAs of the pair, each from
// its own shared memory (same address) into its own TMEM; the MMA spans both CTAs (M =
// 256), each holding its 128 rows of A, half of B's rows, the scale factors of its A rows
// and those of all of B's rows.
__device__ __forceinline__ void tc_cp_32x128b_x4_pair(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}
// 128 rows x 256 bits from each CTA's shared memory into TMEM lanes 0..127 (8 columns from
// `taddr`) of each CTA of the pair; the source is K-major without swizzle: row r's two 16-byte
// halves at r * 16 (8-row groups `sbo` apart) and `lbo` bytes further.
__device__ __forceinline__ void tc_cp_128x256b_pair(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::mxf8f6f4 with an E4M3 A, UE8M0 scales, fp32 D:
//   bits 4-5 B scale-factor id, 7-9 A format (0 = E4M3), 10-12 B format (0 = E4M3,
//   5 = E2M1), 15/16 majorness (0 = K-major), 17-22 N>>3, bit 23 scale type (1 =
//   UE8M0), 24-28 M>>4, 29-30 A scale-factor id (which byte of each 32-bit scale word).
constexpr int MX_FMT_E4M3 = 0;
constexpr int MX_FMT_E2M1 = 5;
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_id, int b_fmt = MX_FMT_E4M3) {
  return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(b_fmt) << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) |
         (static_cast<uint32_t>(sf_id) << 29);
}

}  // namespace moe
