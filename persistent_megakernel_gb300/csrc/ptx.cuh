// Inline-PTX helpers for sm_103a: mbarriers, bulk asynchronous copies (the TMA engine's
// non-tensor mode), GPU-scope acquire/release on global counters, %globaltimer.
#pragma once
#include <stdint.h>

#include "dec_internal.h"

namespace decimpl {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of a phase's completion.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Generic-proxy accesses to shared memory before this point are ordered before async-proxy
// (bulk copy) accesses after it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Global -> shared bulk copy completing `bytes` transactions on mbarrier `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The same copy with an L2 cache policy (createpolicy): weights and KV history stream through
// L2 once per step, so they are marked evict-first and leave the step's activations resident.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// TMA tensor copy of one 2D box (coordinates: column x, row y of the tensor map) into shared
// memory, completing its bytes on mbarrier `bar`. x times the element size must be a multiple of
// 16 bytes; dst 1024-byte aligned for a 128-byte swizzle.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Four 8x8 matrices of 16-bit elements from shared memory (lane l gives the address of row l % 8
// of matrix l / 8); register q receives row (lane / 4), columns 2 (lane % 4) .. +1 of matrix q.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// The same, each matrix transposed: register q receives column (lane / 4), rows 2 (lane % 4) .. +1.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A B + D on the tensor cores, one warp: A 16x16 bf16 (row-major fragments), B 16x8 bf16
// (column fragments), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
      " {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> packed bf16x2 (round to nearest even; the first in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Order this thread's earlier generic-proxy view of global memory before its later bulk
// (async-proxy) copies.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ int32_t ld_relaxed_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_s32(int32_t* p, int32_t v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Arrival with no ordering: the data it announces carries its own tags.
__device__ __forceinline__ void red_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Barrier of the consumer threads only (the producer warp never joins). Not .aligned: a
// thread may arrive from a slow path its warp-mates skipped (a late word, a counter wait), and
// an aligned barrier reached by a diverged warp is undefined.
__device__ __forceinline__ void consumer_sync() {
  asm volatile("barrier.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Barrier of the consumers that also ANDs a predicate over them: every thread gets the same
// verdict, so no consumer can leave a loop that the others stay in. Not .aligned (see above).
__device__ __forceinline__ bool consumer_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.and.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(kConsumerThreads)
      : "memory");
  return r != 0u;
}

// Data-carrying flags: an activation element is a 64-bit word, the fp32 value in the low half
// and the tag of the step that wrote it in the high half, stored with one relaxed 8-byte store
// (single-copy atomic). A reader polls the data itself until the tag is the current step's:
// no fence on the writer's side, no counter round trip on the reader's (the sentinel-in-data
// idea of the Muse Spark Open megakernel article, section "three bills").
__device__ __forceinline__ uint64_t tagged(float v, uint32_t tag) {
  return ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
}

__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(tagged(v, tag)) : "memory");
}

__device__ __forceinline__ void st_tagged4(uint64_t* p, float4 v, uint32_t tag) {  // p 32-byte aligned
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(tagged(v.x, tag)), "l"(tagged(v.y, tag))
               : "memory");
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p + 2), "l"(tagged(v.z, tag)), "l"(tagged(v.w, tag))
               : "memory");
}

#ifndef DEC_TAGGED_LD_CG
#define DEC_TAGGED_LD_CG 0
#endif
#if DEC_TAGGED_LD_CG
// Build option: tagged words read with weak L2 loads (cache-global, L1 bypassed). Timed against
// the relaxed form below, the two differ by 0.2 % per step; weak loads racing with the writers'
// relaxed stores are outside the memory model, so they are not the default.
#define DEC_LD_TAGGED "ld.global.cg"
#else
// Tagged words are read with relaxed gpu-scope loads: each 8-byte element is single-copy atomic
// with the writer's relaxed 8-byte store, so a word's tag vouches for its value, and a re-poll is
// guaranteed to see the store eventually. volatile keeps a re-poll from being folded.
#define DEC_LD_TAGGED "ld.relaxed.gpu.global"
#endif
__device__ __forceinline__ void ld_tagged2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile(DEC_LD_TAGGED ".v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
  uint64_t a;
  asm volatile(DEC_LD_TAGGED ".b64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
  return a;
}

__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float value_of(uint64_t w) { return __uint_as_float((uint32_t)w); }

// Two fp32 fused multiply-adds in one instruction: (a.x*b.x + c.x, a.y*b.y + c.y), each rounded
// as fmaf would.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two e4m3fn codes (low byte = first element) -> two floats; exact (e4m3 is a subset of f16).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes) {
  float2 r;
  asm("{ .reg .b16 t, lo, hi; .reg .b32 h; cvt.u16.u32 t, %2; cvt.rn.f16x2.e4m3x2 h, t; mov.b32 {lo, hi}, h;"
      " cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
      : "=f"(r.x), "=f"(r.y)
      : "r"(two_bytes));
  return r;
}

// Two e2m1 codes in one byte (low nibble = first element) -> two floats; exact.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  float2 r;
  asm("{ .reg .b8 t; .reg .b16 s, lo, hi; .reg .b32 h; cvt.u16.u32 s, %2; cvt.u8.u16 t, s;"
      " cvt.rn.f16x2.e2m1x2 h, t; mov.b32 {lo, hi}, h; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
      : "=f"(r.x), "=f"(r.y)
      : "r"(byte));
  return r;
}

// fp32 -> e4m3fn code: round to nearest even, saturated to +-448 (cvt.rn.satfinite; the second
// source converts into the low byte).
__device__ __forceinline__ uint8_t e4m3_rn_satfinite(float x) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.f), "f"(x));
  return (uint8_t)(h & 0xFFu);
}

// E8M0 scale code -> 2^(e-127) as float (e = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
  return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

}  // namespace decimpl
