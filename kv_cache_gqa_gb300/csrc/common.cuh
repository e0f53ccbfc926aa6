// Device helpers shared by the kernels of the KV-cache GQA attention step.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kv_attn.h"

namespace kva {

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Element types: float (KVA_F32) and raw bf16 bits (KVA_BF16)
// ---------------------------------------------------------------------------
struct bf16_t { uint16_t bits; };

template <typename T> struct ElemSize;
template <> struct ElemSize<float> { static constexpr int value = 4; };
template <> struct ElemSize<bf16_t> { static constexpr int value = 2; };

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// float -> bf16 bits, round to nearest, ties to even (inputs are finite).
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two floats to packed bf16 pairs, round to nearest even, lo in bits 0..15: one instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Load 8 consecutive elements (16-byte aligned for bf16, 32-byte for float) as floats.
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16_t* p, float (&x)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
  x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
}
// Store 8 floats as 8 consecutive elements with 128-bit stores.
__device__ __forceinline__ void store8(float* p, const float (&y)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
}
__device__ __forceinline__ void store8(bf16_t* p, const float (&y)[8]) {
  uint4 w;
  w.x = pack_bf16x2(y[0], y[1]); w.y = pack_bf16x2(y[2], y[3]);
  w.z = pack_bf16x2(y[4], y[5]); w.w = pack_bf16x2(y[6], y[7]);
  *reinterpret_cast<uint4*>(p) = w;
}

__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const bf16_t* p) { return __uint_as_float(((uint32_t)p->bits) << 16); }

// ---------------------------------------------------------------------------
// Ordered 64-bit keys for an argmax with ties toward the lowest index:
// the high word orders float values, the low word holds ~index.  -0.0 is keyed as +0.0,
// so a logit of -0 and one of +0 are equal and the lower index wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t float_order_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_from_order_bits(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  return ((unsigned long long)float_order_bits(v) << 32) | (unsigned long long)(0xffffffffu - idx);
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier and bulk async copies (global -> shared)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// cos and sin of the rotary angle a = p * inv, with inv = ih + il split into a float pair on
// the host.  For |p| < 2^24 the position is exact in float and the product is carried as
// hi + lo (the rounding error of p * ih recovered with an fma), then reduced by 2 pi in the
// Cody-Waite way with a two-part constant (the first product k * C1 cancels exactly), so
// the float sin/cos see a short argument (within pi, or 2 pi when the float estimate of k
// is off by one for very large angles) accurate to a few float ulps of pi.  Larger
// positions take the same steps in float64.
__device__ __forceinline__ void rope_cos_sin(int32_t p, float ih, float il, double inv, float* c, float* s) {
  if (p > -(1 << 24) && p < (1 << 24)) {
    const float pf = (float)p;
    const float hi = pf * ih;
    const float lo = fmaf(pf, ih, -hi) + pf * il;
    const float k = rintf(hi * 0.159154943f);
    float r = fmaf(-k, 6.28318548f, hi);                  // C1 = float(2 pi): exact
    r = fmaf(-k, -1.74845553e-7f, r) + lo;                // C2 = 2 pi - C1
    sincosf(r, s, c);
  } else {
    const double a = (double)p * inv;
    const double k = rint(a * 0.15915494309189535);
    sincosf((float)fma(-k, 6.283185307179586, a), s, c);
  }
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization may
// start while the grid before it on the stream is still running: it sets up shared memory,
// then griddep_wait() blocks until that grid has completed and its writes are visible.  No
// global memory may be read or written before the wait.  griddep_launch_dependents() lets the
// grid after this one start its own set-up (it still waits for this grid to complete).
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
// Bring [p, p + bytes) into L2 (bulk; p 16-byte aligned, bytes a multiple of 16; a hint).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}
// Bring the 128-byte line holding p into L2 (a hint: no data returned, nothing to wait for).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(phase) : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits that gave up in the kernels of this translation unit since the last reset (each unit
// has its own copy; the host side sums them, see register_wait_counter below).
static __device__ unsigned int g_wait_timeouts;

// Bounded wait: polls the barrier and gives up after WAIT_LIMIT_NS of wall time, counts the
// give-up in g_wait_timeouts and returns false (the caller stops using the buffer and marks
// its outputs), so a lost transaction can never hang the GPU.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, phase)) return true;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      atomicAdd(&g_wait_timeouts, 1u);
      return false;
    }
  }
}

// Host side: every translation unit that includes this header registers a reader of its
// g_wait_timeouts when the library loads; kva_wait_timeouts() sums them.
void register_wait_counter(cudaError_t (*read)(unsigned* value, bool reset));
namespace {
cudaError_t read_wait_timeouts_here(unsigned* value, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_wait_timeouts, sizeof(unsigned));
  if (e == cudaSuccess && reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero));
  }
  return e;
}
struct WaitCounterRegistration {
  WaitCounterRegistration() { register_wait_counter(&read_wait_timeouts_here); }
};
const WaitCounterRegistration g_wait_counter_registration;
}  // namespace

// 1-D bulk copy global -> shared, completion signalled on `bar` as transaction bytes.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}


}  // namespace kva
