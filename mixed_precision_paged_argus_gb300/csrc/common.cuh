// Shared device helpers of the argus library: hand-written PTX wrappers for
// mbarriers, bulk asynchronous copies, fp8 / fp16 / bf16 conversions, the
// m16n8k16 tensor-core MMA and register-level 8x8 transposes, plus host-side
// status reporting.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/argus.h"

namespace argus {

// ----------------------------------------------------------------------------
// Host side: status reporting
// ----------------------------------------------------------------------------
argus_status fail(argus_status s, const char* fmt, ...);
argus_status launch_status(const char* what);
int device_sm_count();

// Device address of a pool's codes and meta: device pools as given; host pools
// (ARGUS_PLACE_HOST, page-locked) through cudaHostGetDevicePointer.  Returns
// ARGUS_E_INVALID for an unknown placement or host memory the device cannot map.
argus_status pool_device_ptrs(const argus_pool& pool, const void** codes, const void** meta);

// Identifier of the calling thread's current CUDA context, unique for the life
// of the process; 0 when no context is current or the driver cannot say.
unsigned long long context_id();

// One-time setup per device that must be redone in a new context: kernel
// attributes, resolved symbol addresses.  A device's context changes when it is
// destroyed and created again (cudaDeviceReset), and whatever was set up in the
// old one no longer holds, so the record is keyed on the context identifier.
struct PerContext {
  unsigned long long ctx[64] = {};
  std::mutex mu;

  // Runs setup(dev) unless it already succeeded in the current context of the
  // current device; returns its status.  Without a context identifier the
  // setup runs on every call.
  template <class F>
  argus_status ensure(F&& setup) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
      return fail(ARGUS_E_LAUNCH, "no current CUDA device");
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = context_id();
    if (id != 0 && ctx[dev] == id) return ARGUS_OK;
    const argus_status st = setup(dev);
    ctx[dev] = (st == ARGUS_OK) ? context_id() : 0ull;   // setup may have created the context
    return st;
  }
};

// Upper bound on any wait (nanoseconds of %globaltimer); a wait that runs out
// sets the top bit of the caller-visible status word and the kernel winds down.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr uint32_t kStatusTimeoutBit = 0x80000000u;

// ----------------------------------------------------------------------------
// mbarrier and bulk-copy PTX
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
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

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity; false if it never came
// within kWaitLimitNs, or if *abort (a CTA-wide error flag in shared memory)
// was raised meanwhile, so that one failed wait ends every other wait quickly.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const volatile uint32_t* abort = nullptr,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (abort && *abort) return false;
      if (global_ns() - t0 > limit_ns) return false;
    }
  }
}

// One-dimensional bulk copy global -> shared, completion signalled on `bar`
// as transaction bytes.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ----------------------------------------------------------------------------
// Conversions
// ----------------------------------------------------------------------------
// Two e4m3 codes (low byte -> low half) to an exact f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t out;
  uint16_t in = static_cast<uint16_t>(two_codes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
  return out;
}

// Two fp32 values to e4m3 codes, round to nearest even, saturating at +-448:
// returns lo's code in bits 0..7 and hi's code in bits 8..15.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t out;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(out) : "r"(a), "r"(b), "r"(sel));
  return out;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  // (a & mask) | orv
  uint32_t out;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(out) : "r"(a), "r"(mask), "r"(orv));
  return out;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Two IEEE fp32 operations in one instruction (packed f32x2, sm_100 and later):
// each lane is rounded to nearest even exactly as its scalar form, and nothing
// is contracted into a fused multiply-add that the scalar code would not form.
#define ARGUS_F2_BINARY(name, op)                                                              \
  __device__ __forceinline__ void name(float& d0, float& d1, float a0, float a1, float b0, float b1) { \
    asm("{\n\t.reg .b64 a, b, d;\n\t"                                                         \
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t" op                                   \
        " d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"                                               \
        : "=f"(d0), "=f"(d1)                                                                    \
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));                                                 \
  }
ARGUS_F2_BINARY(f2_add, "add.rn.f32x2")
ARGUS_F2_BINARY(f2_sub, "sub.rn.f32x2")
ARGUS_F2_BINARY(f2_mul, "mul.rn.f32x2")
#undef ARGUS_F2_BINARY
__device__ __forceinline__ void f2_fma(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                       float c1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------------------
// Tensor-core MMA (m16n8k16, fp32 accumulate) and 8x8 register transpose
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

}  // namespace argus
