// Device helpers shared by the bf16 tensor-core kernels: bounded waits with a
// CTA-wide abort flag, the gate's logistic function, packed-fp16 arithmetic and
// swizzled shared-memory addressing.
#pragma once

#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_shapes.h"

namespace tri_tc {

struct Abort {
  int* flag;              // shared-memory flag: nonzero once any role gave up
  unsigned int* dev_err;  // handle's device error word
  long long polls;        // poll cap of ordinary waits
};

// Bounded wait; on time-out or when another role has already aborted, raises
// the abort flag (and records a time-out) and returns false.
__device__ __forceinline__ bool wait_or_abort_slow(uint64_t* bar, uint32_t parity, const Abort a) {
  const uint64_t t0 = tc::global_timer_ns();
  for (long long n = 1; n < a.polls; ++n) {
    // Sleeps up to 20 us per poll instead of spinning; the phase wakes it.
    if (tc::mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if (tc::lds_volatile(a.flag)) return false;
    if ((n & 15) == 0 && tc::global_timer_ns() - t0 > 2000000000ull) break;
  }
  *(volatile int*)a.flag = 1;
  atomicOr(a.dev_err, TRI_DEV_ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const Abort& a) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  return wait_or_abort_slow(bar, parity, a);
}

// Warp-uniform form for warps that go on to issue warp-collective tcgen05
// loads: every lane waits, and the warp proceeds only if all lanes succeeded.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, const Abort& a) {
  const bool ok = wait_or_abort(bar, parity, a);
  return __all_sync(0xffffffffu, ok);
}

// Drain wait used at teardown: ignores the abort flag and the poll cap so that
// copies and MMAs still in flight land before the CTA releases its memory.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  tc::mbar_wait(bar, parity, 1ll << 40);
}

// Logistic function for the gate, 1/(1 + e^-z) = (1 + tanh(z/2)) / 2, with the
// hardware tanh approximation (one special-function operation; its error is
// well below the bf16 rounding the gate gets).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_approx(float z) {
  return fmaf(0.5f, tanh_approx(0.5f * z), 0.5f);
}

// Packed fp16 arithmetic of the attention's softmax. cvt_f16x2: two fp32
// values rounded to an fp16 pair (lo in the low half); hadd2: pairwise sum;
// ex2_f16x2: 2^x of both halves in one special-function operation (relative
// error about 2^-10, subnormal results kept, 2^-inf = 0).
__device__ __forceinline__ uint32_t cvt_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t r;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
// The two halves of an fp16 pair, each widened to fp32, added in fp32.
__device__ __forceinline__ float f16x2_sum(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(h));
  return lo + hi;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Programmatic dependent launch. Every kernel of the path is launched so that
// it may start while the previous kernel on the stream is still running; its
// threads run the prologue that reads nothing another kernel writes (barrier
// setup, tensor-memory allocation, the resident weights), then pdl_wait()
// blocks until the previous kernel has completed and its writes are visible.
// pdl_trigger() lets the next kernel start as soon as every CTA of this one has
// called it (or exited); it only releases the launch, not the data.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Shared-memory descriptor swizzle mode for rows of `bytes` (32, 64 or 128).
__host__ __device__ constexpr uint32_t swz_mode(int bytes) {
  return bytes == 128 ? tc::SWZ_128B : bytes == 64 ? tc::SWZ_64B : tc::SWZ_32B;
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile whose rows are
// `row_bytes` (32, 64 or 128) long, swizzled as TMA writes it with the swizzle
// of the same span: address bits 4.. XOR the bits 7.. of the same address.
__host__ __device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk, uint32_t row_bytes) {
  return row_bytes == 32 ? row * 32u + ((chunk ^ ((row >> 2) & 1u)) << 4)
                         : tc::swz_offset(row, chunk, row_bytes);
}

}  // namespace tri_tc
