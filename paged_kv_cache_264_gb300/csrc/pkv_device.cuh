// pkv_device.cuh -- small device helpers for sm_103a: shared-memory mbarriers, bulk
// asynchronous global->shared copies (the 1-D form of the tensor-memory-accelerator
// copy), a bounded mbarrier wait, and bit-level conversions of bf16 and int8 to fp32.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the asynchronous proxy before any copy
// signals the barrier.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// asynchronous-proxy writes to the same memory (a stage is refilled after it was read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Test the phase; while it is incomplete the thread may be suspended for up to
// `suspend_ns` (it wakes as soon as the phase completes), so a waiting warp does not spin
// on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity,
                                              uint32_t suspend_ns = 1000000u) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the barrier phase with the given parity to complete.  Gives up (returns
// false) after limit_ns of wall time (kWaitTimeoutNs in the kernels) or 2^26 polls,
// whichever comes first, so that a lost copy can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// Shared-memory load by shared-window address (ld.shared rather than a generic load).
// Volatile, so it stays after the mbarrier wait (also volatile asm) that publishes the data.
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// 2^x for the softmax (x <= 0 in practice): the hardware base-2 exponential, flushing
// subnormal results to zero (weights below 2^-126 do not matter next to the largest, 1).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^e as an fp32 for an integer e in [-126, 127], built from its exponent bits.
__device__ __forceinline__ float pow2i(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// L2 policy for data read once per call (the K/V tiles): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for data read again soon by another CTA (the K/V tiles of a kv head whose query
// columns are split into chunks): evict last.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (multiple of 16) from global to this CTA's shared memory;
// completion is signalled on `bar` through its transaction count.  Both addresses
// must be 16-byte aligned.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled tensor copy global -> shared through a tensor map (TMA); completion is
// signalled on `bar`.  x is the inner (element) coordinate, y the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Four 8x8 b16 matrices from shared memory; lane l gives the row address of matrix l / 8.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held one row pair per lane (lane 4i+j: row i, cols 2j, 2j+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D(16x8, fp32) += A(16x16) * B(16x8), bf16 or fp16 operands.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Two int8 codes -> fp16x2 holding 1152 + code, exactly.  `u` holds codes with their sign
// bits flipped (u = x + 128); `sel` picks two bytes (0x4140: bytes 0 and 1, 0x4342: bytes 2
// and 3).  Placing u in the low mantissa byte of the fp16 1024 (0x6400) gives 1024 + u
// exactly (fp16 has 10 mantissa bits).  Callers remove the 1152 offset after the matrix
// product.
__device__ __forceinline__ uint32_t f16x2_biased(uint32_t u, uint32_t sel) {
  return __byte_perm(u, 0x64646464u, sel);
}

// True in exactly one lane of the (fully active) warp: elect.sync picks a leader.  Copy
// issue code runs on the whole warp with warp-uniform values and only the copy
// instructions sit under this test; measured on GB300 that costs fewer instructions than
// running the whole issue path in lane 0 alone (int8_cb decode 172.9 -> 166.9 us, 6 %
// fewer instructions).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialisation
// may start while the previous kernel in the stream is still finishing; griddep_wait()
// returns once that kernel has completed and its writes are visible, so it must precede
// every read of data a previous kernel may have written.  griddep_launch_dependents()
// lets the next kernel's launch begin once every CTA of this one has called it (or exited);
// the decode kernels call it when a CTA has no more work, the append kernels at their
// start.  Both are no-ops for ordinary launches.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- FP8 E4M3.  Every E4M3 value (|x| <= 448, spacing >= 2^-9) is exact in fp16.
// Four E4M3 codes of a word -> two fp16x2: bytes 0,1 -> lo (byte 0 in the low half), bytes
// 2,3 -> hi.  The word is split into its 16-bit halves by register aliasing.
__device__ __forceinline__ void f16x2x2_from_e4m3x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Nearest E4M3 codes of two fp32 values, ties to even, saturating at +-448: lo -> byte 0,
// hi -> byte 1.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four E4M3 codes of a word -> four fp32 values.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
  uint32_t lo, hi;
  f16x2x2_from_e4m3x4(w, lo, hi);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// ---- conversions.  A bf16 is the upper 16 bits of an fp32, so widening is a shift.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// int8 -> fp32 without the integer-to-float unit: for a code x, the byte u = x + 128
// (x with its sign bit flipped) placed in the low mantissa bits of 2^23 gives the fp32
// value 2^23 + u exactly (binary32 has 23 mantissa bits); subtracting 2^23 + 128 leaves
// x exactly.  `u4` holds four codes with their sign bits already flipped.
__device__ __forceinline__ float i8_from_flipped(uint32_t u4, int i) {
  const uint32_t bits = __byte_perm(u4, 0x4B000000u, 0x7540u | static_cast<uint32_t>(i));
  return __uint_as_float(bits) - 8388736.0f;
}

}  // namespace pkv
