// Device helpers shared by the coli_moe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define COLI_DEV __device__ __forceinline__

namespace coli {

// Status codes latched on the device (same values as coli_status).
constexpr int kErrDevice = -5;
constexpr int kErrTimeout = -6;

// Every bounded wait gives up after this long (a healthy wait takes µs).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// First error wins; later errors leave the word untouched.
COLI_DEV void latch_error(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

COLI_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- bf16 <-> f32 --------------------------------------------------------
COLI_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
COLI_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <typename T>
COLI_DEV float to_f32(T v);
template <>
COLI_DEV float to_f32<float>(float v) { return v; }
template <>
COLI_DEV float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Two floats -> packed bf16x2 (low half = a), round to nearest even.
COLI_DEV uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}

// ---- global loads ----------------------------------------------------------
// Streamed once (expert weights): bypass L1, 256-byte L2 fetch granule.
COLI_DEV uint4 ldg_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
// Re-read by neighbouring warps (activations): keep in L1.
COLI_DEV uint4 ldg_keep(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// 16-byte asynchronous global -> shared copy (L1 bypassed, 256-byte L2 fetch),
// grouped with cp_async_commit and completed with cp_async_wait<N>.
COLI_DEV void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(dst), "l"(src)
               : "memory");
}
COLI_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
COLI_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
COLI_DEV uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

COLI_DEV uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// ---- warp-level tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate) --------
COLI_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A x B with a zero accumulator input (no registers to clear first).
COLI_DEV void mma_bf16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// ---- shared memory / mbarrier ---------------------------------------------
COLI_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

COLI_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

COLI_DEV void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

COLI_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}

COLI_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false once
// timeout_ns has passed (the caller latches kErrTimeout and unwinds).
COLI_DEV bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// ---- int4 -> bf16 ------------------------------------------------------------
// int4 -> bf16 without an offset subtraction. A repacked word holds the 8
// indices 8w..8w+7 with even ones in nibbles 0-3 and odd ones in 4-7, so
// nibbles (p, p+4) are the consecutive pair (2p, 2p+1). One LOP3 per pair
// flips the nibble's sign bit and drops it into the low mantissa bits of a
// bf16 whose exponent makes the value exactly 136 + q:
//   ((w >> 4p) & 0x000F000F) ^ 0x43084308  ->  bf16x2 (136 + q_2p, 136 + q_2p+1)
// The decode MMA thus sums (136 + q) x and subtracts 136 * sum(x) over the
// group (a per-token table) to leave the exact sum q x; the prefill
// converter subtracts the 136 from the bf16 values instead.
COLI_DEV uint32_t nib_pair136(uint32_t w, int p) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(w >> (4 * p)), "r"(0x000F000Fu),
      "r"(0x43084308u));
  return r;  // (v & mask) ^ x
}

COLI_DEV uint4 dequant136(uint32_t w) {
  return make_uint4(nib_pair136(w, 0), nib_pair136(w, 1), nib_pair136(w, 2), nib_pair136(w, 3));
}

COLI_DEV uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// bf16x2 a * b + c, one rounding per half (round to nearest even).
COLI_DEV uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

COLI_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

// ---- OCP Microscaling element codes ------------------------------------------
// Every E4M3 and E2M1 value is exact in fp16; the hardware converts two codes
// to an fp16 pair in one instruction.
// 8 E4M3 codes (two words, lower address first) -> four fp16 pairs.
COLI_DEV void e4m3x8_f16(uint32_t w0, uint32_t w1, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b16 a, b, c, d;\n\t"
      "mov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t"
      "cvt.rn.f16x2.e4m3x2 %2, c;\n\tcvt.rn.f16x2.e4m3x2 %3, d;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w0), "r"(w1));
}

// 8 E2M1 codes (one word, low nibble = even index) -> four fp16 pairs.
COLI_DEV void e2m1x8_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 a, b, c, d;\n\t"
      "mov.b32 {a, b, c, d}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, a;\n\tcvt.rn.f16x2.e2m1x2 %1, b;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c;\n\tcvt.rn.f16x2.e2m1x2 %3, d;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

}  // namespace coli
