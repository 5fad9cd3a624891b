// Shared device-side definitions of the Kitty GB300 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kitty.h"

namespace kitty {

constexpr int kD = 128;      // head_dim
constexpr int kPage = 32;    // tokens per page
constexpr int kVGroup = 32;  // channels per Value group

// Byte offsets inside one (page, kv-head) blob for a given n_hi (multiple of 16),
// Key plane width w = lo_bit (2: the (4, 2) configuration, 4: (8, 4)) and Value
// code width v (2, or 4 with w = 4).
struct BlobLayout {
  int n_hi;
  int kbase, kextra, ks, km, kch, vbase, vs, vm, bytes;
  __host__ __device__ BlobLayout(int nh, int w, int v) : n_hi(nh) {
    kbase = 0;
    kextra = 512 * w;
    ks = kextra + nh * 4 * w;
    km = ks + 256;
    kch = km + 256;
    vbase = kch + nh;
    vs = vbase + 512 * v;
    vm = vs + 256;
    bytes = vm + 256;
  }
};

__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

template <int DT>
__device__ __forceinline__ float load16(const uint16_t* p) {
  const uint16_t b = *p;
  if (DT == KITTY_BF16) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float bits16_to_f32(uint16_t b, int dt) {
  return dt == KITTY_BF16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Start pulling [ptr, ptr + bytes) into L2 (no completion to wait for);
// ptr 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void l2_prefetch(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}



__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Polls a barrier phase at most `limit` times; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_test(bar, parity)) return true;
    if (i > 64) __nanosleep(32);
  }
  return false;
}


// Barrier arrive / expect-tx and 1-D bulk copy on 32-bit shared-space
// addresses (precomputed once, so the hot loop does no generic-to-shared
// conversion).  bulk_g2s_s: global -> shared, completion counted on `bar`;
// bytes % 16 == 0, both addresses 16-byte aligned.
__device__ __forceinline__ void mbar_arrive_expect_tx_s(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_s(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ bool mbar_test_s(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s_s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Packed fp32x2 arithmetic: two IEEE round-to-nearest operations (no flush to
// zero) in one instruction, lane for lane the same results as __fadd_rn etc.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ void add2_rn(float& a, float& b, float c, float d) {  // (a, b) += (c, d)
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2pack(a, b)), "l"(f2pack(c, d)));
  f2unpack(r, a, b);
}
__device__ __forceinline__ void sub2_rn(float& ra, float& rb, float a, float b, float c, float d) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2pack(a, b)), "l"(f2pack(c, d)));
  f2unpack(r, ra, rb);
}
__device__ __forceinline__ void mul2_rn(float& ra, float& rb, float a, float b, float c, float d) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2pack(a, b)), "l"(f2pack(c, d)));
  f2unpack(r, ra, rb);
}

// D(16x8 f32) += A(16x16 f16) * B(16x8 f16), warp-wide.
__device__ __forceinline__ void mma_f16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// D(16x8 f32) += A(16x16) * B(16x8), both 16-bit of type DT.
template <int DT>
__device__ __forceinline__ void mma16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if (DT == KITTY_BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

// (high, rest) of a probability in the 16-bit type: the high part keeps the
// type's significand (11 bits for fp16, 8 for bf16) exactly, the rest is
// rounded once.
template <int DT>
__device__ __forceinline__ uint32_t prob_pair(float p) {
  if (DT == KITTY_BF16) {
    const float t = __uint_as_float(__float_as_uint(p) & 0xFFFF0000u);
    const __nv_bfloat162 h = __floats2bfloat162_rn(t, p - t);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  const float t = __uint_as_float(__float_as_uint(p) & 0xFFFFE000u);
  return h2_bits(__floats2half2_rn(t, p - t));
}

// 16-byte asynchronous global-to-shared copy (L2 only), its group commit and wait.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace kitty
