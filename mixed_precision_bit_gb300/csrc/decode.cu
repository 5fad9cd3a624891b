// Kitty split-K paged decode attention for GB300 (sm_103a).
//
// Paper: "Kitty: Accurate and Efficient 2-bit KV Cache Quantization with
// Dynamic Channel-wise Precision Boost", Abstract (page dequantization over a
// coalesced page-centric layout, no scattered reads or per-channel masks);
// FlashAttention-style online softmax and PagedAttention block tables (both
// cited there).
//
// One CTA = (kv head, sequence, group of up to 4 query heads, split); 4 warps,
// each streaming every 4th page of the split.  (Query groups above 4 in the
// (4, 2) format take decode8_kernel: 8 heads per CTA, two head sets per warp.)
// Split sizes shrink from the first split to the last and the grid is
// split-major, so the CTAs dispatched last are the short ones
// (longest-processing-time-first order: the grid ends with little idle time on
// the SMs).  A split's page range does not depend on the sequence length, so a
// CTA requests its lengths, query rows and block-table entries together and
// starts its page copies one memory round trip after it starts.  A warp stages
// whole (page, kv-head) blobs into shared memory with 1-D bulk copies
// (cp.async.bulk + mbarrier; 4 stages per warp for 2-bit Key planes, 3 for 4-bit
// planes), then computes, for its g <= 4 query heads:
//   scores  S^T[t][n] = sum_c code[t][c] * B[c][n] on the tensor cores
//           (mma.m16n8k16, fp32 accumulate) with B = q*S, the per-channel Key
//           step folded into the query: the query is split into a high part
//           (4 significant bits, column 2h of head h) and the rest (column
//           2h+1), and a stored step has at most 7 significant bits, so each
//           column is one exact fp16 multiply; plus the extra plane of the
//           boosted channels (B = q*S/2^W gathered through the channel list,
//           W = Key plane width) and the q.M term as a one-row MMA;
//   softmax fp32 online (max, rescale, exp2) in registers;
//   PV      O^T[c][n] = sum_t vcode[c][t] * P'[t][n] with P' = p*S_v per
//           Value group, p split the same way (high part exact times S_v, the
//           rest rounded once), plus the sum_t p*M_v term.
// Codes are unpacked with one AND per two: the planes are stored in fragment
// order with every word rotated left by two bits, so a masked 16-bit half is
// the fp16 subnormal code * 2^(2*tau + 2 - 24) (2-bit planes) or
// code * 2^(4*(tau & 1) + 2 - 24) (4-bit planes); the power of two depends only
// on the tile row and is folded into the score scale (Keys) or the final output
// (Values).  The 4 warps merge their states in the fragment layout through
// their own idle stage buffers, each warp finishing a quarter of the channels;
// splits merge in a separate combine kernel.  The rotation keeps the codes out of the lowest mantissa bits:
// measured on the GB300, the PV products of codes in mantissa bits 0-1 kept an
// error near 2^-13 of the output's scale over an 8192-token sequence, 4 to 8
// times that of the next two bits up.
#include "kitty_common.cuh"
#include "quant_tile.cuh"
#include "host_common.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <type_traits>
#include <utility>

namespace kitty {
namespace {

constexpr int kDWarps = 4;
// Page stages per warp: 4 for 2-bit Key planes; 3 for 4-bit planes, whose
// larger blobs would otherwise allow only 2 CTAs per SM.
__host__ __device__ constexpr int stages_for(int w) { return w == 4 ? 3 : 4; }
constexpr int kDMinBlocks = 4;  // resident CTAs per SM the register budget is sized for
// An unpacked code c of tile-row class tau has the fp16 value
// c * 2^(row exponent - kCodeExp): the smallest fp16 subnormal is 2^-24, and the
// planes' two-bit rotation lifts every code by 2^2.
constexpr int kCodeExp = 22;
// Query heads per CTA: the 8 columns of an m16n8k16 B operand hold 4 heads as
// (high, low) pairs.  Larger groups (g = Hq/Hkv up to kMaxGroup) take
// ceil(g / 4) head-group CTAs per (sequence, kv head, split), adjacent in the
// grid, which read the same pages (the second read mostly from L2).
constexpr int kHeadsPerCta = 4;
constexpr int kMaxGroup = 32;
constexpr int kDThreads = kDWarps * 32;
// a flush quantizes the tail in the stage buffers: they must hold the page
// quantizer's shared state at the smallest blob (n_hi = 0) of either width
static_assert(sizeof(QuantSmem) <= (size_t)kDWarps * stages_for(2) * 3072 &&
                  sizeof(QuantSmem) <= (size_t)kDWarps * stages_for(4) * 4096,
              "page quantizer state does not fit in the decode stage buffers");
// Row stride (halves) of the extra-plane query tables: 130 rather than 128, so
// that the eight tables (4 heads x high/low part) put one channel's entries in
// eight different shared-memory banks, and the lanes of a warp gathering the
// same channel for different heads and parts do not conflict.
constexpr int kQx = kD + 2;
constexpr uint32_t kWaitLimit = 1u << 22;  // polls of one barrier phase (~0.1-1 s)
constexpr int kPartial = kD + 4;           // split partial: m, l, 2 unused, o[128] (16-byte aligned)
constexpr int kMaxSplits = 256;            // splits per sequence, at most
// Running-max floor (log2 units): finite, so masked scores (-inf) give p = 0 exactly.
constexpr float kNegBig = -1.0e30f;

// Fused append (kitty_append_decode): the new token of every (sequence, kv
// head), written into the tail by that pair's split-0 CTA, which also quantizes
// a full tail into the caller's page.  k_new == nullptr: plain decode.
struct AppendParams {
  const uint16_t* k_new;  // [B][Hkv][128]
  const uint16_t* v_new;
  uint16_t* tail_k;       // the decode's tail_k / tail_v, writable
  uint16_t* tail_v;
  int32_t* tail_len;
  int32_t* num_pages;
  int32_t* block_table;
  float* run_sum;         // running statistics (running or sequence mode), else null
  float* run_sumsq;
  int32_t* run_count;
  const int32_t* flush_page_ids;
  uint8_t* pool;
  int running;
};

struct DecodeParams {
  AppendParams ap;
  const uint16_t* q;
  const uint8_t* pool;
  const int32_t* block_table;
  const int32_t* num_pages;
  const uint16_t* tail_k;
  const uint16_t* tail_v;
  const int32_t* tail_len;
  void* out;
  float* ws;
  int32_t* d_status;
  float sm_log2;  // sm_scale * log2(e)
  uint32_t wait_polls;  // bound of a page wait, in polls of its barrier
  int pool_pages, max_pages, out_dtype, splits, Hkv, Hq, g, HG, n_hi, blob, in_dtype;  // HG: head groups
  // Split s of a sequence with np pages covers pages [starts[s], min(np, starts[s+1]));
  // starts[] rises from 0 to starts[splits] = max_pages.  A split holds work only
  // when it holds a page, except split 0, which always runs (it takes the tail
  // tokens and is the one an empty sequence reports from).
  int32_t starts[kMaxSplits + 1];
};

// Split s holds work for a sequence of np pages.
__device__ __forceinline__ bool split_active(const DecodeParams& p, int s, int np) {
  return np > p.starts[s] || s == 0;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: a dependent grid may start once every CTA of
// this grid has called trigger_dependents (or exited); wait blocks until this
// grid has completed and its memory is visible.  Both are no-ops for a grid
// launched without the attribute.
__device__ __forceinline__ void trigger_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Shared-memory loads from a 32-bit shared address plus a compile-time offset.
template <int OFF>
__device__ __forceinline__ uint32_t ld_s32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 ld_s64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 ld_s128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}
__device__ __forceinline__ uint16_t ld_s16r(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) { return h2_bits(__hmul2(bits_h2(a), bits_h2(b))); }
__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) { return h2_bits(__hsub2(bits_h2(a), bits_h2(b))); }
// An fp16 pair in the 16-bit input type: unchanged for fp16; for bf16 exact
// when the values came from bf16 (at most 8 significant bits).
template <int DT>
__device__ __forceinline__ uint32_t half2_to16(uint32_t h2) {
  if (DT == KITTY_BF16) {
    const __nv_bfloat162 b = __float22bfloat162_rn(__half22float2(bits_h2(h2)));
    return *reinterpret_cast<const uint32_t*>(&b);
  }
  return h2;
}
// The high part of an fp16 value: sign, exponent and the top 3 mantissa bits
// (4 significant bits).  Times a step of at most 7 significant bits it is exact
// in fp16, and the rest (value - high part, exact) has at most 7 significant
// bits left.
__device__ __forceinline__ __half high_part(__half x) {
  return __ushort_as_half((uint16_t)(__half_as_ushort(x) & 0xFF80u));
}


// Four consecutive channels i..i+3 (i % 4 == 0): one vector store when the
// output array is 16-byte aligned, else four scalar stores.
__device__ __forceinline__ void store_out4(void* out, int dt, size_t i, float4 v) {
  if ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
    if (dt == KITTY_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = v;
    } else if (dt == KITTY_BF16) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), c = __floats2bfloat162_rn(v.z, v.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + i) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&c));
    } else {
      *reinterpret_cast<uint2*>(static_cast<__half*>(out) + i) =
          make_uint2(h2_bits(__floats2half2_rn(v.x, v.y)), h2_bits(__floats2half2_rn(v.z, v.w)));
    }
    return;
  }
  if (dt == KITTY_F32) {
    float* o = static_cast<float*>(out) + i;
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  } else if (dt == KITTY_BF16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + i;
    o[0] = __float2bfloat16_rn(v.x); o[1] = __float2bfloat16_rn(v.y);
    o[2] = __float2bfloat16_rn(v.z); o[3] = __float2bfloat16_rn(v.w);
  } else {
    __half* o = static_cast<__half*>(out) + i;
    o[0] = __float2half_rn(v.x); o[1] = __float2half_rn(v.y);
    o[2] = __float2half_rn(v.z); o[3] = __float2half_rn(v.w);
  }
}

__device__ __forceinline__ void store_out(void* out, int dt, size_t i, float v) {
  if (dt == KITTY_F32) static_cast<float*>(out)[i] = v;
  else if (dt == KITTY_BF16) static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else static_cast<__half*>(out)[i] = __float2half_rn(v);
}

// Compile-time blob offsets for NX = n_hi/16 extra-plane k-steps, Key plane
// width W (2: (4, 2) configuration, 4: (8, 4)) and Value code width V (2 or 4).
template <int NX, int W, int V>
struct Off {
  static constexpr int kx = 512 * W, ks = kx + 64 * W * NX, km = ks + 256, kch = km + 256;
  static constexpr int vb = kch + 16 * NX, vs = vb + 512 * V, vm = vs + 256, bytes = vm + 256;
};

// Power of two (exponent + kCodeExp) that an unpacked Value code of
// channel-tile row (m-tile mc, 8-row half rh) carries: 2-bit planes place rows
// at bit 2*tau + 2 (tau = 2*(mc & 1) + rh), 4-bit planes at bit 4*rh + 2.
__host__ __device__ constexpr int vrow_exp(int V, int mc, int rh) {
  return V == 4 ? 4 * rh : 2 * (2 * (mc & 1) + rh);
}

// Lane roles.  Thread (r = lane/4, qq = lane%4) owns head qq in the C
// fragments (column 2qq = high part, 2qq+1 = low part) and, as a B-fragment
// lane, column n = lane/4 = (head lane/8, part (lane/4)&1).
struct Lane {
  int lane, r, qq;
  __device__ Lane() {
    lane = threadIdx.x & 31;
    r = lane >> 2;
    qq = lane & 3;
  }
};

// Per-warp online-softmax state of head qq.
struct WarpState {
  float acc[8][4];  // O^T fragments, m-tile mc = channels 16mc..16mc+15
  float vm[4];      // sum_t p*M_v fragment (rows = Value groups)
  float m;          // running max (log2 units), uniform over the lanes of a head
  float l;          // this thread's partial softmax denominator
};

__device__ __forceinline__ void rescale(WarpState& w, float pm) {
  const float nm = fmaxf(w.m, pm);
  if (__any_sync(0xFFFFFFFFu, nm > w.m)) {
    const float a = ex2(w.m - nm);
#pragma unroll
    for (int mc = 0; mc < 8; ++mc)
#pragma unroll
      for (int i = 0; i < 4; ++i) w.acc[mc][i] *= a;
#pragma unroll
    for (int i = 0; i < 4; ++i) w.vm[i] *= a;
    w.l *= a;
    w.m = nm;
  }
}

// Unpack of a rotated 2-bit plane word: tau 0, 1 (codes in mantissa bits 2-3,
// 4-5) or tau 2, 3 (bits 6-7, 8-9); the word rotated by 8 holds the tile's
// columns 8..15 in the same places.
__device__ __forceinline__ void unpack_rows01(uint32_t x, uint32_t* a) {  // tau 0,1
  const uint32_t x2 = __funnelshift_r(x, x, 8);
  a[0] = x & 0x000C000Cu; a[1] = x & 0x00300030u; a[2] = x2 & 0x000C000Cu; a[3] = x2 & 0x00300030u;
}
// 4-bit planes: one word is one A fragment (rows r, r+8 = mantissa bits 2-5,
// 6-9 of each 16-bit half; the word rotated by 8 holds columns 8..15).
__device__ __forceinline__ void unpack_nib(uint32_t x, uint32_t* a) {
  const uint32_t x2 = __funnelshift_r(x, x, 8);
  a[0] = x & 0x003C003Cu; a[1] = x & 0x03C003C0u; a[2] = x2 & 0x003C003Cu; a[3] = x2 & 0x03C003C0u;
}
__device__ __forceinline__ void unpack_rows23(uint32_t x, uint32_t* a) {  // tau 2,3
  const uint32_t x2 = __funnelshift_r(x, x, 8);
  a[0] = x & 0x00C000C0u; a[1] = x & 0x03000300u; a[2] = x2 & 0x00C000C0u; a[3] = x2 & 0x03000300u;
}

// Scores of one staged (page, kv-head) blob, in log2 units: s[2*mt + rh] is
// token 16*mt + 8*rh + r of head qq.
//   pa: shared-space address of the staged blob
//   qf[j][0..1]: this lane's B-fragment query pairs for k-step j: the high or
//                the low part (column parity) of the query of head lane/8
//   qxa: shared-space address of the same part of q/2^W of head lane/8, in
//        channel order (extra-plane gather)
template <int NX, int W, int V>
__device__ __forceinline__ void page_scores(const uint32_t pa, const uint32_t (&qf)[8][2],
                                            const uint32_t qxa, const Lane& L,
                                            const float (&kscale)[4], float beta,
                                            float (&s)[4]) {
  using O = Off<NX, W, V>;
  const int lane = L.lane, qq = L.qq;
  const uint32_t a_lane = pa + 4 * W * 4 * lane;  // this lane's 16*W bytes of the base plane
  const uint32_t a_qq = pa + 4 * qq;              // this lane's fp16 pair in each 16-wide group

  // ---------------- scores: base plane, q.M row, extra plane
  float cs[2][4] = {};
  uint32_t kw[4 * W];  // W = 2: one word per k-step; W = 4: two (16-token blocks 0, 1)
  {
    const uint4 kb0 = ld_s128<0>(a_lane);
    const uint4 kb1 = ld_s128<16>(a_lane);
    kw[0] = kb0.x; kw[1] = kb0.y; kw[2] = kb0.z; kw[3] = kb0.w;
    kw[4] = kb1.x; kw[5] = kb1.y; kw[6] = kb1.z; kw[7] = kb1.w;
    if (W == 4) {
      const uint4 kb2 = ld_s128<32>(a_lane);
      const uint4 kb3 = ld_s128<48>(a_lane);
      kw[8 % (4 * W)] = kb2.x; kw[9 % (4 * W)] = kb2.y; kw[10 % (4 * W)] = kb2.z; kw[11 % (4 * W)] = kb2.w;
      kw[12 % (4 * W)] = kb3.x; kw[13 % (4 * W)] = kb3.y; kw[14 % (4 * W)] = kb3.z; kw[15 % (4 * W)] = kb3.w;
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t S0, S1;
    switch (j) {  // compile-time offsets (the loop is unrolled)
#define KITTY_KS(J) case J: S0 = ld_s32<O::ks + 32 * J>(a_qq); S1 = ld_s32<O::ks + 32 * J + 16>(a_qq); break;
      KITTY_KS(0) KITTY_KS(1) KITTY_KS(2) KITTY_KS(3) KITTY_KS(4) KITTY_KS(5) KITTY_KS(6) default: KITTY_KS(7)
#undef KITTY_KS
    }
    // this lane's part of q (high or low) times the step: exact in fp16
    const uint32_t b0 = hmul2u(qf[j][0], S0);
    const uint32_t b1 = hmul2u(qf[j][1], S1);
    uint32_t a[4];
    if (W == 2) {
      unpack_rows01(kw[j], a);
      mma_f16(cs[0], a, b0, b1);
      unpack_rows23(kw[j], a);
      mma_f16(cs[1], a, b0, b1);
    } else {
      unpack_nib(kw[(2 * j) % (4 * W)], a);
      mma_f16(cs[0], a, b0, b1);
      unpack_nib(kw[(2 * j + 1) % (4 * W)], a);
      mma_f16(cs[1], a, b0, b1);
    }
  }
  if (NX > 0) {
    const uint32_t a_id = pa + 4 * qq;
    const uint32_t a_x = pa + 2 * W * NX * lane;
#pragma unroll
    for (int js = 0; js < NX; ++js) {
      uint32_t ids;
      uint2 x = make_uint2(0u, 0u);  // W = 2: x.x; W = 4: x.x, x.y for 16-token blocks 0, 1
      switch (js) {  // channel-list rows 2qq, 2qq+1, 2qq+8, 2qq+9 are one word (fragment order)
#define KITTY_KX(J) case J: ids = ld_s32<O::kch + 16 * J>(a_id); \
                            if (W == 2) x.x = ld_s32<O::kx + 4 * J>(a_x); \
                            else x = ld_s64<O::kx + 8 * J>(a_x); break;
        KITTY_KX(0) KITTY_KX(1) KITTY_KX(2) KITTY_KX(3) KITTY_KX(4) KITTY_KX(5) KITTY_KX(6) default: KITTY_KX(7)
#undef KITTY_KX
      }
      const uint32_t c0 = (ids << 1) & 0xFEu, c1 = (ids >> 7) & 0xFEu;
      const uint32_t c2 = (ids >> 15) & 0xFEu, c3 = (ids >> 23) & 0xFEu;
      const uint32_t q01 = ld_s16r(qxa + c0) | ((uint32_t)ld_s16r(qxa + c1) << 16);
      const uint32_t q23 = ld_s16r(qxa + c2) | ((uint32_t)ld_s16r(qxa + c3) << 16);
      const uint32_t s01 = ld_s16r(pa + O::ks + c0) | ((uint32_t)ld_s16r(pa + O::ks + c1) << 16);
      const uint32_t s23 = ld_s16r(pa + O::ks + c2) | ((uint32_t)ld_s16r(pa + O::ks + c3) << 16);
      const uint32_t b0 = hmul2u(q01, s01);
      const uint32_t b1 = hmul2u(q23, s23);
      uint32_t a[4];
      if (W == 2) {
        unpack_rows01(x.x, a);
        mma_f16(cs[0], a, b0, b1);
        unpack_rows23(x.x, a);
        mma_f16(cs[1], a, b0, b1);
      } else {
        unpack_nib(x.x, a);
        mma_f16(cs[0], a, b0, b1);
        unpack_nib(x.y, a);
        mma_f16(cs[1], a, b0, b1);
      }
    }
  }

#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh)
      s[2 * mt + rh] = fmaf(cs[mt][2 * rh] + cs[mt][2 * rh + 1], kscale[2 * mt + rh], beta);
}

// q.M bias (log2 units) of two pages with one set of one-row MMAs: B is the
// split query (the same for every page), whose two columns of a head add up to
// q.M; A rows r even carry page A's Key minima and odd rows page B's; each lane
// reads its own row and its neighbour's.
template <int NX, int W, int V>
__device__ __forceinline__ void pair_beta(const uint32_t paA, const uint32_t paB,
                                          const uint32_t (&qf)[8][2], const Lane& L,
                                          float sm_log2, float& bA, float& bB) {
  using O = Off<NX, W, V>;
  // this lane's 16 minima pairs are contiguous (fragment order): 4 x 16 bytes
  const uint32_t a_m = ((L.r & 1) ? paB : paA) + 64 * L.qq;
  const uint4 m0 = ld_s128<O::km>(a_m), m1 = ld_s128<O::km + 16>(a_m);
  const uint4 m2 = ld_s128<O::km + 32>(a_m), m3 = ld_s128<O::km + 48>(a_m);
  const uint32_t M[16] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w,
                          m2.x, m2.y, m2.z, m2.w, m3.x, m3.y, m3.z, m3.w};
  float cm[4] = {};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t am[4] = {M[2 * j], 0u, M[2 * j + 1], 0u};
    mma_f16(cm, am, qf[j][0], qf[j][1]);
  }
  const float mine = (cm[0] + cm[1]) * sm_log2;
  const float other = __shfl_xor_sync(0xFFFFFFFFu, mine, 4);
  bA = (L.r & 1) ? other : mine;
  bB = (L.r & 1) ? mine : other;
}

// Probabilities of one page against the running max, split into a high part
// rounded to 4 significant bits (exact times a 7-bit Value step) and the rest
// (signed, at most 2^-4 of p), as fp16, and transposed into PV B fragments
// (column 2h = high, 2h+1 = rest).  Rounding the high part rather than
// truncating it halves the rest, and with it the two fp16 roundings the rest
// takes (its own and its product with the step).  p <= 1, so the rounded
// high part stays finite.
__device__ __forceinline__ void page_probs(WarpState& w, const float (&s)[4], uint32_t (&T)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float p = ex2(s[i] - w.m);
    w.l += p;
    const float t = __uint_as_float((__float_as_uint(p) + 0x00080000u) & 0xFFF00000u);
    T[i] = movmatrix_t(h2_bits(__floats2half2_rn(t, p - t)));  // (high, rest) -> B columns
  }
}

// Value minima term and PV of one page with its probability fragments T.
template <int NX, int W, int V>
__device__ __forceinline__ void page_pv(WarpState& w, const uint32_t pa, const uint32_t (&T)[4],
                                        const Lane& L) {
  using O = Off<NX, W, V>;
  const int lane = L.lane, r = L.r, qq = L.qq;
  const uint32_t a_lane = pa + 32 * lane;
  const uint32_t a_q16 = pa + 16 * qq;  // this lane group's Value steps (fragment order)
  // ---------------- Value minima: rows = groups (r & 3), k = tokens (fragment order)
  {
    const uint4 vm = ld_s128<O::vm>(pa + 64 * (r & 3) + 16 * qq);
    const uint32_t am0[4] = {vm.x, 0u, vm.y, 0u};
    mma_f16(w.vm, am0, T[0], T[1]);
    const uint32_t am1[4] = {vm.z, 0u, vm.w, 0u};
    mma_f16(w.vm, am1, T[2], T[3]);
  }

  // ---------------- PV with the Value step folded into this lane's part of P
  // (high part: exact product; the rest: rounded once, relative 2^-11 of a
  // term of at most 2^-4 of p)
  // 2-bit Values: a lane's 8 bytes of group G are words (kt = 0, 1), each
  // holding both m-tiles; 4-bit Values: its 16 bytes are words (kt, m-tile
  // parity), each one A fragment
  const uint32_t a_lane4 = pa + 64 * lane;
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    uint4 vv;
    uint32_t S[4];
    switch (G) {
#define KITTY_VG(J) case J: { if (V == 4) { vv = ld_s128<O::vb + 16 * J>(a_lane4); } \
                            else { const uint2 v2 = ld_s64<O::vb + 8 * J>(a_lane); \
                                   vv = make_uint4(v2.x, v2.y, 0u, 0u); } \
                            const uint4 sv = ld_s128<O::vs + 64 * J>(a_q16); \
                            S[0] = sv.x; S[1] = sv.y; S[2] = sv.z; S[3] = sv.w; } break;
      KITTY_VG(0) KITTY_VG(1) KITTY_VG(2) default: KITTY_VG(3)
#undef KITTY_VG
    }
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      uint32_t bg[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = 2 * kt + k;
        bg[k] = hmul2u(T[i], S[i]);
      }
      uint32_t a[4];
      if (V == 4) {
        unpack_nib(kt ? vv.z : vv.x, a);
        mma_f16(w.acc[2 * G], a, bg[0], bg[1]);
        unpack_nib(kt ? vv.w : vv.y, a);
        mma_f16(w.acc[2 * G + 1], a, bg[0], bg[1]);
      } else {
        const uint32_t x = kt ? vv.y : vv.x;
        unpack_rows01(x, a);
        mma_f16(w.acc[2 * G], a, bg[0], bg[1]);
        unpack_rows23(x, a);
        mma_f16(w.acc[2 * G + 1], a, bg[0], bg[1]);
      }
    }
  }
}

// Unquantized tail tokens (0..31 per sequence).  Warp wid takes tokens wid,
// wid+4, ... (at most 8).  All of its K and V rows are loaded at once (8 bytes
// a lane per row; the rows were prefetched into L2 when the CTA started) and
// pass through the warp's idle stage buffer to the tensor cores, in the input
// type: the scores of its tokens against the 4 query heads (8 MMAs; lane
// (r, qq) gets token r of head qq, so one rescale covers them all), then the
// PV (one MMA per 16 channels), brought to the paged codes' per-row power of
// two.
template <int DT, int V>
__device__ void tail_tokens(WarpState& w, const DecodeParams& p, const __half* qs, int b, int kvh,
                            int tl, int wid, const Lane& L, uint8_t* vbuf) {
  const int lane = L.lane, r = L.r, qq = L.qq;
  const int nw = tl > wid ? (tl - wid + kDWarps - 1) / kDWarps : 0;  // warp-uniform
  if (nw == 0) return;
  const size_t base = ((size_t)b * p.Hkv + kvh) * kPage * kD + 4 * lane;
  uint2 kx[8], vx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const size_t off = base + (size_t)(wid + kDWarps * i) * kD;
    // L2-coherent loads: a fused append wrote the newest row in this launch
    kx[i] = i < nw ? __ldcg(reinterpret_cast<const uint2*>(p.tail_k + off)) : make_uint2(0u, 0u);
    vx[i] = i < nw ? __ldcg(reinterpret_cast<const uint2*>(p.tail_v + off)) : make_uint2(0u, 0u);
  }
  // K and V rows through the warp's idle stage buffer, rows padded to kTailRow
  // bytes (conflict-free ldmatrix); rows past nw are zero
  constexpr int kTailRow = 2 * kD + 16;
  uint8_t* kbuf = vbuf + 8 * kTailRow;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    *reinterpret_cast<uint2*>(vbuf + i * kTailRow + 8 * lane) = vx[i];
    *reinterpret_cast<uint2*>(kbuf + i * kTailRow + 8 * lane) = kx[i];
  }
  __syncwarp();
  // scores on the tensor cores in the input type (the products are exact):
  // A = the K rows (tokens x channels) by ldmatrix, B = q with head h in
  // column 2h (odd columns zero), so lane (r, qq) gets token r of head qq
  float cs[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t ka = smem_u32(kbuf) + (lane & 7) * kTailRow + (lane >> 3) * 16;
    const uint32_t qa = smem_u32(qs + (r >> 1) * kD + 2 * qq);
    const bool qcol = (r & 1) == 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t a4[4];
      ldsm_x4(ka + 64 * g, a4);  // channel blocks 4g .. 4g+3 of 8 channels
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int j = 2 * g + k;  // k-step: channels 16j .. 16j+15
        const uint32_t a[4] = {a4[2 * k], 0u, a4[2 * k + 1], 0u};
        uint32_t qb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t h2;
          switch (2 * j + e) {  // compile-time offsets (the loops are unrolled)
#define KITTY_QT(K) case K: h2 = ld_s32<2 * (16 * (K / 2) + 8 * (K % 2))>(qa); break;
            KITTY_QT(0) KITTY_QT(1) KITTY_QT(2) KITTY_QT(3) KITTY_QT(4) KITTY_QT(5) KITTY_QT(6) KITTY_QT(7)
            KITTY_QT(8) KITTY_QT(9) KITTY_QT(10) KITTY_QT(11) KITTY_QT(12) KITTY_QT(13) KITTY_QT(14)
            default: KITTY_QT(15)
#undef KITTY_QT
          }
          qb[e] = qcol ? half2_to16<DT>(h2) : 0u;
        }
        mma16<DT>(cs, a, qb[0], qb[1]);
      }
    }
  }
  const float sc = r < nw ? cs[0] * p.sm_log2 : -INFINITY;
  float pm = fmaxf(sc, __shfl_xor_sync(0xFFFFFFFFu, sc, 4));
  pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
  pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
  rescale(w, pm);
  const float pr = r < nw ? ex2(sc - w.m) : 0.f;
  w.l += pr;
  // PV on the tensor cores in the input type: A = V^T (channels x this warp's
  // tokens) by transposing ldmatrix, B = p as (high, rest) pairs in the input
  // type: column n = r takes part r & 1 of head r / 2, k = tokens 2qq, 2qq+1
  // (tokens 8..15 of the k-step are absent: B's second register is zero)
  const uint32_t u0 = prob_pair<DT>(__shfl_sync(0xFFFFFFFFu, pr, 8 * qq + (r >> 1)));
  const uint32_t u1 = prob_pair<DT>(__shfl_sync(0xFFFFFFFFu, pr, 8 * qq + 4 + (r >> 1)));
  const uint32_t b0 = __byte_perm(u0, u1, (r & 1) ? 0x7632u : 0x5410u);
  const uint32_t va = smem_u32(vbuf) + (lane & 7) * kTailRow + (lane >> 3) * 16;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t a4[4];
    ldsm_x4_t(va + 64 * g, a4);  // channel blocks 4g .. 4g+3 of 8 channels
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int mc = 2 * g + k;
      const uint32_t a[4] = {a4[2 * k], a4[2 * k + 1], 0u, 0u};
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma16<DT>(c, a, b0, 0u);
#pragma unroll
      for (int i = 0; i < 4; ++i)  // to the codes' scale: the row's power of two
        w.acc[mc][i] += c[i] * __uint_as_float((uint32_t)(127 - kCodeExp + vrow_exp(V, mc, i >> 1)) << 23);
    }
  }
}

// Quantize the full tail of (sequence, kv head) sh into page fid with the
// page quantizer (running statistics updated in running mode), staging through
// sm.  Not inlined: it runs on a flush only (one call in 32 per sequence) and
// keeps its registers out of the attention loop.  Called by all 128 threads.
template <int DT, int W, int V>
__device__ __noinline__ void flush_tail(QuantSmem* sm, const AppendParams ap, size_t sh, int fid,
                                        int kvh, int Hkv, int n_hi, int32_t* d_status) {
  const int c = threadIdx.x;
  float rs = 0.f, rq = 0.f;
  int rc = 0;
  if (ap.running) {
    rs = ap.run_sum[sh * kD + c];
    rq = ap.run_sumsq[sh * kD + c];
    rc = ap.run_count[sh];
  }
  const BlobLayout lay(n_hi, W, V);
  quantize_tile<DT, W, V>(*sm, ap.tail_k + sh * kPage * kD, ap.tail_v + sh * kPage * kD, kD, n_hi,
                    ap.running != 0, rs, rq, rc, ap.pool + ((size_t)fid * Hkv + kvh) * lay.bytes,
                    d_status);
  if (ap.running) {
    ap.run_sum[sh * kD + c] = rs;
    ap.run_sumsq[sh * kD + c] = rq;
    if (c == 0) ap.run_count[sh] = rc;
  }
}

// Merge of the 4 warps' states in fragment layout, in two halves around one
// block barrier.  merge_put: a warp leaves its O and Value-minima fragments and
// (m, l) in its own stage buffers (idle after the page loop; 4608 bytes from
// `scratch`).  merge_get: warp w then merges m-tiles 2w, 2w+1 (channels
// 32w..32w+31, Value group w) of every warp, in warp order, at the common
// maximum, and writes those channels of its heads to the output (one split) or
// to the split's partials.
constexpr int kMergeBytes = 32 * 16 * 9;  // per warp: 8 O float4 + (vm0, vm1, m, l) per lane

__device__ __forceinline__ void merge_put(WarpState& w, uint8_t* scratch, const Lane& L) {
  __syncwarp();  // the warp's reads of its buffers (tail rows) are done
  w.l += __shfl_xor_sync(0xFFFFFFFFu, w.l, 4);
  w.l += __shfl_xor_sync(0xFFFFFFFFu, w.l, 8);
  w.l += __shfl_xor_sync(0xFFFFFFFFu, w.l, 16);
  float4* f = reinterpret_cast<float4*>(scratch);
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
    f[mc * 32 + L.lane] = make_float4(w.acc[mc][0], w.acc[mc][1], w.acc[mc][2], w.acc[mc][3]);
  f[8 * 32 + L.lane] = make_float4(w.vm[0], w.vm[1], w.m, w.l);
}

// stages: the CTA's stage buffers (warp ww's at + ww * warp_bytes); off: the
// offset of this head set's scratch within each warp's buffers.
template <int V>
__device__ __forceinline__ void merge_get(const uint8_t* stages, const int warp_bytes, const int off,
                                          const DecodeParams& p, const int b, const int s,
                                          const int h0, const int gh, const Lane& L) {
  const int wid = threadIdx.x >> 5;
  const int r = L.r, qq = L.qq;
  float4 ml[kDWarps];
#pragma unroll
  for (int ww = 0; ww < kDWarps; ++ww)
    ml[ww] = reinterpret_cast<const float4*>(stages + ww * warp_bytes + off)[8 * 32 + L.lane];
  float ms = -INFINITY;
#pragma unroll
  for (int ww = 0; ww < kDWarps; ++ww) ms = fmaxf(ms, ml[ww].z);
  float e[kDWarps], Lsum = 0.f, vmt = 0.f;
#pragma unroll
  for (int ww = 0; ww < kDWarps; ++ww) {
    e[ww] = (ms == -INFINITY || ml[ww].z == -INFINITY) ? 0.f : ex2(ml[ww].z - ms);
    Lsum += ml[ww].w * e[ww];
    vmt += (ml[ww].x + ml[ww].y) * e[ww];  // Value group r & 3 of head qq
  }
  const float vg = __shfl_sync(0xFFFFFFFFu, vmt, 4 * wid + qq);  // group wid of head qq
  const int hq = h0 + qq;
  float* part = p.ws + (((size_t)b * p.Hq + hq) * p.splits + s) * kPartial;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int mc = 2 * wid + k;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < kDWarps; ++ww) {
      const float4 x = reinterpret_cast<const float4*>(stages + ww * warp_bytes + off)[mc * 32 + L.lane];
      a[0] += x.x * e[ww];
      a[1] += x.y * e[ww];
      a[2] += x.z * e[ww];
      a[3] += x.w * e[ww];
    }
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const float sc = __uint_as_float((uint32_t)(127 + kCodeExp - vrow_exp(V, mc, rh)) << 23);
      const float o = (a[2 * rh] + a[2 * rh + 1]) * sc + vg;
      const int c = 16 * mc + 8 * rh + r;
      if (qq < gh) {
        if (p.splits == 1) store_out(p.out, p.out_dtype, ((size_t)b * p.Hq + hq) * kD + c,
                                     Lsum > 0.f ? o / Lsum : 0.f);
        else part[4 + c] = o;
      }
    }
  }
  if (wid == 0 && r == 0 && qq < gh) {
    if (p.splits == 1) {
      if (!(Lsum > 0.f)) set_status(p.d_status, KITTY_ST_EMPTY);
    } else {
      part[0] = ms;
      part[1] = Lsum;
    }
  }
}

template <int DT, int NX, int W, int V>
__global__ void __launch_bounds__(kDThreads, kDMinBlocks) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  trigger_dependents();  // the combine step may be scheduled once every CTA is running
  const int u = blockIdx.x, s = blockIdx.y;
  const int bk = u / p.HG, hgi = u - bk * p.HG;  // (sequence, kv head), head group
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int h0 = kvh * p.g + kHeadsPerCta * hgi;            // first query head of this CTA
  const int gh = min(kHeadsPerCta, p.g - kHeadsPerCta * hgi);  // its query heads
  const int tid = threadIdx.x, wid = tid >> 5;
  const Lane L;
  const int lane = L.lane, qq = L.qq;
  constexpr int kBlob = Off<NX, W, V>::bytes;
  constexpr int kDStages = stages_for(W);
  static_assert(kMergeBytes <= kDStages * kBlob, "merge scratch fits in a warp's stage buffers");
  const int sbeg = p.starts[s], send = p.starts[s + 1];
  // Independent loads first, all in flight together: the lengths, this warp's
  // first 32 block-table entries (up to the split's nominal end, which is
  // inside the row) and the query rows (thread tid = channel tid of 4 heads).
  int np = p.num_pages[b];
  int tl = p.tail_len != nullptr ? p.tail_len[b] : 0;
  const int first = sbeg + wid;  // this warp's pages: first + kDWarps*i, i < npw
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages;
  int bt_cache = first + kDWarps * lane < send ? bt[first + kDWarps * lane] : -1;
  float qv[4];
#pragma unroll
  for (int h = 0; h < 4; ++h)
    qv[h] = h < gh ? load16<DT>(p.q + ((size_t)b * p.Hq + h0 + h) * kD + tid) : 0.f;
  // the tensor cores take the query as fp16: a value it cannot hold is reported
  // (it would turn the scores of the query group into inf or NaN)
  if (s == 0) {
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (!(fabsf(qv[h]) <= 65504.0f))
        set_status(p.d_status, fabsf(qv[h]) < INFINITY ? KITTY_ST_RANGE : KITTY_ST_NONFINITE);
  }
  const bool lens_ok =
      !(np < 0 || np > p.max_pages || tl < 0 || tl > kPage || (tl > 0 && p.tail_k == nullptr));
  if (!lens_ok) {  // nothing is appended either
    if (tid == 0 && s == 0 && kvh == 0 && hgi == 0) set_status(p.d_status, KITTY_ST_BAD_LEN);
    np = 0;
    tl = 0;
  }
  if (!split_active(p, s, np)) {
    // no pages here: mark the partials empty (the combine then needs no lengths)
    if (tid < gh) p.ws[(((size_t)b * p.Hq + h0 + tid) * p.splits + s) * kPartial] = -INFINITY;
    return;
  }
  const int pbeg = sbeg, pend = min(np, send);
  // ---- fused append (split 0 owns the (sequence, kv head) tail)
  int flush_id = -1;  // >= 0: quantize the full tail into this page after the page loop
  if (p.ap.k_new != nullptr && s == 0 && lens_ok && tl == kPage) {
    if (tid == 0) set_status(p.d_status, KITTY_ST_TAIL_FULL);
  } else if (p.ap.k_new != nullptr && s == 0 && lens_ok) {
    const size_t sh = (size_t)b * p.Hkv + kvh;
    p.ap.tail_k[(sh * kPage + tl) * kD + tid] = p.ap.k_new[sh * kD + tid];
    p.ap.tail_v[(sh * kPage + tl) * kD + tid] = p.ap.v_new[sh * kD + tid];
    const int n = tl + 1;
    const int fid = p.ap.flush_page_ids[b];
    if (fid >= 0 && n < kPage) {
      if (tid == 0) set_status(p.d_status, KITTY_ST_BAD_FLUSH);
    } else if (fid >= 0 && np >= p.max_pages) {
      if (tid == 0) set_status(p.d_status, KITTY_ST_TABLE_FULL);
    } else if (fid >= p.pool_pages) {
      if (tid == 0) set_status(p.d_status, KITTY_ST_BAD_PAGE);
    } else if (fid >= 0) {
      flush_id = fid;
    }
    tl = flush_id >= 0 ? 0 : n;  // tokens the tail holds for this call's attention
  }

  uint8_t* stages = dsm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + kDWarps * kDStages * kBlob);
  __half* qs = reinterpret_cast<__half*>(bars + kDWarps * kDStages);  // q      [4][128]
  __half* qs4 = qs + 4 * kD;  // q / 2^W split: high parts [4][kQx], then low parts [4][kQx]

  // ---- start this warp's page copies (its barriers are its own)
  const int npw = pend > first ? (pend - first + kDWarps - 1) / kDWarps : 0;
  uint8_t* wst = stages + (size_t)wid * kDStages * kBlob;
  uint64_t* wbar = bars + wid * kDStages;
  if (lane == 0) {
    for (int st = 0; st < kDStages; ++st) mbar_init(&wbar[st], 1);
    fence_mbar_init();
  }
  const uint8_t* head_base = p.pool + (size_t)kvh * kBlob;
  const size_t page_stride = (size_t)p.Hkv * kBlob;
  int bt_base = 0;
  uint32_t valid_mask = 0;  // bit st: stage st holds a valid page
  const uint32_t stage0 = smem_u32(wst), bar0 = smem_u32(wbar);  // 32-bit shared addresses
  auto issue = [&](int i) {
    if (i - bt_base >= 32) {
      bt_base = i;
      bt_cache = (i + lane < npw) ? bt[first + (i + lane) * kDWarps] : -1;
    }
    const int pid = __shfl_sync(0xFFFFFFFFu, bt_cache, i - bt_base);
    const int st = i % kDStages;
    const bool ok = pid >= 0 && pid < p.pool_pages;
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * st;
      if (ok) {
        mbar_arrive_expect_tx_s(bar, (uint32_t)kBlob);
        bulk_g2s_s(stage0 + st * kBlob, head_base + (size_t)pid * page_stride, (uint32_t)kBlob, bar);
      } else {
        set_status(p.d_status, KITTY_ST_BAD_PAGE);
        mbar_arrive_s(bar);
      }
    }
    valid_mask = ok ? (valid_mask | (1u << st)) : (valid_mask & ~(1u << st));
  };
  // refill of a pair: pages i and i + 1 (if any) under one elected-lane branch
  auto issue2 = [&](int i) {
    const bool has1 = i + 1 < npw;
    if (i + 1 - bt_base >= 32) {
      bt_base = i;
      bt_cache = (i + lane < npw) ? bt[first + (i + lane) * kDWarps] : -1;
    }
    const int pid0 = __shfl_sync(0xFFFFFFFFu, bt_cache, i - bt_base);
    const int pid1 = __shfl_sync(0xFFFFFFFFu, bt_cache, i + 1 - bt_base);
    const int st0 = i % kDStages, st1 = (i + 1) % kDStages;
    const bool ok0 = pid0 >= 0 && pid0 < p.pool_pages;
    const bool ok1 = has1 && pid1 >= 0 && pid1 < p.pool_pages;
    if (lane == 0) {
      const uint32_t b0 = bar0 + 8 * st0, b1 = bar0 + 8 * st1;
      if (ok0) {
        mbar_arrive_expect_tx_s(b0, (uint32_t)kBlob);
        bulk_g2s_s(stage0 + st0 * kBlob, head_base + (size_t)pid0 * page_stride, (uint32_t)kBlob, b0);
      } else {
        set_status(p.d_status, KITTY_ST_BAD_PAGE);
        mbar_arrive_s(b0);
      }
      if (ok1) {
        mbar_arrive_expect_tx_s(b1, (uint32_t)kBlob);
        bulk_g2s_s(stage0 + st1 * kBlob, head_base + (size_t)pid1 * page_stride, (uint32_t)kBlob, b1);
      } else if (has1) {
        set_status(p.d_status, KITTY_ST_BAD_PAGE);
        mbar_arrive_s(b1);
      }
    }
    valid_mask = ok0 ? (valid_mask | (1u << st0)) : (valid_mask & ~(1u << st0));
    if (has1) valid_mask = ok1 ? (valid_mask | (1u << st1)) : (valid_mask & ~(1u << st1));
  };
  const int pro = min(npw, kDStages);
  for (int i = 0; i < pro; ++i) issue(i);
  // the tail rows are read after the pages: start pulling them into L2 now
  if (pbeg == 0 && tl > 0 && tid == 0) {
    const size_t off = ((size_t)b * p.Hkv + kvh) * kPage * kD;
    l2_prefetch(p.tail_k + off, (uint32_t)tl * kD * 2);
    l2_prefetch(p.tail_v + off, (uint32_t)tl * kD * 2);
  }

#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const __half hv = __float2half_rn(qv[h]);
    qs[h * kD + tid] = hv;
    const __half hx = __hmul(hv, __float2half_rn(1.0f / (1 << W)));  // exact: power of two
    const __half hh = high_part(hx);
    qs4[h * kQx + tid] = hh;
    qs4[(4 + h) * kQx + tid] = __hsub(hx, hh);  // exact
  }
  __syncthreads();

  // B-fragment query pairs: column 2h takes the high part of q, 2h+1 the rest
  const bool low_col = (lane >> 2) & 1;
  uint32_t qf[8][2];
  {
    const uint32_t qa = smem_u32(qs + (lane >> 3) * kD + 2 * qq);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        uint32_t q2;
        switch (2 * j + e) {  // compile-time offsets (the loops are unrolled)
#define KITTY_QF(K) case K: q2 = ld_s32<2 * (16 * (K / 2) + 8 * (K % 2))>(qa); break;
          KITTY_QF(0) KITTY_QF(1) KITTY_QF(2) KITTY_QF(3) KITTY_QF(4) KITTY_QF(5) KITTY_QF(6) KITTY_QF(7)
          KITTY_QF(8) KITTY_QF(9) KITTY_QF(10) KITTY_QF(11) KITTY_QF(12) KITTY_QF(13) KITTY_QF(14)
          default: KITTY_QF(15)
#undef KITTY_QF
        }
        const uint32_t h2 = q2 & 0xFF80FF80u;  // high parts of both halves
        qf[j][e] = low_col ? hsub2u(q2, h2) : h2;
      }
    }
  }
  const uint32_t qxa = smem_u32(qs4 + ((low_col ? 4 : 0) + (lane >> 3)) * kQx);
  float kscale[4];
#pragma unroll
  for (int tau = 0; tau < 4; ++tau)
    // a code sits at 2^(2 tau - 24) (2-bit planes) or 2^(4 (tau & 1) - 24) (4-bit)
    kscale[tau] = p.sm_log2 *
                  __uint_as_float((uint32_t)(127 + kCodeExp - (W == 2 ? 2 * tau : 4 * (tau & 1))) << 23);

  WarpState w;
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int i = 0; i < 4; ++i) w.acc[mc][i] = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) w.vm[i] = 0.f;
  w.m = kNegBig;
  w.l = 0.f;
  bool timed_out = false;
  // Pages are taken two at a time: two independent score chains, one joint max
  // and rescale, then both PVs.  A missing or invalid page is masked (score -inf).
  for (int i = 0; i < npw; i += 2) {
    const bool hasB = i + 1 < npw;
    // every lane observes the phase completion itself (acquire of the copied
    // bytes); the exit is warp-uniform and the wait is bounded
    bool done = false;
    for (uint32_t it = 0;; ++it) {
      done = done || (mbar_test_s(bar0 + 8 * (i % kDStages), (uint32_t)(i / kDStages) & 1u) &&
                      (!hasB || mbar_test_s(bar0 + 8 * ((i + 1) % kDStages),
                                            (uint32_t)((i + 1) / kDStages) & 1u)));
      if (__all_sync(0xFFFFFFFFu, done) || it >= p.wait_polls) break;
      if (it > 64) __nanosleep(32);
    }
    if (!__all_sync(0xFFFFFFFFu, done)) {
      timed_out = true;
      // give up: report, then wait (bounded) for every copy still in flight
      if (lane == 0) {
        set_status(p.d_status, KITTY_ST_TIMEOUT);
        for (int k = i; k < min(npw, i + kDStages); ++k)
          mbar_wait_bounded(&wbar[k % kDStages], (uint32_t)(k / kDStages) & 1u, kWaitLimit);
      }
      __syncwarp();
      break;
    }
    const int stA = i % kDStages, stB = (i + 1) % kDStages;
    const bool vA = (valid_mask >> stA) & 1u;
    const uint32_t paA = stage0 + stA * kBlob;
    const uint32_t paB = hasB ? stage0 + stB * kBlob : paA;
    float bA, bB;
    pair_beta<NX, W, V>(paA, paB, qf, L, p.sm_log2, bA, bB);
    float sA[4];
    page_scores<NX, W, V>(paA, qf, qxa, L, kscale, bA, sA);
    if (hasB) {
      const bool vB = (valid_mask >> stB) & 1u;
      float sB[4];
      page_scores<NX, W, V>(paB, qf, qxa, L, kscale, bB, sB);
      if (!(vA && vB)) {  // a page id was out of range (warp-uniform, rare)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          sA[k] = vA ? sA[k] : -INFINITY;
          sB[k] = vB ? sB[k] : -INFINITY;
        }
      }
      float pm = fmaxf(fmaxf(fmaxf(sA[0], sA[1]), fmaxf(sA[2], sA[3])),
                       fmaxf(fmaxf(sB[0], sB[1]), fmaxf(sB[2], sB[3])));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
      rescale(w, pm);
      uint32_t TA[4], TB[4];
      page_probs(w, sA, TA);
      page_probs(w, sB, TB);
      page_pv<NX, W, V>(w, paA, TA, L);
      page_pv<NX, W, V>(w, paB, TB, L);
    } else {  // last page of an odd count
#pragma unroll
      for (int k = 0; k < 4; ++k) sA[k] = vA ? sA[k] : -INFINITY;
      float pm = fmaxf(fmaxf(sA[0], sA[1]), fmaxf(sA[2], sA[3]));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
      rescale(w, pm);
      uint32_t TA[4];
      page_probs(w, sA, TA);
      page_pv<NX, W, V>(w, paA, TA, L);
    }
    __syncwarp();
    if (i + kDStages < npw) issue2(i + kDStages);
  }
  if (flush_id >= 0) {
    // the full tail becomes page flush_id (quantized in the idle stage buffers),
    // and this CTA attends to it from shared memory: the page the finalize step
    // appends at index np
    __syncthreads();
    QuantSmem* qsm = reinterpret_cast<QuantSmem*>(dsm);
    flush_tail<DT, W, V>(qsm, p.ap, (size_t)b * p.Hkv + kvh, flush_id, kvh, p.Hkv, p.n_hi, p.d_status);
    if (wid == 0) {
      const uint32_t pa = smem_u32(qsm->blob);
      float bA, bB;
      pair_beta<NX, W, V>(pa, pa, qf, L, p.sm_log2, bA, bB);
      float sA[4];
      page_scores<NX, W, V>(pa, qf, qxa, L, kscale, bA, sA);
      float pm = fmaxf(fmaxf(sA[0], sA[1]), fmaxf(sA[2], sA[3]));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
      rescale(w, pm);
      uint32_t TA[4];
      page_probs(w, sA, TA);
      page_pv<NX, W, V>(w, pa, TA, L);
    }
  }
  // the tail tokens go with the sequence's first split (dispatched earliest);
  // they reuse the stage buffers, which are idle unless a copy timed out
  if (pbeg == 0 && tl > 0 && !timed_out) tail_tokens<DT, V>(w, p, qs, b, kvh, tl, wid, L, wst);

  // a flushed page was read from the first warps' buffers, where the merge now writes
  if (flush_id >= 0) __syncthreads();
  merge_put(w, wst, L);
  __syncthreads();
  merge_get<V>(stages, kDStages * kBlob, 0, p, b, s, h0, gh, L);
}

// Merge the split partials of a (sequence, query head) row: the maximum of the
// partials' m, then L = sum l * 2^(m - max) and O = sum o * 2^(m - max) in split
// order; splits without pages left m = -inf.  In a fused append, the row of query
// head 0 then does the sequence's append bookkeeping (every decode CTA has read
// the old lengths by now).  Both merge kernels are launched as programmatic
// dependents of the decode kernel: they may be scheduled while the decode grid
// drains, and wait for the whole grid (and its memory) before reading.
__device__ __forceinline__ void merge_split(float m, float l, float4 o, float ms, float& L,
                                            float4& O) {
  if (m == -INFINITY) return;  // no pages: l, o were never written
  const float e = ex2(m - ms);
  L += l * e;
  O.x += o.x * e;
  O.y += o.y * e;
  O.z += o.z * e;
  O.w += o.w * e;
}

__device__ __forceinline__ void finish_row(const DecodeParams& p, int bh, int lane, float L,
                                           float4 O) {
  const bool ok = L > 0.f;
  const float4 r = ok ? make_float4(O.x / L, O.y / L, O.z / L, O.w / L)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  store_out4(p.out, p.out_dtype, (size_t)bh * kD + 4 * lane, r);
  const int b = bh / p.Hq;
  if (lane == 0 && !ok) set_status(p.d_status, KITTY_ST_EMPTY);
  if (p.ap.k_new != nullptr && lane == 0 && bh - b * p.Hq == 0)
    append_finalize_one(b, p.ap.tail_len, p.ap.flush_page_ids, p.ap.block_table, p.max_pages,
                        p.ap.num_pages, p.pool_pages);
}

constexpr int kCombineSplits = 8;  // splits one 32-thread row merges in one round of loads

// Up to kCombineSplits splits: 32 threads per row, four channels a thread
// (16-byte loads), four rows per 128-thread CTA; every split's (m, l, o) in one
// round of independent loads.
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p, int rows) {
  grid_dependency_wait();
  const int bh = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (bh >= rows) return;
  const float* base = p.ws + (size_t)bh * p.splits * kPartial;
  const float4* obase = reinterpret_cast<const float4*>(base + 4) + lane;  // kPartial / 4 apart
  constexpr int kQ = kPartial / 4, kU = kCombineSplits;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float m[kU], l[kU];
  float4 o[kU];
#pragma unroll
  for (int s = 0; s < kU; ++s) {
    m[s] = s < p.splits ? base[s * kPartial] : -INFINITY;
    l[s] = s < p.splits ? base[s * kPartial + 1] : 0.f;
    o[s] = s < p.splits ? obase[s * kQ] : zero;
  }
  float ms = -INFINITY, L = 0.f;
  float4 O = zero;
#pragma unroll
  for (int s = 0; s < kU; ++s) ms = fmaxf(ms, m[s]);
  if (ms != -INFINITY) {
#pragma unroll
    for (int s = 0; s < kU; ++s) merge_split(m[s], l[s], o[s], ms, L, O);
  }
  finish_row(p, bh, lane, L, O);
}

// More splits (the long-context layers): one 128-thread CTA per row.  Warp w
// merges splits w, w + 4, w + 8, ... (up to kCombineSplits of them per round of
// independent loads, with a running maximum across rounds), then warp 0 merges
// the four warps' results through shared memory.  Two dependent rounds of
// loads instead of one per 16 splits (maxima) plus one per 8 (sums).
__global__ void __launch_bounds__(128) combine_wide_kernel(const DecodeParams p, int rows) {
  grid_dependency_wait();
  __shared__ float4 wo[4][32];
  __shared__ float wm[4], wl[4];
  const int bh = blockIdx.x, wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (bh >= rows) return;
  const float* base = p.ws + (size_t)bh * p.splits * kPartial;
  const float4* obase = reinterpret_cast<const float4*>(base + 4) + lane;
  constexpr int kQ = kPartial / 4, kU = kCombineSplits;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float ms = -INFINITY, L = 0.f;
  float4 O = zero;
  for (int s0 = wid; s0 < p.splits; s0 += 4 * kU) {
    float m[kU], l[kU];
    float4 o[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int s = s0 + 4 * k;
      const bool in = s < p.splits;
      m[k] = in ? base[(size_t)s * kPartial] : -INFINITY;
      l[k] = in ? base[(size_t)s * kPartial + 1] : 0.f;
      o[k] = in ? obase[(size_t)s * kQ] : zero;
    }
    float mr = ms;
#pragma unroll
    for (int k = 0; k < kU; ++k) mr = fmaxf(mr, m[k]);
    if (mr == -INFINITY) continue;
    if (ms != -INFINITY && mr > ms) {  // rescale the running sums to the new maximum
      const float e = ex2(ms - mr);
      L *= e;
      O.x *= e;
      O.y *= e;
      O.z *= e;
      O.w *= e;
    }
    ms = mr;
#pragma unroll
    for (int k = 0; k < kU; ++k) merge_split(m[k], l[k], o[k], ms, L, O);
  }
  if (lane == 0) {
    wm[wid] = ms;
    wl[wid] = L;
  }
  wo[wid][lane] = O;
  __syncthreads();
  if (wid != 0) return;
  const float M = fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]));
  float Lt = 0.f;
  float4 Ot = zero;
  if (M != -INFINITY) {
#pragma unroll
    for (int w = 0; w < 4; ++w) merge_split(wm[w], wl[w], wo[w][lane], M, Lt, Ot);
  }
  finish_row(p, bh, lane, Lt, Ot);
}

// Fused append bookkeeping when there is no combine step (one split).
__global__ void finalize_kernel(const DecodeParams p, int B) {
  grid_dependency_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B)
    append_finalize_one(b, p.ap.tail_len, p.ap.flush_page_ids, p.ap.block_table, p.max_pages,
                        p.ap.num_pages, p.pool_pages);
}

// ---------------------------------------------------------------- 8 heads per warp
// Query groups above 4 in the (4, 2) format: a warp carries two sets of 4 query
// heads (n-tiles), each its own 8-column B operands and online-softmax state,
// against every unpacked A fragment, so each code is unpacked once for 8 heads
// rather than once per head-group CTA.  The query's B fragments sit in a shared
// table [n-tile][k-step][lane][2 words] (8 bytes a lane: conflict-free loads)
// instead of registers; the second state costs registers, so 3 CTAs fit per SM.
constexpr int kDMinBlocks8 = 3;
constexpr int kQft = 2 * 8 * 32 * 2;  // query B-fragment table, 32-bit words

template <class F, int... I>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, I...>) {
  (f(std::integral_constant<int, I>{}), ...);
}
// f(std::integral_constant<int, i>) for i = 0 .. N-1, each i a compile-time constant
template <int N, class F>
__device__ __forceinline__ void static_for(F&& f) {
  static_for_impl(f, std::make_integer_sequence<int, N>{});
}

// q.M bias of both head sets for a page pair (see pair_beta).
template <int NX>
__device__ __forceinline__ void pair_beta8(const uint32_t paA, const uint32_t paB,
                                           const uint32_t qft_lane, const Lane& L, float sm_log2,
                                           float (&bA)[2], float (&bB)[2]) {
  using O = Off<NX, 2, 2>;
  const uint32_t a_m = ((L.r & 1) ? paB : paA) + 64 * L.qq;
  const uint4 m0 = ld_s128<O::km>(a_m), m1 = ld_s128<O::km + 16>(a_m);
  const uint4 m2 = ld_s128<O::km + 32>(a_m), m3 = ld_s128<O::km + 48>(a_m);
  const uint32_t M[16] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w,
                          m2.x, m2.y, m2.z, m2.w, m3.x, m3.y, m3.z, m3.w};
  static_for<2>([&](auto NT) {
    constexpr int nt = decltype(NT)::value;
    float cm[4] = {};
    static_for<8>([&](auto J) {
      constexpr int j = decltype(J)::value;
      const uint2 qb = ld_s64<(nt * 8 + j) * 256>(qft_lane);
      const uint32_t am[4] = {M[2 * j], 0u, M[2 * j + 1], 0u};
      mma_f16(cm, am, qb.x, qb.y);
    });
    const float mine = (cm[0] + cm[1]) * sm_log2;
    const float other = __shfl_xor_sync(0xFFFFFFFFu, mine, 4);
    bA[nt] = (L.r & 1) ? other : mine;
    bB[nt] = (L.r & 1) ? mine : other;
  });
}

// Scores of one staged blob for both head sets (see page_scores; 2-bit Key
// planes): each unpacked A fragment feeds one MMA per head set.
template <int NX>
__device__ __forceinline__ void page_scores8(const uint32_t pa, const uint32_t qft_lane,
                                             const uint32_t (&qxa)[2], const Lane& L,
                                             const float (&kscale)[4], const float (&beta)[2],
                                             float (&s)[2][4]) {
  using O = Off<NX, 2, 2>;
  const int lane = L.lane, qq = L.qq;
  const uint32_t a_lane = pa + 32 * lane;  // this lane's 32 bytes of the base plane
  const uint32_t a_qq = pa + 4 * qq;
  float cs[2][2][4] = {};
  const uint4 kb0 = ld_s128<0>(a_lane);
  const uint4 kb1 = ld_s128<16>(a_lane);
  const uint32_t kw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
  static_for<8>([&](auto J) {
    constexpr int j = decltype(J)::value;
    const uint32_t S0 = ld_s32<O::ks + 32 * j>(a_qq), S1 = ld_s32<O::ks + 32 * j + 16>(a_qq);
    uint32_t a01[4], a23[4];
    unpack_rows01(kw[j], a01);
    unpack_rows23(kw[j], a23);
    static_for<2>([&](auto NT) {
      constexpr int nt = decltype(NT)::value;
      const uint2 qb = ld_s64<(nt * 8 + j) * 256>(qft_lane);
      const uint32_t b0 = hmul2u(qb.x, S0), b1 = hmul2u(qb.y, S1);
      mma_f16(cs[nt][0], a01, b0, b1);
      mma_f16(cs[nt][1], a23, b0, b1);
    });
  });
  if (NX > 0) {
    const uint32_t a_id = pa + 4 * qq;
    const uint32_t a_x = pa + 4 * NX * lane;
    static_for<NX>([&](auto JS) {
      constexpr int js = decltype(JS)::value;
      const uint32_t ids = ld_s32<O::kch + 16 * js>(a_id);
      const uint32_t x = ld_s32<O::kx + 4 * js>(a_x);
      const uint32_t c0 = (ids << 1) & 0xFEu, c1 = (ids >> 7) & 0xFEu;
      const uint32_t c2 = (ids >> 15) & 0xFEu, c3 = (ids >> 23) & 0xFEu;
      const uint32_t s01 = ld_s16r(pa + O::ks + c0) | ((uint32_t)ld_s16r(pa + O::ks + c1) << 16);
      const uint32_t s23 = ld_s16r(pa + O::ks + c2) | ((uint32_t)ld_s16r(pa + O::ks + c3) << 16);
      uint32_t a01[4], a23[4];
      unpack_rows01(x, a01);
      unpack_rows23(x, a23);
      static_for<2>([&](auto NT) {
        constexpr int nt = decltype(NT)::value;
        const uint32_t q01 = ld_s16r(qxa[nt] + c0) | ((uint32_t)ld_s16r(qxa[nt] + c1) << 16);
        const uint32_t q23 = ld_s16r(qxa[nt] + c2) | ((uint32_t)ld_s16r(qxa[nt] + c3) << 16);
        const uint32_t b0 = hmul2u(q01, s01), b1 = hmul2u(q23, s23);
        mma_f16(cs[nt][0], a01, b0, b1);
        mma_f16(cs[nt][1], a23, b0, b1);
      });
    });
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh)
        s[nt][2 * mt + rh] =
            fmaf(cs[nt][mt][2 * rh] + cs[nt][mt][2 * rh + 1], kscale[2 * mt + rh], beta[nt]);
}

// Value minima term and PV of one page for both head sets (2-bit Values): each
// unpacked A fragment feeds one MMA per head set.
template <int NX>
__device__ __forceinline__ void page_pv8(WarpState (&w)[2], const uint32_t pa,
                                         const uint32_t (&T)[2][4], const Lane& L) {
  using O = Off<NX, 2, 2>;
  const int lane = L.lane, r = L.r, qq = L.qq;
  const uint32_t a_lane = pa + 32 * lane;
  const uint32_t a_q16 = pa + 16 * qq;
  {
    const uint4 vm = ld_s128<O::vm>(pa + 64 * (r & 3) + 16 * qq);
    const uint32_t am0[4] = {vm.x, 0u, vm.y, 0u};
    const uint32_t am1[4] = {vm.z, 0u, vm.w, 0u};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      mma_f16(w[nt].vm, am0, T[nt][0], T[nt][1]);
      mma_f16(w[nt].vm, am1, T[nt][2], T[nt][3]);
    }
  }
  static_for<4>([&](auto GG) {
    constexpr int G = decltype(GG)::value;
    const uint2 vv = ld_s64<O::vb + 8 * G>(a_lane);
    const uint4 sv = ld_s128<O::vs + 64 * G>(a_q16);
    const uint32_t S[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      uint32_t a01[4], a23[4];
      unpack_rows01(kt ? vv.y : vv.x, a01);
      unpack_rows23(kt ? vv.y : vv.x, a23);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t bg0 = hmul2u(T[nt][2 * kt], S[2 * kt]);
        const uint32_t bg1 = hmul2u(T[nt][2 * kt + 1], S[2 * kt + 1]);
        mma_f16(w[nt].acc[2 * G], a01, bg0, bg1);
        mma_f16(w[nt].acc[2 * G + 1], a23, bg0, bg1);
      }
    }
  });
}

// Running max of one head set over a page pair (or one page): scores of head qq
// of this lane's set, reduced over the 8 lanes that hold the same head.
__device__ __forceinline__ float head_max(const float (&a)[4], const float (&b)[4], bool hasB) {
  float pm = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
  if (hasB) pm = fmaxf(pm, fmaxf(fmaxf(b[0], b[1]), fmaxf(b[2], b[3])));
  pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 4));
  pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
  pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
  return pm;
}

// Decode with 8 query heads per CTA (the (4, 2) format, 2-bit Values, plain
// decode: no fused append).  The same schedule, staging and merge as
// decode_kernel; per head set the same arithmetic.
template <int DT, int NX>
__global__ void __launch_bounds__(kDThreads, kDMinBlocks8) decode8_kernel(const DecodeParams p) {
  constexpr int W = 2, V = 2;
  extern __shared__ __align__(128) uint8_t dsm[];
  trigger_dependents();
  const int u = blockIdx.x, s = blockIdx.y;
  const int bk = u / p.HG, hgi = u - bk * p.HG;
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int h0 = kvh * p.g + 2 * kHeadsPerCta * hgi;
  const int gh = min(2 * kHeadsPerCta, p.g - 2 * kHeadsPerCta * hgi);
  const int tid = threadIdx.x, wid = tid >> 5;
  const Lane L;
  const int lane = L.lane, qq = L.qq;
  constexpr int kBlob = Off<NX, W, V>::bytes;
  constexpr int kDStages = stages_for(W);
  static_assert(2 * kMergeBytes <= kDStages * kBlob, "merge scratch fits in a warp's stage buffers");
  const int sbeg = p.starts[s], send = p.starts[s + 1];
  int np = p.num_pages[b];
  int tl = p.tail_len != nullptr ? p.tail_len[b] : 0;
  const int first = sbeg + wid;
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages;
  int bt_cache = first + kDWarps * lane < send ? bt[first + kDWarps * lane] : -1;
  float qv[8];
#pragma unroll
  for (int h = 0; h < 8; ++h)
    qv[h] = h < gh ? load16<DT>(p.q + ((size_t)b * p.Hq + h0 + h) * kD + tid) : 0.f;
  if (s == 0) {
#pragma unroll
    for (int h = 0; h < 8; ++h)
      if (!(fabsf(qv[h]) <= 65504.0f))
        set_status(p.d_status, fabsf(qv[h]) < INFINITY ? KITTY_ST_RANGE : KITTY_ST_NONFINITE);
  }
  const bool lens_ok =
      !(np < 0 || np > p.max_pages || tl < 0 || tl > kPage || (tl > 0 && p.tail_k == nullptr));
  if (!lens_ok) {
    if (tid == 0 && s == 0 && kvh == 0 && hgi == 0) set_status(p.d_status, KITTY_ST_BAD_LEN);
    np = 0;
    tl = 0;
  }
  if (!split_active(p, s, np)) {
    if (tid < gh) p.ws[(((size_t)b * p.Hq + h0 + tid) * p.splits + s) * kPartial] = -INFINITY;
    return;
  }
  const int pbeg = sbeg, pend = min(np, send);

  uint8_t* stages = dsm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + kDWarps * kDStages * kBlob);
  __half* qs = reinterpret_cast<__half*>(bars + kDWarps * kDStages);  // q [8][128]
  __half* qs4 = qs + 8 * kD;  // q / 2^W: high parts [8][kQx], then low parts [8][kQx]
  uint32_t* qft = reinterpret_cast<uint32_t*>(qs4 + 16 * kQx);  // [2][8][32][2]

  const int npw = pend > first ? (pend - first + kDWarps - 1) / kDWarps : 0;
  uint8_t* wst = stages + (size_t)wid * kDStages * kBlob;
  uint64_t* wbar = bars + wid * kDStages;
  if (lane == 0) {
    for (int st = 0; st < kDStages; ++st) mbar_init(&wbar[st], 1);
    fence_mbar_init();
  }
  const uint8_t* head_base = p.pool + (size_t)kvh * kBlob;
  const size_t page_stride = (size_t)p.Hkv * kBlob;
  int bt_base = 0;
  uint32_t valid_mask = 0;
  const uint32_t stage0 = smem_u32(wst), bar0 = smem_u32(wbar);
  auto issue = [&](int i) {
    if (i - bt_base >= 32) {
      bt_base = i;
      bt_cache = (i + lane < npw) ? bt[first + (i + lane) * kDWarps] : -1;
    }
    const int pid = __shfl_sync(0xFFFFFFFFu, bt_cache, i - bt_base);
    const int st = i % kDStages;
    const bool ok = pid >= 0 && pid < p.pool_pages;
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * st;
      if (ok) {
        mbar_arrive_expect_tx_s(bar, (uint32_t)kBlob);
        bulk_g2s_s(stage0 + st * kBlob, head_base + (size_t)pid * page_stride, (uint32_t)kBlob, bar);
      } else {
        set_status(p.d_status, KITTY_ST_BAD_PAGE);
        mbar_arrive_s(bar);
      }
    }
    valid_mask = ok ? (valid_mask | (1u << st)) : (valid_mask & ~(1u << st));
  };
  const int pro = min(npw, kDStages);
  for (int i = 0; i < pro; ++i) issue(i);
  if (pbeg == 0 && tl > 0 && tid == 0) {
    const size_t off = ((size_t)b * p.Hkv + kvh) * kPage * kD;
    l2_prefetch(p.tail_k + off, (uint32_t)tl * kD * 2);
    l2_prefetch(p.tail_v + off, (uint32_t)tl * kD * 2);
  }

#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const __half hv = __float2half_rn(qv[h]);
    qs[h * kD + tid] = hv;
    const __half hx = __hmul(hv, __float2half_rn(1.0f / (1 << W)));  // exact: power of two
    const __half hh = high_part(hx);
    qs4[h * kQx + tid] = hh;
    qs4[(8 + h) * kQx + tid] = __hsub(hx, hh);  // exact
  }
  __syncthreads();
  const bool low_col = (lane >> 2) & 1;
  {  // the B-fragment table (warp wid: k-steps 2 wid, 2 wid + 1 of both head
     // sets): column 2h takes the high part of q, 2h+1 the rest
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const __half* qh = qs + (4 * nt + (lane >> 3)) * kD;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * wid + jj;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const __half2 q2 = *reinterpret_cast<const __half2*>(qh + 16 * j + 2 * qq + 8 * e);
          const __half2 h2 = __halves2half2(high_part(__low2half(q2)), high_part(__high2half(q2)));
          qft[((nt * 8 + j) * 32 + lane) * 2 + e] = h2_bits(low_col ? __hsub2(q2, h2) : h2);
        }
      }
    }
  }
  __syncthreads();
  const uint32_t qft_lane = smem_u32(qft) + 8 * lane;
  const uint32_t qxa[2] = {smem_u32(qs4 + ((low_col ? 8 : 0) + (lane >> 3)) * kQx),
                           smem_u32(qs4 + ((low_col ? 8 : 0) + 4 + (lane >> 3)) * kQx)};
  float kscale[4];
#pragma unroll
  for (int tau = 0; tau < 4; ++tau)
    kscale[tau] = p.sm_log2 * __uint_as_float((uint32_t)(127 + kCodeExp - 2 * tau) << 23);

  WarpState w[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int mc = 0; mc < 8; ++mc)
#pragma unroll
      for (int i = 0; i < 4; ++i) w[nt].acc[mc][i] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) w[nt].vm[i] = 0.f;
    w[nt].m = kNegBig;
    w[nt].l = 0.f;
  }
  bool timed_out = false;
  for (int i = 0; i < npw; i += 2) {
    const bool hasB = i + 1 < npw;
    bool done = false;
    for (uint32_t it = 0;; ++it) {
      done = done || (mbar_test_s(bar0 + 8 * (i % kDStages), (uint32_t)(i / kDStages) & 1u) &&
                      (!hasB || mbar_test_s(bar0 + 8 * ((i + 1) % kDStages),
                                            (uint32_t)((i + 1) / kDStages) & 1u)));
      if (__all_sync(0xFFFFFFFFu, done) || it >= p.wait_polls) break;
      if (it > 64) __nanosleep(32);
    }
    if (!__all_sync(0xFFFFFFFFu, done)) {
      timed_out = true;
      if (lane == 0) {
        set_status(p.d_status, KITTY_ST_TIMEOUT);
        for (int k = i; k < min(npw, i + kDStages); ++k)
          mbar_wait_bounded(&wbar[k % kDStages], (uint32_t)(k / kDStages) & 1u, kWaitLimit);
      }
      __syncwarp();
      break;
    }
    const int stA = i % kDStages, stB = (i + 1) % kDStages;
    const bool vA = (valid_mask >> stA) & 1u;
    const bool vB = hasB && ((valid_mask >> stB) & 1u);
    const uint32_t paA = stage0 + stA * kBlob;
    const uint32_t paB = hasB ? stage0 + stB * kBlob : paA;
    float bA[2], bB[2];
    pair_beta8<NX>(paA, paB, qft_lane, L, p.sm_log2, bA, bB);
    float sA[2][4], sB[2][4];
    page_scores8<NX>(paA, qft_lane, qxa, L, kscale, bA, sA);
    if (hasB) page_scores8<NX>(paB, qft_lane, qxa, L, kscale, bB, sB);
    if (!vA || (hasB && !vB)) {  // a page id was out of range (warp-uniform, rare)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          sA[nt][k] = vA ? sA[nt][k] : -INFINITY;
          if (hasB) sB[nt][k] = vB ? sB[nt][k] : -INFINITY;
        }
    }
    uint32_t TA[2][4], TB[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      rescale(w[nt], head_max(sA[nt], sB[nt], hasB));
      page_probs(w[nt], sA[nt], TA[nt]);
      if (hasB) page_probs(w[nt], sB[nt], TB[nt]);
    }
    page_pv8<NX>(w, paA, TA, L);
    if (hasB) page_pv8<NX>(w, paB, TB, L);
    __syncwarp();
    if (i + kDStages < npw) issue(i + kDStages);
    if (i + 1 + kDStages < npw) issue(i + 1 + kDStages);
  }
  if (pbeg == 0 && tl > 0 && !timed_out) {
    tail_tokens<DT, V>(w[0], p, qs, b, kvh, tl, wid, L, wst);
    if (gh > kHeadsPerCta) {
      __syncwarp();  // the stage buffer is rewritten
      tail_tokens<DT, V>(w[1], p, qs + kHeadsPerCta * kD, b, kvh, tl, wid, L, wst);
    }
  }
  merge_put(w[0], wst, L);
  merge_put(w[1], wst + kMergeBytes, L);
  __syncthreads();
  merge_get<V>(stages, kDStages * kBlob, 0, p, b, s, h0, min(kHeadsPerCta, gh), L);
  if (gh > kHeadsPerCta)
    merge_get<V>(stages, kDStages * kBlob, kMergeBytes, p, b, s, h0 + kHeadsPerCta, gh - kHeadsPerCta, L);
}

template <int DT, int NX, int W, int V>
cudaError_t launch_decode(dim3 grid, size_t smem, cudaStream_t s, const DecodeParams& p) {
  // the shared-memory opt-in is a per-device function attribute (smem is fixed
  // per instantiation): set it on the first launch on each device only
  static std::atomic<uint64_t> opted_in{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || (opted_in.load() & bit) == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<DT, NX, W, V>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit);
  }
  decode_kernel<DT, NX, W, V><<<grid, kDThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int DT, int NX>
cudaError_t launch_decode8(dim3 grid, size_t smem, cudaStream_t s, const DecodeParams& p) {
  static std::atomic<uint64_t> opted_in{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || (opted_in.load() & bit) == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode8_kernel<DT, NX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit);
  }
  decode8_kernel<DT, NX><<<grid, kDThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_decode8_nx(int nx, dim3 grid, size_t smem, cudaStream_t s, const DecodeParams& p) {
  switch (nx) {
    case 0: return launch_decode8<DT, 0>(grid, smem, s, p);
    case 1: return launch_decode8<DT, 1>(grid, smem, s, p);
    case 2: return launch_decode8<DT, 2>(grid, smem, s, p);
    case 3: return launch_decode8<DT, 3>(grid, smem, s, p);
    case 4: return launch_decode8<DT, 4>(grid, smem, s, p);
    case 5: return launch_decode8<DT, 5>(grid, smem, s, p);
    case 6: return launch_decode8<DT, 6>(grid, smem, s, p);
    case 7: return launch_decode8<DT, 7>(grid, smem, s, p);
    default: return launch_decode8<DT, 8>(grid, smem, s, p);
  }
}

template <int DT, int W, int V>
cudaError_t launch_decode_nx(int nx, dim3 grid, size_t smem, cudaStream_t s, const DecodeParams& p) {
  switch (nx) {
    case 0: return launch_decode<DT, 0, W, V>(grid, smem, s, p);
    case 1: return launch_decode<DT, 1, W, V>(grid, smem, s, p);
    case 2: return launch_decode<DT, 2, W, V>(grid, smem, s, p);
    case 3: return launch_decode<DT, 3, W, V>(grid, smem, s, p);
    case 4: return launch_decode<DT, 4, W, V>(grid, smem, s, p);
    case 5: return launch_decode<DT, 5, W, V>(grid, smem, s, p);
    case 6: return launch_decode<DT, 6, W, V>(grid, smem, s, p);
    case 7: return launch_decode<DT, 7, W, V>(grid, smem, s, p);
    default: return launch_decode<DT, 8, W, V>(grid, smem, s, p);
  }
}

}  // namespace
}  // namespace kitty

using namespace kitty;

namespace {

// Query groups above 4 in the (4, 2) format with 2-bit Values take the
// 8-heads-per-CTA kernel.
bool heads8(const kitty_cfg* cfg) {
  return cfg->num_q_heads / cfg->num_kv_heads > kHeadsPerCta && cfg->lo_bit == 2 && v_bits(cfg) == 2;
}

size_t decode_smem(int blob, int w, bool h8) {
  const int st = stages_for(w);
  const size_t q = h8 ? (8 * kD + 16 * kQx) * 2 + kQft * sizeof(uint32_t) : (4 * kD + 8 * kQx) * 2;
  return (size_t)kDWarps * st * blob + kDWarps * st * sizeof(uint64_t) + q;
}

// Head-group CTAs per (sequence, kv head, split): ceil(g / 8) on the
// 8-heads-per-CTA kernel, else ceil(g / 4).
int head_groups(const kitty_cfg* cfg) {
  const int g = cfg->num_q_heads / cfg->num_kv_heads;
  const int per = heads8(cfg) ? 2 * kHeadsPerCta : kHeadsPerCta;
  return (g + per - 1) / per;
}

// CTAs of the decode kernel resident at once on the device: kDMinBlocks (or
// kDMinBlocks8) per SM unless shared memory allows fewer (large n_hi).
long resident_ctas(int blob, int w, bool h8) {
  int dev = 0, smem_sm = 0;
  int per_sm = h8 ? kDMinBlocks8 : kDMinBlocks;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
      smem_sm > 0) {
    const long fit = (long)smem_sm / (long)(decode_smem(blob, w, h8) + 1024);
    per_sm = (int)std::max(1L, std::min<long>(per_sm, fit));
  }
  return (long)sm_count() * per_sm;
}

struct Schedule {
  int splits;     // splits per sequence
  int largest;    // pages in the largest split
  int32_t starts[kMaxSplits + 1];
};

// Split sizes, in dispatch order, for the (sequence, kv head, head group) units
// of up to M pages on `slots` resident CTAs.
//  * fixed > 0: splits of `fixed` pages (raised to ceil(M / kMaxSplits) if that
//    is larger), the remainder last.
//  * fixed = 0: sizes that shrink towards the end of the grid.  Built from the
//    last split backwards: the last split has m pages, and each earlier one is
//    at most rho = units / slots times the pages that follow it, so a CTA
//    dispatched in round s finishes no later than the work still queued behind
//    it (rounded down to 8 pages; at least m).  The first split takes what is
//    left; if that is smaller than the second, the two are merged and halved.
//    m starts at 16 pages (2 pairs per warp), or at 32 when the batch holds
//    fewer than 64 pages per resident CTA: there every CTA is short and its
//    fixed start and merge cost outweighs the balance of the last round
//    (measured on GB300: 16 x 4096-token Llama-3-8B-shaped layer +7%; the
//    larger layers are 1-2% faster with 16).  m doubles if more than
//    kMaxSplits splits would be needed.
//    With cfg->decode_max_pages (the longest sequence's page count) the sizes
//    are built over that many pages instead of M, and the last split is
//    extended to M, so the table's headroom past every sequence adds no CTA.
//    With cfg->decode_total_pages (the batch's page count) the growth factor is
//    2 rho, and no split exceeds one resident CTA's fair share of the whole
//    batch (Hkv * total / slots pages), which keeps ragged batches balanced;
//    without it the factor stays rho (measured on GB300: +2% on the serving
//    step, +5% on qwen3_8b, +2% on the ragged long-context batch).
//  * With both hints showing equal lengths (total = B * longest) and the units
//    filling at most half of the resident CTAs: k = slots / units equal
//    splits (at least 8 pages each), one wave of equal CTAs.
void plan(const kitty_cfg* cfg, int B, int M, int blob, Schedule* sc) {
  int sz[kMaxSplits];
  int n = 0;
  if (M <= 0) {
    sz[n++] = 0;
  } else if (cfg->decode_pages_per_split > 0) {
    const int c = std::max(cfg->decode_pages_per_split, (M + kMaxSplits - 1) / kMaxSplits);
    const int k = (M + c - 1) / c;
    for (int i = 0; i < k; ++i) sz[n++] = i == k - 1 ? M - (k - 1) * c : c;
  } else {
    const long slots = resident_ctas(blob, cfg->lo_bit, heads8(cfg));
    const bool hinted = cfg->decode_total_pages > 0;
    const long heads = (long)cfg->num_kv_heads * head_groups(cfg);  // CTAs per sequence and split
    const double rho = (hinted ? 2.0 : 1.0) * (double)B * heads / (double)slots;
    const long fair = hinted ? heads * cfg->decode_total_pages / slots / 8 * 8 : (1L << 30);
    const int Ms = cfg->decode_max_pages > 0 ? std::min(M, cfg->decode_max_pages) : M;
    const double work = hinted ? (double)heads * cfg->decode_total_pages
                               : (double)B * heads * Ms;  // page-heads (at most)
    const int m0 = work < 64.0 * (double)slots ? 32 : 16;
    const long units = (long)B * heads;
    if (hinted && cfg->decode_max_pages > 0 && (long)B * Ms == cfg->decode_total_pages &&
        2 * units <= slots) {
      // every sequence holds Ms pages and the units fill at most half of the
      // resident CTAs: k equal splits make one wave of equal CTAs
      const int k = (int)std::min<long>(kMaxSplits, slots / units);
      const int c = std::max(8, (Ms + k - 1) / k);
      for (int t = 0; t < Ms; t += c) sz[n++] = std::min(c, Ms - t);
      sz[n - 1] += M - Ms;  // the last split reaches the end of the table
    } else {
      long T = 0;
      for (int m = m0;; m *= 2) {
        n = 0;
        T = 0;
        long c = m;
        while (T < Ms && n < kMaxSplits) {
          sz[n++] = (int)c;
          T += c;
          c = std::max<long>(m, std::min<long>(fair, (long)(rho * (double)T) / 8 * 8));
        }
        if (T >= Ms) break;
      }
      std::reverse(sz, sz + n);
      sz[0] -= (int)(T - Ms);
      sz[n - 1] += M - Ms;  // the last split reaches the end of the table
      if (n > 1 && sz[0] < sz[1]) {
        const int tot = sz[0] + sz[1];
        const int h = (tot / 2 + 7) / 8 * 8;
        if (h >= tot) {
          sz[0] = tot;
          for (int i = 1; i + 1 < n; ++i) sz[i] = sz[i + 1];
          --n;
        } else {
          sz[0] = h;
          sz[1] = tot - h;
        }
      }
    }
  }
  sc->splits = n;
  sc->largest = 0;
  sc->starts[0] = 0;
  for (int i = 0; i < n; ++i) {
    sc->starts[i + 1] = sc->starts[i] + sz[i];
    sc->largest = std::max(sc->largest, sz[i]);
  }
}

size_t workspace_bytes(const kitty_cfg* cfg, int B, const Schedule& sc) {
  return sc.splits > 1 ? (size_t)B * cfg->num_q_heads * sc.splits * kPartial * sizeof(float) : 0;
}

}  // namespace

extern "C" int kitty_decode_plan(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                 int32_t* splits, int32_t* pages_per_split) {
  int rc = check_cfg(cfg, kMaxGroup);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || !splits || !pages_per_split) return KITTY_ERR_INVALID_ARG;
  Schedule sc;
  plan(cfg, B, max_pages, (int)blob_bytes(cfg->n_hi, cfg->lo_bit, v_bits(cfg)), &sc);
  *splits = sc.splits;
  *pages_per_split = sc.largest;
  return KITTY_OK;
}

extern "C" int kitty_decode_workspace_bytes(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                            size_t* bytes) {
  int rc = check_cfg(cfg, kMaxGroup);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || !bytes) return KITTY_ERR_INVALID_ARG;
  Schedule sc;
  plan(cfg, B, max_pages, (int)blob_bytes(cfg->n_hi, cfg->lo_bit, v_bits(cfg)), &sc);
  *bytes = workspace_bytes(cfg, B, sc);
  return KITTY_OK;
}

namespace {

// Checks and launch shared by the plain and the fused (append + decode) calls.
int attention(const kitty_cfg* cfg, const void* q, const void* pool, int32_t pool_pages,
              const int32_t* block_table, int32_t max_pages, const int32_t* num_pages,
              const void* tail_k, const void* tail_v, const int32_t* tail_len, float sm_scale,
              void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes_in, int32_t B,
              int32_t* d_status, void* stream, const AppendParams& ap) {
  int rc = check_cfg(cfg, kMaxGroup);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (out_dtype != KITTY_F32 && out_dtype != KITTY_BF16 && out_dtype != KITTY_F16)
    return KITTY_ERR_INVALID_ARG;
  if (B == 0) return KITTY_OK;
  if (B > 65535) return KITTY_ERR_UNSUPPORTED;
  if (!q || !out || !num_pages || (max_pages > 0 && (!block_table || !pool)) ||
      (pool && !aligned16(pool)) || ((tail_k == nullptr) != (tail_v == nullptr)) ||
      (tail_k && (!aligned16(tail_k) || !aligned16(tail_v))) ||
      (tail_k && !tail_len) || !std::isfinite(sm_scale))
    return KITTY_ERR_INVALID_ARG;
  const int blob = (int)blob_bytes(cfg->n_hi, cfg->lo_bit, v_bits(cfg));
  DecodeParams p = {};
  Schedule sc;
  plan(cfg, B, max_pages, blob, &sc);
  const size_t need = workspace_bytes(cfg, B, sc);
  if (workspace_bytes_in < need || (need > 0 && (!workspace || !aligned16(workspace))))
    return KITTY_ERR_WORKSPACE;
  for (int i = 0; i <= sc.splits; ++i) p.starts[i] = sc.starts[i];
  p.ap = ap;
  p.q = static_cast<const uint16_t*>(q);
  p.pool = static_cast<const uint8_t*>(pool);
  p.block_table = block_table;
  p.num_pages = num_pages;
  p.tail_k = static_cast<const uint16_t*>(tail_k);
  p.tail_v = static_cast<const uint16_t*>(tail_v);
  p.tail_len = tail_k ? tail_len : nullptr;
  p.out = out;
  p.ws = static_cast<float*>(workspace);
  p.d_status = d_status;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.wait_polls = cfg->decode_wait_polls > 0 ? (uint32_t)cfg->decode_wait_polls : kWaitLimit;
  p.pool_pages = pool_pages;
  p.max_pages = max_pages;
  p.out_dtype = out_dtype;
  p.splits = sc.splits;
  p.Hkv = cfg->num_kv_heads;
  p.Hq = cfg->num_q_heads;
  p.g = cfg->num_q_heads / cfg->num_kv_heads;
  p.HG = head_groups(cfg);
  p.n_hi = cfg->n_hi;
  p.blob = blob;
  p.in_dtype = cfg->in_dtype;
  const bool h8 = heads8(cfg);  // never with a fused append (query groups up to 4 there)
  const size_t smem = decode_smem(p.blob, cfg->lo_bit, h8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid((unsigned)B * cfg->num_kv_heads * p.HG, sc.splits);
  const int nx = cfg->n_hi / 16, v = v_bits(cfg);
  const cudaError_t e = h8 ? (cfg->in_dtype == KITTY_BF16 ? launch_decode8_nx<KITTY_BF16>(nx, grid, smem, s, p)
                                                          : launch_decode8_nx<KITTY_F16>(nx, grid, smem, s, p))
      : cfg->in_dtype == KITTY_BF16
      ? (cfg->lo_bit == 4 ? (v == 4 ? launch_decode_nx<KITTY_BF16, 4, 4>(nx, grid, smem, s, p)
                                    : launch_decode_nx<KITTY_BF16, 4, 2>(nx, grid, smem, s, p))
                          : launch_decode_nx<KITTY_BF16, 2, 2>(nx, grid, smem, s, p))
      : (cfg->lo_bit == 4 ? (v == 4 ? launch_decode_nx<KITTY_F16, 4, 4>(nx, grid, smem, s, p)
                                    : launch_decode_nx<KITTY_F16, 4, 2>(nx, grid, smem, s, p))
                          : launch_decode_nx<KITTY_F16, 2, 2>(nx, grid, smem, s, p));
  if (e != cudaSuccess) return KITTY_ERR_CUDA;
  // the merge step follows the decode grid as a programmatic dependent
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e2 = cudaSuccess;
  if (sc.splits > 1) {
    const int rows = B * cfg->num_q_heads;
    lc.blockDim = dim3(128);
    if (sc.splits <= kCombineSplits) {
      lc.gridDim = dim3((unsigned)(rows + 3) / 4);
      e2 = cudaLaunchKernelEx(&lc, combine_kernel, p, rows);
    } else {
      lc.gridDim = dim3((unsigned)rows);
      e2 = cudaLaunchKernelEx(&lc, combine_wide_kernel, p, rows);
    }
  } else if (ap.k_new != nullptr) {
    lc.gridDim = dim3((unsigned)(B + 127) / 128);
    lc.blockDim = dim3(128);
    e2 = cudaLaunchKernelEx(&lc, finalize_kernel, p, (int)B);
  }
  return e2 == cudaSuccess && cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
}

}  // namespace

extern "C" int kitty_decode_attention(const kitty_cfg* cfg, const void* q, const void* pool,
                                      int32_t pool_pages, const int32_t* block_table,
                                      int32_t max_pages, const int32_t* num_pages,
                                      const void* tail_k, const void* tail_v,
                                      const int32_t* tail_len, float sm_scale, void* out,
                                      int32_t out_dtype, void* workspace, size_t workspace_bytes_in,
                                      int32_t B, int32_t* d_status, void* stream) {
  const AppendParams none = {};
  return attention(cfg, q, pool, pool_pages, block_table, max_pages, num_pages, tail_k, tail_v,
                   tail_len, sm_scale, out, out_dtype, workspace, workspace_bytes_in, B, d_status,
                   stream, none);
}

extern "C" int kitty_append_decode(const kitty_cfg* cfg, const void* k_new, const void* v_new,
                                   const void* q, void* tail_k, void* tail_v, int32_t* tail_len,
                                   float* run_sum, float* run_sumsq, int32_t* run_count,
                                   const int32_t* flush_page_ids, int32_t* block_table,
                                   int32_t max_pages, int32_t* num_pages, void* pool,
                                   int32_t pool_pages, float sm_scale, void* out, int32_t out_dtype,
                                   void* workspace, size_t workspace_bytes, int32_t B,
                                   int32_t* d_status, void* stream) {
  int rc = check_cfg(cfg, kHeadsPerCta);  // one CTA per (sequence, kv head) owns the append
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (B == 0) return KITTY_OK;
  if (!k_new || !v_new || !tail_k || !tail_v || !tail_len || !flush_page_ids || !block_table ||
      !num_pages || !pool)
    return KITTY_ERR_INVALID_ARG;
  const bool running = cfg->rank_mode != KITTY_RANK_PAGE;  // sequence mode appends as running
  if (running && (!run_sum || !run_sumsq || !run_count)) return KITTY_ERR_INVALID_ARG;
  AppendParams ap = {};
  ap.k_new = static_cast<const uint16_t*>(k_new);
  ap.v_new = static_cast<const uint16_t*>(v_new);
  ap.tail_k = static_cast<uint16_t*>(tail_k);
  ap.tail_v = static_cast<uint16_t*>(tail_v);
  ap.tail_len = tail_len;
  ap.num_pages = num_pages;
  ap.block_table = block_table;
  ap.run_sum = running ? run_sum : nullptr;
  ap.run_sumsq = running ? run_sumsq : nullptr;
  ap.run_count = running ? run_count : nullptr;
  ap.flush_page_ids = flush_page_ids;
  ap.pool = static_cast<uint8_t*>(pool);
  ap.running = running ? 1 : 0;
  return attention(cfg, q, pool, pool_pages, block_table, max_pages, num_pages, tail_k, tail_v,
                   tail_len, sm_scale, out, out_dtype, workspace, workspace_bytes, B, d_status,
                   stream, ap);
}

// ------------------------------------------------------------------ no-allocation variant
// Split-K partials in a fixed device array instead of a caller workspace.  Every
// GPU that loads this library holds kNoAllocScratchBytes of it until exit.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (host code must not pass the symbol itself: it names a host stand-in).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KITTY_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return KITTY_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KITTY_OK;
}

}  // namespace

extern "C" int kitty_decode_attention_noalloc(const kitty_cfg* cfg, const void* q, const void* pool,
                                              int32_t pool_pages, const int32_t* block_table,
                                              int32_t max_pages, const int32_t* num_pages,
                                              const void* tail_k, const void* tail_v,
                                              const int32_t* tail_len, float sm_scale, void* out,
                                              int32_t out_dtype, int32_t B, int32_t* d_status,
                                              void* stream) {
  size_t need = 0;
  int rc = kitty_decode_workspace_bytes(cfg, B, max_pages, &need);
  if (rc != KITTY_OK) return rc;
  if (need > kNoAllocScratchBytes) return KITTY_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    rc = scratch_on_current_device(&scratch);
    if (rc != KITTY_OK) return rc;
  }
  return kitty_decode_attention(cfg, q, pool, pool_pages, block_table, max_pages, num_pages, tail_k,
                                tail_v, tail_len, sm_scale, out, out_dtype, scratch,
                                need > 0 ? kNoAllocScratchBytes : 0, B, d_status, stream);
}
