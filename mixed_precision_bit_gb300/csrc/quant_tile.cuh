// Kitty page quantizer, device side: one (page, kv-head) tile quantized by a
// 128-thread CTA into the page-centric blob.  Shared by the quantize/append
// kernels and the fused append + decode kernel.
//
// Paper: "Kitty: Accurate and Efficient 2-bit KV Cache Quantization with
// Dynamic Channel-wise Precision Boost", Abstract.  Steps: "Kitty -- Dynamic
// Channel-wise Mixed-Precision Keys" (VeloxQuant-MLX docs), How it works,
// Prefill phase steps 1-3 and 5, Decode phase steps 1-3.
//
// Every fp32 step uses an explicitly rounded intrinsic (no contraction), in the
// order that defines the page bytes, so the packed pages are bit-exact with a
// plain sequential implementation.  Thread c owns Key channel c; thread 4t+G
// owns Value group G of token t.
#pragma once

#include "kitty_common.cuh"

namespace kitty {
namespace {

constexpr int kQThreads = 128;
constexpr int kMaxBlobWords = (4096 + 17 * kD) / 4;  // largest blob: (8, 4) planes, n_hi = 128

constexpr int kRowH = kD + 8;  // 16-bit elements per staged row (16-byte pad: fewer bank conflicts)

struct QuantSmem {
  uint16_t xk[kPage][kRowH];  // raw 16-bit inputs, token-major
  uint16_t xv[kPage][kRowH];
  uint32_t blob[kMaxBlobWords];
  int warp_cnt[kQThreads / 32];
  int bad;
};

// Fixed pairwise tree over 32 values (upper half folded onto lower half, 16, 8,
// 4, 2, 1 apart) -- the order the page bytes are defined with.
__device__ __forceinline__ float tree32(float* a) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] = __fadd_rn(a[i], a[i + w]);
  }
  return a[0];
}

// sigma^2 ~ sumsq/n - (sum/n)^2, each operation rounded once.
__device__ __forceinline__ float running_var(float sum, float sumsq, float n) {
  const float a = __fdiv_rn(sumsq, n);
  const float b = __fdiv_rn(sum, n);
  return __fsub_rn(a, __fmul_rn(b, b));
}

struct QuantParams {
  float M, u, ru;  // stored minimum and step as fp32, approximate 1/u
  uint16_t Sbits, Mbits;
};

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Asymmetric min/max group quantizer: fp16 minimum and step, codes computed
// against the stored values; a boosted Key channel (2w-bit code) stores
// F = 2^w times its own step, the step of its high w-bit plane.
__device__ __forceinline__ QuantParams qparams(float mn, float mx, int levels, bool boosted,
                                               float F = 4.0f) {
  QuantParams q;
  const __half Mh = __float2half_rn(mn);
  q.M = __half2float(Mh);
  q.Mbits = __half_as_ushort(Mh);
  const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)levels);
  if (boosted) {
    const __half Sh = __float2half_rn(__fmul_rn(F, s));
    q.Sbits = __half_as_ushort(Sh);
    q.u = __fmul_rn(__half2float(Sh), 1.0f / F);
  } else {
    const __half Sh = __float2half_rn(s);
    q.Sbits = __half_as_ushort(Sh);
    q.u = __half2float(Sh);
  }
  q.ru = rcp_approx(q.u);
  return q;
}

// rint(fl(d / u)): the correctly rounded division, out of line (it is taken
// only near a rounding tie, and inlining it at every code site bloats the code).
__device__ __noinline__ float rint_div(float d, float u) { return rintf(__fdiv_rn(d, u)); }

// code = clamp(rint(fl((x - M) / u)), 0, L), bit-exact with an IEEE division.
// The quotient is taken as (x - M) * (1/u), within 2^-21 relative of the true
// value (so within 2^-17 for L <= 15 and 2^-13 for L = 255 inside the clamp
// range); where that lands within 2^-15 (L <= 15) or 2^-12 (L = 255) of a
// rounding tie, the correctly rounded division decides.  u == 0 gives code 0.
__device__ __forceinline__ uint32_t qcode(float x, const QuantParams& q, int levels) {
  if (q.u == 0.0f) return 0u;
  const float d = __fsub_rn(x, q.M);
  const float y = __fmul_rn(d, q.ru);
  float n = rintf(y);
  const float window = levels > 15 ? 0x1p-12f : 0x1p-15f;
  // near a tie (|y - n| is at most 1/2) the division decides; outside [0, L] the
  // clamp makes it moot, but taking it there too is harmless
  if (fabsf(__fsub_rn(y, n)) > 0.5f - window) n = rint_div(d, q.u);
  // n is integral: a saturating conversion clamps below at 0, min() above at L
  return min(__float2uint_rz(n), (uint32_t)levels);
}

// Class of the largest |16-bit input| m (sign bits cleared): 0 ok, RANGE, NONFINITE.
template <int DT>
__device__ __forceinline__ int range_class_of(uint32_t m) {
  if (DT == KITTY_BF16) return m >= 0x7F80u ? KITTY_ST_NONFINITE : (m >= 0x4780u ? KITTY_ST_RANGE : 0);
  return m >= 0x7C00u ? KITTY_ST_NONFINITE : 0;  // fp16 finite values never exceed 65504
}

// Order-preserving key of an fp32 variance (larger var -> larger key), with
// -0 == +0 as in a float comparison.
__device__ __forceinline__ uint32_t var_key(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k boost flag of channel threadIdx.x: true iff fewer than n_hi channels have
// a larger variance, or an equal variance and a lower index.  The n_hi-th
// largest key T is found by a bitwise threshold search; ties at T go to the
// lowest channels.  Called by all 128 threads.
__device__ __forceinline__ bool topk_flag(QuantSmem& sm, float var, int n_hi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (n_hi >= kD) return true;
  if (n_hi <= 0) return false;
  const uint32_t key = var_key(var);
  uint32_t T = 0u;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    if (__syncthreads_count(key >= cand) >= n_hi) T = cand;
  }
  const int n_gt = __syncthreads_count(key > T);
  const bool tie = key == T;
  const uint32_t tb = __ballot_sync(0xFFFFFFFFu, tie);
  if (lane == 0) sm.warp_cnt[warp] = __popc(tb);
  __syncthreads();
  int tie_rank = __popc(tb & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) tie_rank += sm.warp_cnt[w];
  __syncthreads();
  return key > T || (tie && tie_rank < n_hi - n_gt);
}

// Tree-ordered sum and sum of squares of Key channel threadIdx.x over one
// page's 32 tokens (ksrc at token 0, token t at +t*row_stride); stages only K.
template <int DT>
__device__ void tile_stats(QuantSmem& sm, const uint16_t* ksrc, size_t row_stride, float& s1,
                           float& s2) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int it = 0; it < kPage * (kD / 8) / kQThreads; ++it) {
    const int idx = tid + it * kQThreads;
    const int t = idx >> 4, ch = (idx & 15) * 8;
    *reinterpret_cast<uint4*>(&sm.xk[t][ch]) =
        *reinterpret_cast<const uint4*>(ksrc + (size_t)t * row_stride + ch);
  }
  __syncthreads();
  float a[kPage], b[kPage];
#pragma unroll
  for (int t = 0; t < kPage; ++t) {
    a[t] = bits16_to_f32(sm.xk[t][tid], DT);
    b[t] = __fmul_rn(a[t], a[t]);
  }
  s1 = tree32(a);
  s2 = tree32(b);
  __syncthreads();
}

// Quantize one (page, kv-head).  ksrc/vsrc point at token 0 of the tile; token t
// is at +t*row_stride elements.  rsum/rsq/rcount: running accumulators of
// channel `threadIdx.x` (running mode only).  Writes the blob to dst.
// fixed: -1 ranks this page (page or running statistics); 0 / 1 imposes the
// channel's boost flag (sequence-wide ranking), skipping the statistics; -2
// ranks on rsum/rsq/rcount as given (running totals that already include this
// page), leaving them unchanged.
// W = Key plane width (lo_bit): 2 for the (4, 2) configuration, 4 for (8, 4).
template <int DT, int W>
__device__ void quantize_tile(QuantSmem& sm, const uint16_t* ksrc, const uint16_t* vsrc,
                              size_t row_stride, int n_hi, bool running, float& rsum, float& rsq,
                              int& rcount, uint8_t* dst, int32_t* d_status, int fixed = -1) {
  static_assert(W == 2 || W == 4, "Key planes are 2 or 4 bits wide");
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const BlobLayout lay(n_hi, W);
  const int nwords = lay.bytes / 4;
  if (tid == 0) sm.bad = 0;
  for (int i = tid; i < nwords; i += kQThreads) sm.blob[i] = 0u;

  // ---- stage the raw 16-bit tile (16-byte loads and stores), classify the range
  uint32_t amax = 0u;  // per 16-bit half: the largest |input| bits seen
#pragma unroll
  for (int it = 0; it < kPage * (kD / 8) / kQThreads; ++it) {
    const int idx = tid + it * kQThreads;
    const int t = idx >> 4, ch = (idx & 15) * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(ksrc + (size_t)t * row_stride + ch);
    const uint4 b = *reinterpret_cast<const uint4*>(vsrc + (size_t)t * row_stride + ch);
    *reinterpret_cast<uint4*>(&sm.xk[t][ch]) = a;
    *reinterpret_cast<uint4*>(&sm.xv[t][ch]) = b;
    amax = __vmaxu2(amax, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                   __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
    amax = __vmaxu2(amax, __vmaxu2(__vmaxu2(b.x & 0x7FFF7FFFu, b.y & 0x7FFF7FFFu),
                                   __vmaxu2(b.z & 0x7FFF7FFFu, b.w & 0x7FFF7FFFu)));
  }
  __syncthreads();  // tile staged; sm.bad reset by thread 0 is visible
  const int bad = range_class_of<DT>(max(amax & 0xFFFFu, amax >> 16));
  if (bad) atomicCAS(&sm.bad, 0, bad);

  // ---- Key channel statistics and variance (thread = channel c)
  const int c = tid;
  float x[kPage], tmp[kPage];
#pragma unroll
  for (int t = 0; t < kPage; ++t) x[t] = bits16_to_f32(sm.xk[t][c], DT);
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int t = 1; t < kPage; ++t) {
    mn = fminf(mn, x[t]);
    mx = fmaxf(mx, x[t]);
  }
  float var = 0.f;
  if (fixed == -2) {
    var = running_var(rsum, rsq, __int2float_rn(rcount));
  } else if (fixed < 0) {
#pragma unroll
    for (int t = 0; t < kPage; ++t) tmp[t] = x[t];
    const float s1 = tree32(tmp);
#pragma unroll
    for (int t = 0; t < kPage; ++t) tmp[t] = __fmul_rn(x[t], x[t]);
    const float s2 = tree32(tmp);
    if (running) {
      rsum = __fadd_rn(rsum, s1);
      rsq = __fadd_rn(rsq, s2);
      rcount += kPage;
      var = running_var(rsum, rsq, __int2float_rn(rcount));
    } else {
      var = running_var(s1, s2, (float)kPage);
    }
  }

  // ---- top-k (or the caller's fixed boost set)
  const bool boosted = fixed >= 0 ? (fixed != 0) : topk_flag(sm, var, n_hi);
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, boosted);
  if (lane == 0) sm.warp_cnt[warp] = __popc(bal);
  __syncthreads();
  int row = __popc(bal & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) row += sm.warp_cnt[w];

  // ---- Key quantization of channel c and packing in fragment order
  {
    constexpr int kLw = (1 << W) - 1;  // w-bit levels; boosted channels have 2w bits
    const int levels = boosted ? (1 << (2 * W)) - 1 : kLw;
    const QuantParams q = qparams(mn, mx, levels, boosted, (float)(1 << W));
    uint16_t* b16 = reinterpret_cast<uint16_t*>(sm.blob);
    b16[lay.ks / 2 + c] = q.Sbits;
    // minima in fragment order: channel 16j + 8h + 2qq + e at ((qq*8 + j)*2 + h)*2 + e
    b16[lay.km / 2 + (((((c >> 1) & 3) * 8 + (c >> 4)) * 2 + ((c >> 3) & 1)) * 2 + (c & 1))] = q.Mbits;
    uint32_t code[kPage];
#pragma unroll
    for (int t = 0; t < kPage; ++t) code[t] = qcode(x[t], q, levels);
    const int j = c >> 4, half = (c >> 3) & 1, qq = (c >> 1) & 3, e = c & 1;
    const int bitbase = 16 * e + 8 * half;
    const int js = row >> 4, hx = (row >> 3) & 1, qx = (row >> 1) & 3, ex = row & 1;
    const int bx = 16 * ex + 8 * hx;
    if (W == 2) {
      // 2-bit codes: word (lane 4r+qq, tile j) holds tokens 16mt + 8rh + r at 2*(2mt + rh)
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        // the four codes of this lane's byte, at 2*tau, then shifted into place once
        const int sh = boosted ? 2 : 0;
        const uint32_t w = (code[r] >> sh) | ((code[r + 8] >> sh) << 2) |
                           ((code[r + 16] >> sh) << 4) | ((code[r + 24] >> sh) << 6);
        atomicOr(&sm.blob[lay.kbase / 4 + (4 * r + qq) * 8 + j], w << bitbase);
      }
      if (boosted) {
        const int wpl = n_hi / 16;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const uint32_t w = (code[r] & 3u) | ((code[r + 8] & 3u) << 2) |
                             ((code[r + 16] & 3u) << 4) | ((code[r + 24] & 3u) << 6);
          atomicOr(&sm.blob[lay.kextra / 4 + (4 * r + qx) * wpl + js], w << bx);
        }
      }
    } else {
      // 4-bit codes: two words per (lane 4r+qq, tile j), one per 16-token block
      // mt; token 16mt + 8rh + r at nibble 4rh
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int t0 = 16 * mt + r, t1 = t0 + 8;
          const uint32_t c0 = boosted ? (code[t0] >> 4) : code[t0];
          const uint32_t c1 = boosted ? (code[t1] >> 4) : code[t1];
          atomicOr(&sm.blob[lay.kbase / 4 + (4 * r + qq) * 16 + 2 * j + mt],
                   (c0 << bitbase) | (c1 << (bitbase + 4)));
        }
      if (boosted) {
        const int wpl = 2 * (n_hi / 16);
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int t0 = 16 * mt + r, t1 = t0 + 8;
            atomicOr(&sm.blob[lay.kextra / 4 + (4 * r + qx) * wpl + 2 * js + mt],
                     ((code[t0] & 15u) << bx) | ((code[t1] & 15u) << (bx + 4)));
          }
      }
    }
    if (boosted) {
      // channel-list row 16js + 8h + 2qq + e stored at byte js*16 + qq*4 + h*2 + e
      const int pos = lay.kch + js * 16 + qx * 4 + hx * 2 + ex;
      atomicOr(&sm.blob[pos / 4], (uint32_t)c << (8 * (pos & 3)));
    }
  }

  // ---- Value quantization: thread 4t+G owns token t, channels 32G..32G+31
  {
    const int t = tid >> 2, G = tid & 3;
    float v[kVGroup];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(&sm.xv[t][G * kVGroup + 8 * k]);
      const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * k + 2 * i] = bits16_to_f32((uint16_t)(ww[i] & 0xFFFFu), DT);
        v[8 * k + 2 * i + 1] = bits16_to_f32((uint16_t)(ww[i] >> 16), DT);
      }
    }
    float vmn = v[0], vmx = v[0];
#pragma unroll
    for (int i = 1; i < kVGroup; ++i) { vmn = fminf(vmn, v[i]); vmx = fmaxf(vmx, v[i]); }
    const QuantParams q = qparams(vmn, vmx, 3, false);
    uint16_t* b16 = reinterpret_cast<uint16_t*>(sm.blob);
    // Value metadata in fragment order: token 16kt + 8h + 2qq + e at G*32 + qq*8 + kt*4 + h*2 + e
    const int vpos = G * kPage + ((t >> 1) & 3) * 8 + (t >> 4) * 4 + ((t >> 3) & 1) * 2 + (t & 1);
    b16[lay.vs / 2 + vpos] = q.Sbits;
    b16[lay.vm / 2 + vpos] = q.Mbits;
    const int qq = (t >> 1) & 3, kt = t >> 4, half = (t >> 3) & 1, e = t & 1;
    const int bitbase = 16 * e + 8 * half;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      // channel 32G + i (i = 16 odd + 8 rh + r) sits at 2*(2 odd + rh): codes of
      // i = r, r + 8, r + 16, r + 24 at 0, 2, 4, 6, shifted into place once
      const uint32_t w = qcode(v[r], q, 3) | (qcode(v[r + 8], q, 3) << 2) |
                         (qcode(v[r + 16], q, 3) << 4) | (qcode(v[r + 24], q, 3) << 6);
      atomicOr(&sm.blob[lay.vbase / 4 + (4 * r + qq) * 8 + G * 2 + kt], w << bitbase);
    }
  }
  __syncthreads();

  uint4* d4 = reinterpret_cast<uint4*>(dst);
  const uint4* s4 = reinterpret_cast<const uint4*>(sm.blob);
  for (int i = tid; i < lay.bytes / 16; i += kQThreads) d4[i] = s4[i];
  if (tid == 0 && sm.bad) set_status(d_status, sm.bad);
  __syncthreads();
}

// Append bookkeeping of sequence b after every head has used the old values:
// a flush (full tail, page id given, room in the table) appends the page id to
// the block table and empties the tail; otherwise the tail grows by one.
// Invalid lengths leave everything unchanged (the append reported them).
__device__ __forceinline__ void append_finalize_one(int b, int32_t* tail_len,
                                                    const int32_t* flush_page_ids,
                                                    int32_t* block_table, int max_pages,
                                                    int32_t* num_pages, int pool_pages) {
  const int len = tail_len[b];
  if (len < 0 || len >= kPage) return;
  const int n = len + 1;
  const int fid = flush_page_ids[b];
  const int np = num_pages[b];
  if (n == kPage && fid >= 0 && np >= 0 && np < max_pages && fid < pool_pages) {
    block_table[(size_t)b * max_pages + np] = fid;
    num_pages[b] = np + 1;
    tail_len[b] = 0;
  } else {
    tail_len[b] = n;
  }
}

}  // namespace
}  // namespace kitty
