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
constexpr int kMaxBlobWords = (5120 + 17 * kD) / 4;  // largest blob: (8, 4), 4-bit Values, n_hi = 128

constexpr int kRowH = kD + 8;  // 16-bit elements per staged row (16-byte pad: fewer bank conflicts)

struct __align__(16) QuantSmem {  // 16-byte vector accesses to xk, xv and blob
  uint16_t xk[kPage][kRowH];  // raw 16-bit inputs, token-major
  uint16_t xv[kPage][kRowH];
  uint32_t blob[kMaxBlobWords];
  uint32_t key[kD];           // order-preserving variance key of each Key channel
  uint32_t boost[kD / 32];    // boost flag of channel c: bit c & 31 of word c >> 5
  float2 kmm[kD];             // Key channel minimum and maximum, kept over the Value phase
  int bad;
};

// Fixed pairwise tree over 32 values (upper half folded onto lower half, 16, 8,
// 4, 2, 1 apart) -- the order the page bytes are defined with.  The adds of a
// level run two at a time as packed fp32x2 operations (the same roundings).
__device__ __forceinline__ float tree32(float* a) {
#pragma unroll
  for (int w = 16; w >= 2; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; i += 2) add2_rn(a[i], a[i + 1], a[i + w], a[i + w + 1]);
  }
  return __fadd_rn(a[0], a[1]);
}

// sigma^2 ~ sumsq/n - (sum/n)^2, each operation rounded once.
__device__ __forceinline__ float running_var(float sum, float sumsq, float n) {
  const float a = __fdiv_rn(sumsq, n);
  const float b = __fdiv_rn(sum, n);
  return __fsub_rn(a, __fmul_rn(b, b));
}

struct QuantParams {
  float M, u, ru;  // stored minimum and step as fp32, 1/u rounded to nearest
  uint16_t Sbits, Mbits;
};

// Stored step for the exact step s >= 0: the smallest fp16 value >= s whose
// significand has at most 7 bits.  The fp32 pattern is rounded up to 6
// explicit mantissa bits (for s >= 0 the pattern order is the value order, and
// a carry moves on into the exponent), then the value is rounded up to the
// fp16 grid, which only changes values below the fp16 normal range.  A 4-bit
// half of a query or probability times such a step is exact in fp16.
__device__ __forceinline__ uint16_t step_f16(float s) {
  const float v = __uint_as_float((__float_as_uint(s) + 0x1FFFFu) & ~0x1FFFFu);
  const __half h = __float2half_rn(v);
  const uint16_t b = __half_as_ushort(h);
  return __half2float(h) < v ? (uint16_t)(b + 1u) : b;  // next fp16 up (v > 0)
}

// Asymmetric min/max group quantizer: fp16 minimum (nearest) and step
// (step_f16), codes computed against the stored values; a boosted Key channel
// (2w-bit code) stores the step of F = 2^w times its own step, the step of its
// high w-bit plane.
__device__ __forceinline__ QuantParams qparams(float mn, float mx, int levels, bool boosted,
                                               float F = 4.0f) {
  QuantParams q;
  const __half Mh = __float2half_rn(mn);
  q.M = __half2float(Mh);
  q.Mbits = __half_as_ushort(Mh);
  const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)levels);
  if (boosted) {
    q.Sbits = step_f16(__fmul_rn(F, s));
    q.u = __fmul_rn(__half2float(__ushort_as_half(q.Sbits)), 1.0f / F);
  } else {
    q.Sbits = step_f16(s);
    q.u = __half2float(__ushort_as_half(q.Sbits));
  }
  // u == 0: ru = 0 makes every code of a finite input 0
  q.ru = q.u == 0.0f ? 0.0f : __frcp_rn(q.u);
  return q;
}

// Codes of four values: code = clamp(rint((x - M) * (1/u)), 0, L), the
// subtraction and the product rounded to nearest fp32 (two at a time as packed
// fp32x2 operations, the same roundings), 1/u the correctly rounded
// reciprocal, rint to the nearest integer (ties to even).  The conversion to
// an unsigned integer rounds to nearest even and saturates (a negative
// quotient gives 0); min() clamps above at L.
__device__ __forceinline__ void qcode4(const float (&x)[4], const QuantParams& q, int levels,
                                       uint32_t (&code)[4]) {
  float d[4], y[4];
  sub2_rn(d[0], d[1], x[0], x[1], q.M, q.M);
  sub2_rn(d[2], d[3], x[2], x[3], q.M, q.M);
  mul2_rn(y[0], y[1], d[0], d[1], q.ru, q.ru);
  mul2_rn(y[2], y[3], d[2], d[3], q.ru, q.ru);
#pragma unroll
  for (int k = 0; k < 4; ++k) code[k] = min(__float2uint_rn(y[k]), (uint32_t)levels);
}

// Minimum and maximum of two packed 16-bit values per word (bf16x2 or f16x2):
// the order of the values, with -0 below +0 as in the fp32 min/max.
template <int DT>
__device__ __forceinline__ uint32_t min2_16(uint32_t a, uint32_t b) {
  if (DT == KITTY_BF16) {
    const __nv_bfloat162 r = __hmin2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
  const __half2 r = __hmin2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
template <int DT>
__device__ __forceinline__ uint32_t max2_16(uint32_t a, uint32_t b) {
  if (DT == KITTY_BF16) {
    const __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
  }
  const __half2 r = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// One byte of four 2-bit codes, at bits 0, 2, 4, 6.
__device__ __forceinline__ uint8_t pack4x2(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return (uint8_t)(a | (b << 2) | (c << 4) | (d << 6));
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

// Boost masks of the n_hi largest keys of sm.key, ties going to the lowest
// channels: channel c is boosted iff fewer than n_hi channels have a larger key,
// or an equal key and a lower index.  Run by one full warp once sm.key is
// visible; lane l holds the keys of channels l, l + 32, l + 64, l + 96.  A
// bitwise threshold search for the n_hi-th largest key T starts below the
// leading bits that every key shares and stops early once exactly n_hi keys
// are >= the threshold so far (then they are the set); no block barrier is
// taken.
__device__ __forceinline__ void topk_masks(const uint32_t* key, uint32_t* boost, int n_hi) {
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kAll = 0xFFFFFFFFu;
  if (n_hi >= kD || n_hi <= 0) {
    if (lane < kD / 32) boost[lane] = n_hi > 0 ? kAll : 0u;
    return;
  }
  uint32_t k[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) k[m] = key[lane + 32 * m];
  const uint32_t kmax = __reduce_max_sync(kAll, max(max(k[0], k[1]), max(k[2], k[3])));
  const uint32_t kmin = __reduce_min_sync(kAll, min(min(k[0], k[1]), min(k[2], k[3])));
  const uint32_t diff = kmax ^ kmin;
  // the shared leading bits, zeros below: every key is >= T, so >= n_hi of them
  const int top = diff ? 31 - __clz(diff) : -1;
  uint32_t T = top >= 0 ? (kmax & ~((2u << top) - 1u)) : kmax;
  bool exact = false;  // exactly n_hi keys are >= T: they are the set
  for (int bit = top; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    const int cnt = __reduce_add_sync(kAll, (int)(k[0] >= cand) + (int)(k[1] >= cand) +
                                                (int)(k[2] >= cand) + (int)(k[3] >= cand));
    if (cnt >= n_hi) {
      T = cand;
      if (cnt == n_hi) { exact = true; break; }
    }
  }
  uint32_t mask[4];
  if (exact) {
#pragma unroll
    for (int m = 0; m < 4; ++m) mask[m] = __ballot_sync(kAll, k[m] >= T);
  } else {
    // T is the n_hi-th largest key: fewer than n_hi keys exceed it, and the rest
    // of the set are ties at T in channel order
    int need = n_hi - __reduce_add_sync(kAll, (int)(k[0] > T) + (int)(k[1] > T) +
                                                  (int)(k[2] > T) + (int)(k[3] > T));
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t tie = __ballot_sync(kAll, k[m] == T);
      const uint32_t take = __ballot_sync(kAll, k[m] == T && __popc(tie & below) < need);
      mask[m] = __ballot_sync(kAll, k[m] > T) | take;
      need -= __popc(tie);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < 4; ++m) boost[m] = mask[m];
  }
}

// Boost flag of channel c and its row in the channel list (the number of
// boosted channels below c), from sm.boost.
__device__ __forceinline__ bool boost_of(const QuantSmem& sm, int c, int& row) {
  const int g = c >> 5;
  const uint32_t m = sm.boost[g];
  row = __popc(m & ((1u << (c & 31)) - 1u));
  for (int w = 0; w < g; ++w) row += __popc(sm.boost[w]);
  return (m >> (c & 31)) & 1u;
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
  for (int t = 0; t < kPage; ++t) a[t] = bits16_to_f32(sm.xk[t][tid], DT);
#pragma unroll
  for (int t = 0; t < kPage; t += 2) mul2_rn(b[t], b[t + 1], a[t], a[t + 1], a[t], a[t + 1]);
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
// W = Key plane width (lo_bit): 2 for the (4, 2) configuration, 4 for (8, 4);
// V = Value code width: 2, or 4 (with W = 4).
//
// Order of work: Key statistics (thread = channel); then warp 0 ranks the
// channels while the other warps start on the Values (thread 4t+G = token t,
// group G); then the Key codes.  Every code byte of the blob is written once
// by one thread with a byte store.
template <int DT, int W, int V>
__device__ void quantize_tile(QuantSmem& sm, const uint16_t* ksrc, const uint16_t* vsrc,
                              size_t row_stride, int n_hi, bool running, float& rsum, float& rsq,
                              int& rcount, uint8_t* dst, int32_t* d_status, int fixed = -1) {
  static_assert(W == 2 || W == 4, "Key planes are 2 or 4 bits wide");
  static_assert(V == 2 || (V == 4 && W == 4), "Values are 2-bit, or 4-bit with 4-bit Key planes");
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const BlobLayout lay(n_hi, W, V);
  uint8_t* b8 = reinterpret_cast<uint8_t*>(sm.blob);
  uint16_t* b16 = reinterpret_cast<uint16_t*>(sm.blob);
  if (tid == 0) sm.bad = 0;
  // every byte of the blob is written below once the boost set has n_hi
  // channels, as a ranking's always has; zeros keep the page deterministic
  // should an imposed set be smaller
  if (fixed >= 0)
    for (int i = tid; i < lay.bytes / 16; i += kQThreads)
      reinterpret_cast<uint4*>(sm.blob)[i] = make_uint4(0u, 0u, 0u, 0u);

  // ---- stage the raw 16-bit tile with asynchronous 16-byte copies, the Keys
  // in one group and the Values in a second, so that the Values land while the
  // Key statistics run; each thread classifies the range of the chunks it
  // copied (read back once its group has landed)
  constexpr int kChunks = kPage * (kD / 8) / kQThreads;  // 16-byte chunks per thread and tensor
  uint32_t amax = 0u;  // per 16-bit half: the largest |input| bits seen
  auto chunk_max = [&](const uint16_t (*x)[kRowH]) {
#pragma unroll
    for (int it = 0; it < kChunks; ++it) {
      const int idx = tid + it * kQThreads;
      const uint4 a = *reinterpret_cast<const uint4*>(&x[idx >> 4][(idx & 15) * 8]);
      amax = __vmaxu2(amax, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                     __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
    }
  };
#pragma unroll
  for (int it = 0; it < kChunks; ++it) {
    const int idx = tid + it * kQThreads;
    const int t = idx >> 4, ch = (idx & 15) * 8;
    cp_async16(smem_u32(&sm.xk[t][ch]), ksrc + (size_t)t * row_stride + ch);
  }
  cp_async_commit();
#pragma unroll
  for (int it = 0; it < kChunks; ++it) {
    const int idx = tid + it * kQThreads;
    const int t = idx >> 4, ch = (idx & 15) * 8;
    cp_async16(smem_u32(&sm.xv[t][ch]), vsrc + (size_t)t * row_stride + ch);
  }
  cp_async_commit();
  cp_async_wait<1>();  // this thread's Key chunks have landed
  chunk_max(sm.xk);
  __syncthreads();  // Key tile staged (blob zeroed if so); sm.bad reset by thread 0 is visible

  // ---- Key channel statistics and variance (thread = channel c)
  const int c = tid;
  {
    float x[kPage], tmp[kPage], var = 0.f;
#pragma unroll
    for (int t = 0; t < kPage; ++t) x[t] = bits16_to_f32(sm.xk[t][c], DT);
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int t = 1; t < kPage; ++t) {
      mn = fminf(mn, x[t]);
      mx = fmaxf(mx, x[t]);
    }
    if (fixed == -2) {
      var = running_var(rsum, rsq, __int2float_rn(rcount));
    } else if (fixed < 0) {
#pragma unroll
      for (int t = 0; t < kPage; ++t) tmp[t] = x[t];
      const float s1 = tree32(tmp);
#pragma unroll
      for (int t = 0; t < kPage; t += 2) mul2_rn(tmp[t], tmp[t + 1], x[t], x[t + 1], x[t], x[t + 1]);
      const float s2 = tree32(tmp);
      if (running) {
        rsum = __fadd_rn(rsum, s1);
        rsq = __fadd_rn(rsq, s2);
        rcount += kPage;
        var = running_var(rsum, rsq, __int2float_rn(rcount));
      } else {
        // n = 32: dividing by a power of two is multiplying by its inverse, exactly
        const float a = __fmul_rn(s2, 1.0f / kPage), b = __fmul_rn(s1, 1.0f / kPage);
        var = __fsub_rn(a, __fmul_rn(b, b));
      }
    }
    sm.kmm[c] = make_float2(mn, mx);
    if (fixed >= 0) {  // the caller's boost set
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, fixed != 0);
      if (lane == 0) sm.boost[warp] = bal;
    } else {
      sm.key[c] = var_key(var);
    }
  }
  cp_async_wait<0>();  // this thread's Value chunks have landed
  chunk_max(sm.xv);
  {
    const int bad = range_class_of<DT>(max(amax & 0xFFFFu, amax >> 16));
    if (bad) atomicCAS(&sm.bad, 0, bad);
  }
  __syncthreads();  // keys (or imposed flags) and the Value tile visible
  if (fixed < 0 && warp == 0) topk_masks(sm.key, sm.boost, n_hi);

  // ---- Value quantization: thread 4t+G owns token t, channels 32G..32G+31
  {
    const int t = tid >> 2, G = tid & 3;
    float v[kVGroup];
    uint32_t pmn = 0u, pmx = 0u;  // packed pairwise minima and maxima in the input type
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(&sm.xv[t][G * kVGroup + 8 * k]);
      const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * k + 2 * i] = bits16_to_f32((uint16_t)(ww[i] & 0xFFFFu), DT);
        v[8 * k + 2 * i + 1] = bits16_to_f32((uint16_t)(ww[i] >> 16), DT);
        pmn = (k | i) ? min2_16<DT>(pmn, ww[i]) : ww[i];
        pmx = (k | i) ? max2_16<DT>(pmx, ww[i]) : ww[i];
      }
    }
    // the min / max of 16-bit values are exact in their own type
    const float vmn = fminf(bits16_to_f32((uint16_t)(pmn & 0xFFFFu), DT), bits16_to_f32((uint16_t)(pmn >> 16), DT));
    const float vmx = fmaxf(bits16_to_f32((uint16_t)(pmx & 0xFFFFu), DT), bits16_to_f32((uint16_t)(pmx >> 16), DT));
    constexpr int kVLevels = (1 << V) - 1;
    const QuantParams q = qparams(vmn, vmx, kVLevels, false);
    // Value metadata in fragment order: token 16kt + 8h + 2qq + e at G*32 + qq*8 + kt*4 + h*2 + e
    const int vpos = G * kPage + ((t >> 1) & 3) * 8 + (t >> 4) * 4 + ((t >> 3) & 1) * 2 + (t & 1);
    b16[lay.vs / 2 + vpos] = q.Sbits;
    b16[lay.vm / 2 + vpos] = q.Mbits;
    const int qq = (t >> 1) & 3, kt = t >> 4, half = (t >> 3) & 1, e = t & 1;
    if (V == 2) {
      // channel 32G + i (i = 16 odd + 8 rh + r) of token t = 16kt + 8h + 2qq + e sits
      // in word (4r + qq)*8 + 2G + kt, byte 2e + h, at bits 2*(2 odd + rh): the codes
      // of i = r, r + 8, r + 16, r + 24 make one byte
      uint8_t* vb = b8 + lay.vbase + (qq * 8 + 2 * G + kt) * 4 + 2 * e + half;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float xs[4] = {v[r], v[r + 8], v[r + 16], v[r + 24]};
        uint32_t cd[4];
        qcode4(xs, q, kVLevels, cd);
        vb[128 * r] = pack4x2(cd[0], cd[1], cd[2], cd[3]);
      }
    } else {
      // 4-bit: channel 32G + i (i = 16 odd + 8 rh + r) sits in word
      // (4r + qq)*16 + 4G + 2kt + odd, byte 2e + h, nibble rh: the codes of
      // i = r, r + 8 make one byte, those of i = r + 16, r + 24 the byte one word on
      uint8_t* vb = b8 + lay.vbase + (qq * 16 + 4 * G + 2 * kt) * 4 + 2 * e + half;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float xs[4] = {v[r], v[r + 8], v[r + 16], v[r + 24]};
        uint32_t cd[4];
        qcode4(xs, q, kVLevels, cd);
        vb[256 * r] = (uint8_t)(cd[0] | (cd[1] << 4));
        vb[256 * r + 4] = (uint8_t)(cd[2] | (cd[3] << 4));
      }
    }
  }
  __syncthreads();  // boost masks visible

  // ---- Key quantization of channel c and packing in fragment order
  {
    int row;
    const bool boosted = boost_of(sm, c, row);
    constexpr int kLw = (1 << W) - 1;  // w-bit levels; boosted channels have 2w bits
    const int levels = boosted ? (1 << (2 * W)) - 1 : kLw;
    const float2 mm = sm.kmm[c];
    const QuantParams q = qparams(mm.x, mm.y, levels, boosted, (float)(1 << W));
    b16[lay.ks / 2 + c] = q.Sbits;
    // minima in fragment order: channel 16j + 8h + 2qq + e at ((qq*8 + j)*2 + h)*2 + e
    b16[lay.km / 2 + (((((c >> 1) & 3) * 8 + (c >> 4)) * 2 + ((c >> 3) & 1)) * 2 + (c & 1))] = q.Mbits;
    const int j = c >> 4, half = (c >> 3) & 1, qq = (c >> 1) & 3, e = c & 1;
    const int js = row >> 4, hx = (row >> 3) & 1, qx = (row >> 1) & 3, ex = row & 1;
    // channel-list row 16js + 8h + 2qq + e stored at byte js*16 + qq*4 + h*2 + e
    if (boosted) b8[lay.kch + js * 16 + qx * 4 + hx * 2 + ex] = (uint8_t)c;
    if (W == 2) {
      // 2-bit codes: word (4r + qq)*8 + j, byte 2e + h holds tokens r, r + 8,
      // r + 16, r + 24 at bits 0, 2, 4, 6; the extra plane uses the row's place
      const int wpl = n_hi / 16;
      uint8_t* kb = b8 + lay.kbase + (qq * 8 + j) * 4 + 2 * e + half;
      uint8_t* kx = b8 + lay.kextra + (qx * wpl + js) * 4 + 2 * ex + hx;
      const int sh = boosted ? 2 : 0;
#pragma unroll 2
      for (int r = 0; r < 8; ++r) {
        float xs[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) xs[k] = bits16_to_f32(sm.xk[r + 8 * k][c], DT);
        uint32_t cd[4];
        qcode4(xs, q, levels, cd);
        kb[128 * r] = pack4x2(cd[0] >> sh, cd[1] >> sh, cd[2] >> sh, cd[3] >> sh);
        if (boosted) kx[16 * wpl * r] = pack4x2(cd[0] & 3u, cd[1] & 3u, cd[2] & 3u, cd[3] & 3u);
      }
    } else {
      // 4-bit codes: word (4r + qq)*16 + 2j + mt, byte 2e + h holds tokens
      // 16mt + r (low nibble) and 16mt + r + 8 (high nibble)
      const int wpl = 2 * (n_hi / 16);
      uint8_t* kb = b8 + lay.kbase + (qq * 16 + 2 * j) * 4 + 2 * e + half;
      uint8_t* kx = b8 + lay.kextra + (qx * wpl + 2 * js) * 4 + 2 * ex + hx;
      const int sh = boosted ? 4 : 0;
#pragma unroll 2
      for (int r = 0; r < 8; ++r) {
        float xs[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) xs[k] = bits16_to_f32(sm.xk[r + 8 * k][c], DT);
        uint32_t cd[4];
        qcode4(xs, q, levels, cd);
        kb[256 * r] = (uint8_t)((cd[0] >> sh) | ((cd[1] >> sh) << 4));
        kb[256 * r + 4] = (uint8_t)((cd[2] >> sh) | ((cd[3] >> sh) << 4));
        if (boosted) {
          kx[16 * wpl * r] = (uint8_t)((cd[0] & 15u) | ((cd[1] & 15u) << 4));
          kx[16 * wpl * r + 4] = (uint8_t)((cd[2] & 15u) | ((cd[3] & 15u) << 4));
        }
      }
    }
  }
  __syncthreads();
  // Copy out.  The planes' words are stored rotated left by two bits: a code
  // masked out of its 16-bit half then sits two bits higher in the fp16
  // mantissa (the decode folds the factor 4 into its scales).  The rotated
  // words also go back to shared memory, where a fused decode attends to a
  // flushed page.  Plane boundaries (ks, vbase, vbase + 512 V) are multiples
  // of 16 bytes.
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  uint4* s4 = reinterpret_cast<uint4*>(sm.blob);
  for (int i = tid; i < lay.bytes / 16; i += kQThreads) {
    uint4 x = s4[i];
    const int b = 16 * i;
    if (b < lay.ks || (b >= lay.vbase && b < lay.vs)) {
      x.x = __funnelshift_l(x.x, x.x, 2);
      x.y = __funnelshift_l(x.y, x.y, 2);
      x.z = __funnelshift_l(x.z, x.z, 2);
      x.w = __funnelshift_l(x.w, x.w, 2);
      s4[i] = x;
    }
    d4[i] = x;
  }
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
