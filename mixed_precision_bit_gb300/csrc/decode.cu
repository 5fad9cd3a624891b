// Kitty split-K paged decode attention for GB300 (sm_103a).
//
// Paper: "Kitty: Accurate and Efficient 2-bit KV Cache Quantization with
// Dynamic Channel-wise Precision Boost", Abstract (page dequantization over a
// coalesced page-centric layout, no scattered reads or per-channel masks);
// FlashAttention-style online softmax and PagedAttention block tables (both
// cited there).
//
// One CTA = (split, kv head, sequence); 4 warps, each streaming every 4th page
// of the split.  A warp stages whole (page, kv-head) blobs into shared memory
// with 1-D bulk copies (cp.async.bulk + mbarrier, 4 stages per warp), then
// computes, for its g <= 4 query heads:
//   scores  S^T[t][n] = sum_c code[t][c] * B[c][n] on the tensor cores
//           (mma.m16n8k16, fp32 accumulate), B = q*S (per-channel Key step
//           folded into the query) as an fp16 hi/lo pair in columns 0-3 / 4-7,
//           plus the extra plane for the boosted channels (B = q*S/4 gathered
//           through the channel list) and the q.M term as a one-row MMA;
//   softmax fp32 online (max, rescale, exp2) in registers;
//   PV      O^T[c][n] = sum_t vcode[c][t] * P'[t][n] with P' = p*S_v per
//           Value group as an fp16 hi/lo pair, plus the sum_t p*M_v term.
// 2-bit codes are unpacked with one AND each: the planes are stored in
// fragment order, so a masked 16-bit half is the fp16 subnormal
// code * 2^(2*tau - 24); the power of two depends only on the tile row and is
// folded into the score scale (Keys) or the final output (Values).
#include "kitty_common.cuh"
#include "host_common.h"

#include <cmath>
#include <mutex>

namespace kitty {
namespace {

constexpr int kDWarps = 4;
constexpr int kDStages = 4;
constexpr int kDThreads = kDWarps * 32;
constexpr uint32_t kWaitLimit = 1u << 22;  // polls of one barrier phase (~0.1-1 s)
constexpr int kPartial = kD + 2;           // split partial: m, l, o[128]

struct DecodeParams {
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
  int pool_pages, max_pages, out_dtype, splits, chunk, Hkv, Hq, g, n_hi, blob, in_dtype;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 hi/lo split of q*S across lanes: lanes with lomask == 0 get fp16(q*S),
// lanes with lomask == ~0 get fp16(q*S - fp16(q*S)) (the exact residual).
__device__ __forceinline__ uint32_t hilo_mul(uint32_t q, uint32_t S, uint32_t lomask) {
  const __half2 qh = bits_h2(q), Sh = bits_h2(S);
  const uint32_t hi = h2_bits(__hmul2(qh, Sh));
  const uint32_t negc = (hi ^ 0x80008000u) & lomask;
  return h2_bits(__hfma2(qh, Sh, bits_h2(negc)));
}

__device__ __forceinline__ void store_out(void* out, int dt, size_t i, float v) {
  if (dt == KITTY_F32) static_cast<float*>(out)[i] = v;
  else if (dt == KITTY_BF16) static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else static_cast<__half*>(out)[i] = __float2half_rn(v);
}

// Per-warp online-softmax state.  Thread (r = lane/4, qq = lane%4) holds heads
// hA = 2*(qq&1), hB = hA+1; accumulator columns 2qq, 2qq+1 are the hi (qq<2) or
// lo (qq>=2) parts of those heads.
struct WarpState {
  float acc[8][4];  // O^T fragments, m-tile mc = channels 16mc..16mc+15
  float vm[4];      // sum_t p*M_v fragment (rows = Value groups)
  float mA, mB;     // running max (log2 units), warp-uniform per head pair
  float lA, lB;     // this thread's partial softmax denominators
};

// Rescale the state when the running max of a head grows.
__device__ __forceinline__ void update_max(WarpState& w, float pmA, float pmB) {
  const float nA = fmaxf(w.mA, pmA), nB = fmaxf(w.mB, pmB);
  if (__any_sync(0xFFFFFFFFu, nA > w.mA || nB > w.mB)) {
    const float aA = ex2(w.mA - nA), aB = ex2(w.mB - nB);
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      w.acc[mc][0] *= aA; w.acc[mc][1] *= aB; w.acc[mc][2] *= aA; w.acc[mc][3] *= aB;
    }
    w.vm[0] *= aA; w.vm[1] *= aB; w.vm[2] *= aA; w.vm[3] *= aB;
    w.lA *= aA;
    w.lB *= aB;
    w.mA = nA;
    w.mB = nB;
  }
}

// One staged (page, kv-head) blob: scores, online softmax, PV.
//   qf[j][0..1]: this lane's B-fragment query pairs for k-step j (head (lane/4)%4)
//   qs: query heads in fp16, [4][128] in shared memory
__device__ __forceinline__ void compute_page(WarpState& w, const uint8_t* __restrict__ pg,
                                             const uint32_t (&qf)[8][2], const __half* qs,
                                             const BlobLayout& lay, const float (&kscale)[4],
                                             float sm_log2) {
  const int lane = threadIdx.x & 31, r = lane >> 2, qq = lane & 3;
  const uint32_t lomask = lane >= 16 ? 0xFFFFFFFFu : 0u;
  const __half* KS = reinterpret_cast<const __half*>(pg + lay.ks);
  const __half* KM = reinterpret_cast<const __half*>(pg + lay.km);

  // ---------------- scores
  float cs[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  float cm[4] = {0.f, 0.f, 0.f, 0.f};
  const uint4 kb0 = *reinterpret_cast<const uint4*>(pg + lay.kbase + 32 * lane);
  const uint4 kb1 = *reinterpret_cast<const uint4*>(pg + lay.kbase + 32 * lane + 16);
  const uint32_t kw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c0 = 16 * j + 2 * qq;
    const uint32_t S0 = *reinterpret_cast<const uint32_t*>(KS + c0);
    const uint32_t S1 = *reinterpret_cast<const uint32_t*>(KS + c0 + 8);
    const uint32_t b0 = hilo_mul(qf[j][0], S0, lomask);
    const uint32_t b1 = hilo_mul(qf[j][1], S1, lomask);
    const uint32_t x = kw[j], x2 = x >> 8;
    const uint32_t a0[4] = {x & 0x00030003u, x & 0x000C000Cu, x2 & 0x00030003u, x2 & 0x000C000Cu};
    const uint32_t a1[4] = {x & 0x00300030u, x & 0x00C000C0u, x2 & 0x00300030u, x2 & 0x00C000C0u};
    mma_f16(cs[0], a0, b0, b1);
    mma_f16(cs[1], a1, b0, b1);
    const uint32_t am[4] = {r == 0 ? *reinterpret_cast<const uint32_t*>(KM + c0) : 0u, 0u,
                            r == 0 ? *reinterpret_cast<const uint32_t*>(KM + c0 + 8) : 0u, 0u};
    mma_f16(cm, am, qf[j][0], qf[j][1]);
  }
  // extra plane: low 2 bits of the boosted channels' 4-bit codes, step S/4
  const int nx = lay.n_hi >> 4;
  const uint8_t* kch = pg + lay.kch;
  const uint32_t* xw = reinterpret_cast<const uint32_t*>(pg + lay.kextra) + lane * nx;
  const __half* qh = qs + (r & 3) * kD;
  const __half2 quarter = __float2half2_rn(0.25f);
  for (int js = 0; js < nx; ++js) {
    const int j0 = 16 * js + 2 * qq;
    const int ch0 = kch[j0] & 127, ch1 = kch[j0 + 1] & 127;
    const int ch2 = kch[j0 + 8] & 127, ch3 = kch[j0 + 9] & 127;
    const __half2 q01 = __halves2half2(qh[ch0], qh[ch1]);
    const __half2 q23 = __halves2half2(qh[ch2], qh[ch3]);
    const __half2 s01 = __hmul2(__halves2half2(KS[ch0], KS[ch1]), quarter);
    const __half2 s23 = __hmul2(__halves2half2(KS[ch2], KS[ch3]), quarter);
    const uint32_t b0 = hilo_mul(h2_bits(q01), h2_bits(s01), lomask);
    const uint32_t b1 = hilo_mul(h2_bits(q23), h2_bits(s23), lomask);
    const uint32_t x = xw[js], x2 = x >> 8;
    const uint32_t a0[4] = {x & 0x00030003u, x & 0x000C000Cu, x2 & 0x00030003u, x2 & 0x000C000Cu};
    const uint32_t a1[4] = {x & 0x00300030u, x & 0x00C000C0u, x2 & 0x00300030u, x2 & 0x00C000C0u};
    mma_f16(cs[0], a0, b0, b1);
    mma_f16(cs[1], a1, b0, b1);
  }
  // combine hi/lo columns (lane ^ 2 holds the other half), add q.M, scale
  const float bA = __shfl_sync(0xFFFFFFFFu, cm[0], qq) * sm_log2;
  const float bB = __shfl_sync(0xFFFFFFFFu, cm[1], qq) * sm_log2;
  float s[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v = cs[mt][i] + __shfl_xor_sync(0xFFFFFFFFu, cs[mt][i], 2);
      s[mt][i] = fmaf(v, kscale[2 * mt + (i >> 1)], (i & 1) ? bB : bA);
    }
  float pmA = fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2]));
  float pmB = fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    pmA = fmaxf(pmA, __shfl_xor_sync(0xFFFFFFFFu, pmA, off));
    pmB = fmaxf(pmB, __shfl_xor_sync(0xFFFFFFFFu, pmB, off));
  }
  update_max(w, pmA, pmB);

  // ---------------- probabilities, hi/lo split, transpose to B fragments
  const bool lo_pre = qq >= 2;
  uint32_t T[4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const float pA = ex2(s[mt][2 * rh] - w.mA);
      const float pB = ex2(s[mt][2 * rh + 1] - w.mB);
      w.lA += pA;
      w.lB += pB;
      const float tA = __uint_as_float(__float_as_uint(pA) & 0xFFFFE000u);
      const float tB = __uint_as_float(__float_as_uint(pB) & 0xFFFFE000u);
      const __half2 pk = __floats2half2_rn(lo_pre ? pA - tA : tA, lo_pre ? pB - tB : tB);
      T[2 * mt + rh] = movmatrix_t(h2_bits(pk));
    }
  // lanes 0-15 hold p_hi (columns 0-3), lanes 16-31 p_lo (columns 4-7)

  // ---------------- Value min term: rows = groups, k = tokens
  const __half* VS = reinterpret_cast<const __half*>(pg + lay.vs);
  const __half* VMv = reinterpret_cast<const __half*>(pg + lay.vm);
#pragma unroll
  for (int kt = 0; kt < 2; ++kt) {
    const int t0 = 16 * kt + 2 * qq;
    const uint32_t am[4] = {r < 4 ? *reinterpret_cast<const uint32_t*>(VMv + r * kPage + t0) : 0u, 0u,
                            r < 4 ? *reinterpret_cast<const uint32_t*>(VMv + r * kPage + t0 + 8) : 0u, 0u};
    mma_f16(w.vm, am, T[2 * kt], T[2 * kt + 1]);
  }

  // ---------------- PV with the Value step folded into P per group
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ph[i] = __shfl_sync(0xFFFFFFFFu, T[i], lane & 15);
    pl[i] = T[i] & lomask;
  }
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(pg + lay.vbase + 32 * lane);
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    const uint2 vv = *reinterpret_cast<const uint2*>(vw + 2 * G);
    const uint32_t vwords[2] = {vv.x, vv.y};
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      uint32_t bg[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int t0 = 16 * kt + 8 * k + 2 * qq;
        const __half2 S = bits_h2(*reinterpret_cast<const uint32_t*>(VS + G * kPage + t0));
        const __half2 a = bits_h2(ph[2 * kt + k]);
        const uint32_t h = h2_bits(__hmul2(a, S));
        const uint32_t negc = (h ^ 0x80008000u) & lomask;
        const __half2 rr = __hfma2(a, S, bits_h2(negc));
        bg[k] = h2_bits(__hfma2(bits_h2(pl[2 * kt + k]), S, rr));
      }
      const uint32_t x = vwords[kt], x2 = x >> 8;
      const uint32_t ae[4] = {x & 0x00030003u, x & 0x000C000Cu, x2 & 0x00030003u, x2 & 0x000C000Cu};
      const uint32_t ao[4] = {x & 0x00300030u, x & 0x00C000C0u, x2 & 0x00300030u, x2 & 0x00C000C0u};
      mma_f16(w.acc[2 * G], ae, bg[0], bg[1]);
      mma_f16(w.acc[2 * G + 1], ao, bg[0], bg[1]);
    }
  }
}

// Unquantized tail tokens (0..31 per sequence), CUDA-core path: warp `wid`
// takes tail tokens wid, wid+4, ...  Contributions go to the hi columns with
// the same per-row power of two as the paged codes.
template <int DT>
__device__ void tail_tokens(WarpState& w, const DecodeParams& p, const __half* qs, int b, int kvh,
                            int tl, int wid) {
  const int lane = threadIdx.x & 31, r = lane >> 2, qq = lane & 3;
  const size_t base = ((size_t)b * p.Hkv + kvh) * kPage * kD;
  float qv[4][4];
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i) qv[h][i] = __half2float(qs[h * kD + 4 * lane + i]);
  for (int t = wid; t < tl; t += kDWarps) {
    const uint16_t* kr = p.tail_k + base + (size_t)t * kD;
    const uint16_t* vr = p.tail_v + base + (size_t)t * kD;
    float kx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) kx[i] = load16<DT>(kr + 4 * lane + i);
    float d[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      d[h] = qv[h][0] * kx[0] + qv[h][1] * kx[1] + qv[h][2] * kx[2] + qv[h][3] * kx[3];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) d[h] += __shfl_xor_sync(0xFFFFFFFFu, d[h], off);
    }
    const int hA = 2 * (qq & 1);
    const float sA = (hA == 0 ? d[0] : d[2]) * p.sm_log2;
    const float sB = (hA == 0 ? d[1] : d[3]) * p.sm_log2;
    update_max(w, sA, sB);
    const float pA = ex2(sA - w.mA), pB = ex2(sB - w.mB);
    if (r == 0) { w.lA += pA; w.lB += pB; }
    if (qq < 2) {
#pragma unroll
      for (int mc = 0; mc < 8; ++mc)
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          const int c = 16 * mc + 8 * rh + r;
          const float sc = __uint_as_float((uint32_t)(127 - 24 + 2 * (2 * (mc & 1) + rh)) << 23);
          const float v = load16<DT>(vr + c) * sc;
          w.acc[mc][2 * rh] += pA * v;
          w.acc[mc][2 * rh + 1] += pB * v;
        }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kDThreads, 4) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, r = lane >> 2, qq = lane & 3;
  int np = p.num_pages[b];
  int tl = p.tail_len != nullptr ? p.tail_len[b] : 0;
  if (np < 0 || np > p.max_pages || tl < 0 || tl > kPage || (tl > 0 && p.tail_k == nullptr)) {
    if (tid == 0 && s == 0 && kvh == 0) set_status(p.d_status, KITTY_ST_BAD_LEN);
    np = 0;
    tl = 0;
  }
  const int n_act = max(1, (np + p.chunk - 1) / p.chunk);
  if (s >= n_act) return;
  const int pbeg = s * p.chunk, pend = min(np, pbeg + p.chunk);
  const BlobLayout lay(p.n_hi);

  uint8_t* stages = dsm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + kDWarps * kDStages * p.blob);
  __half* qs = reinterpret_cast<__half*>(bars + kDWarps * kDStages);
  for (int i = tid; i < 4 * kD; i += kDThreads) {
    const int h = i >> 7, c = i & (kD - 1);
    float v = 0.f;
    if (h < p.g) v = load16<DT>(p.q + ((size_t)b * p.Hq + (size_t)kvh * p.g + h) * kD + c);
    qs[i] = __float2half_rn(v);
  }
  if (lane == 0) {
    for (int st = 0; st < kDStages; ++st) mbar_init(&bars[wid * kDStages + st], 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint32_t qf[8][2];
  {
    const __half* qh = qs + (r & 3) * kD;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qf[j][0] = *reinterpret_cast<const uint32_t*>(qh + 16 * j + 2 * qq);
      qf[j][1] = *reinterpret_cast<const uint32_t*>(qh + 16 * j + 2 * qq + 8);
    }
  }
  float kscale[4];
#pragma unroll
  for (int tau = 0; tau < 4; ++tau)
    kscale[tau] = p.sm_log2 * __uint_as_float((uint32_t)(127 + 24 - 2 * tau) << 23);

  WarpState w;
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int i = 0; i < 4; ++i) w.acc[mc][i] = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) w.vm[i] = 0.f;
  w.mA = w.mB = -INFINITY;
  w.lA = w.lB = 0.f;

  // ---- this warp's pages: pbeg + wid + kDWarps*i, i < npw
  const int first = pbeg + wid;
  const int npw = pend > first ? (pend - first + kDWarps - 1) / kDWarps : 0;
  uint8_t* wst = stages + (size_t)wid * kDStages * p.blob;
  uint64_t* wbar = bars + wid * kDStages;
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages;
  const size_t head_off = (size_t)kvh * p.blob;
  const size_t page_stride = (size_t)p.Hkv * p.blob;
  int bt_cache = -1, bt_base = -64;
  uint32_t valid_mask = 0;  // bit st: stage st holds a valid page
  auto issue = [&](int i) {
    if (i - bt_base >= 32) {
      bt_base = i;
      bt_cache = (i + lane < npw) ? bt[first + (i + lane) * kDWarps] : -1;
    }
    const int pid = __shfl_sync(0xFFFFFFFFu, bt_cache, i - bt_base);
    const int st = i % kDStages;
    const bool ok = pid >= 0 && pid < p.pool_pages;
    if (lane == 0) {
      if (ok) {
        mbar_arrive_expect_tx(&wbar[st], (uint32_t)p.blob);
        bulk_g2s(wst + (size_t)st * p.blob, p.pool + (size_t)pid * page_stride + head_off,
                 (uint32_t)p.blob, &wbar[st]);
      } else {
        set_status(p.d_status, KITTY_ST_BAD_PAGE);
        mbar_arrive(&wbar[st]);
      }
    }
    valid_mask = ok ? (valid_mask | (1u << st)) : (valid_mask & ~(1u << st));
  };
  const int pro = min(npw, kDStages);
  for (int i = 0; i < pro; ++i) issue(i);
  for (int i = 0; i < npw; ++i) {
    const int st = i % kDStages;
    const uint32_t par = (uint32_t)(i / kDStages) & 1u;
    int ok = 0;
    if (lane == 0) ok = mbar_wait_bounded(&wbar[st], par, kWaitLimit) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) {
      // give up: report, then wait (bounded) for every copy still in flight
      if (lane == 0) {
        set_status(p.d_status, KITTY_ST_TIMEOUT);
        for (int k = i + 1; k < min(npw, i + kDStages); ++k)
          mbar_wait_bounded(&wbar[k % kDStages], (uint32_t)(k / kDStages) & 1u, kWaitLimit);
      }
      __syncwarp();
      break;
    }
    if (valid_mask & (1u << st))
      compute_page(w, wst + (size_t)st * p.blob, qf, qs, lay, kscale, p.sm_log2);
    __syncwarp();
    if (i + kDStages < npw) issue(i + kDStages);
  }
  if (s == 0 && tl > 0) {
    if (p.in_dtype == KITTY_BF16) tail_tokens<KITTY_BF16>(w, p, qs, b, kvh, tl, wid);
    else tail_tokens<KITTY_F16>(w, p, qs, b, kvh, tl, wid);
  }

  // ---- merge the 4 warps: per-warp (m, l, O) to shared memory, then per channel
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    w.lA += __shfl_xor_sync(0xFFFFFFFFu, w.lA, off);
    w.lB += __shfl_xor_sync(0xFFFFFFFFu, w.lB, off);
  }
  __syncthreads();
  constexpr int kMergeFloats = kD * 8 + 4 * 8 + 8;
  float* mw = reinterpret_cast<float*>(dsm) + wid * kMergeFloats;
  float* Ow = mw;               // [128][8]
  float* VMw = mw + kD * 8;     // [4][8]
  float* MLw = VMw + 4 * 8;     // m[4], l[4]
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rh = i >> 1;
      const int row = 16 * mc + 8 * rh + r;
      const float sc = __uint_as_float((uint32_t)(127 + 24 - 2 * (2 * (mc & 1) + rh)) << 23);
      Ow[row * 8 + 2 * qq + (i & 1)] = w.acc[mc][i] * sc;
    }
  if (r < 4) {
    VMw[r * 8 + 2 * qq] = w.vm[0];
    VMw[r * 8 + 2 * qq + 1] = w.vm[1];
  }
  if (r == 0 && qq < 2) {
    MLw[2 * qq] = w.mA;
    MLw[2 * qq + 1] = w.mB;
    MLw[4 + 2 * qq] = w.lA;
    MLw[4 + 2 * qq + 1] = w.lB;
  }
  __syncthreads();
  const int c = tid;
  const int G = c >> 5;
  const float* m0 = reinterpret_cast<const float*>(dsm);
  for (int h = 0; h < p.g; ++h) {
    float ms = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kDWarps; ++ww) ms = fmaxf(ms, m0[ww * kMergeFloats + kD * 8 + 32 + h]);
    float L = 0.f, O = 0.f;
    if (ms != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < kDWarps; ++ww) {
        const float* base = m0 + ww * kMergeFloats;
        const float mwv = base[kD * 8 + 32 + h];
        const float e = mwv == -INFINITY ? 0.f : ex2(mwv - ms);
        L += base[kD * 8 + 32 + 4 + h] * e;
        const float o = base[c * 8 + h] + base[c * 8 + h + 4] + base[kD * 8 + G * 8 + h] +
                        base[kD * 8 + G * 8 + h + 4];
        O += o * e;
      }
    }
    const int hq = kvh * p.g + h;
    if (p.splits == 1) {
      store_out(p.out, p.out_dtype, ((size_t)b * p.Hq + hq) * kD + c, L > 0.f ? O / L : 0.f);
      if (c == 0 && !(L > 0.f)) set_status(p.d_status, KITTY_ST_EMPTY);
    } else {
      float* part = p.ws + (((size_t)b * p.Hq + hq) * p.splits + s) * kPartial;
      part[2 + c] = O;
      if (c == 0) { part[0] = ms; part[1] = L; }
    }
  }
}

// Merge the split partials of one (sequence, query head); 128 threads = channels.
__global__ void __launch_bounds__(kD) combine_kernel(const float* __restrict__ ws,
                                                     const int32_t* num_pages, int max_pages,
                                                     int chunk, int splits, int Hq, void* out,
                                                     int out_dtype, int32_t* d_status) {
  const int bh = blockIdx.x, b = bh / Hq, c = threadIdx.x;
  int np = num_pages[b];
  if (np < 0 || np > max_pages) np = 0;
  const int n_act = max(1, (np + chunk - 1) / chunk);
  const float* base = ws + (size_t)bh * splits * kPartial;
  float ms = -INFINITY;
  for (int s = 0; s < n_act; ++s) ms = fmaxf(ms, base[s * kPartial]);
  float L = 0.f, O = 0.f;
  if (ms != -INFINITY) {
    for (int s = 0; s < n_act; ++s) {
      const float m = base[s * kPartial];
      const float e = m == -INFINITY ? 0.f : ex2(m - ms);
      L += base[s * kPartial + 1] * e;
      O += base[s * kPartial + 2 + c] * e;
    }
  }
  store_out(out, out_dtype, (size_t)bh * kD + c, L > 0.f ? O / L : 0.f);
  if (c == 0 && !(L > 0.f)) set_status(d_status, KITTY_ST_EMPTY);
}

}  // namespace
}  // namespace kitty

using namespace kitty;

namespace {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// Split-K plan: enough CTAs for ~3 waves of 4 resident CTAs per SM, at least
// 16 pages (4 per warp) per split unless the sequence is shorter.
void plan(const kitty_cfg* cfg, int B, int max_pages, int* splits, int* chunk) {
  int ch = cfg->decode_pages_per_split;
  if (ch <= 0) {
    const long units = (long)B * cfg->num_kv_heads;
    const long target = 3L * sm_count() * 4;
    const long want = units > 0 ? (target + units - 1) / units : 1;
    long c = (max_pages + want - 1) / (want > 0 ? want : 1);
    if (c < 16) c = 16;
    c = (c + kDWarps - 1) / kDWarps * kDWarps;
    ch = (int)c;
  }
  const int sp = max_pages > 0 ? (max_pages + ch - 1) / ch : 1;
  *splits = sp < 1 ? 1 : sp;
  *chunk = ch;
}

size_t decode_smem(int blob) {
  return (size_t)kDWarps * kDStages * blob + kDWarps * kDStages * sizeof(uint64_t) + 4 * kD * 2;
}

}  // namespace

extern "C" int kitty_decode_plan(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                 int32_t* splits, int32_t* pages_per_split) {
  int rc = check_cfg(cfg, true);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || !splits || !pages_per_split) return KITTY_ERR_INVALID_ARG;
  int sp, ch;
  plan(cfg, B, max_pages, &sp, &ch);
  *splits = sp;
  *pages_per_split = ch;
  return KITTY_OK;
}

extern "C" int kitty_decode_workspace_bytes(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                            size_t* bytes) {
  int rc = check_cfg(cfg, true);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || !bytes) return KITTY_ERR_INVALID_ARG;
  int sp, ch;
  plan(cfg, B, max_pages, &sp, &ch);
  *bytes = sp > 1 ? (size_t)B * cfg->num_q_heads * sp * kPartial * sizeof(float) : 0;
  return KITTY_OK;
}

extern "C" int kitty_decode_attention(const kitty_cfg* cfg, const void* q, const void* pool,
                                      int32_t pool_pages, const int32_t* block_table,
                                      int32_t max_pages, const int32_t* num_pages,
                                      const void* tail_k, const void* tail_v,
                                      const int32_t* tail_len, float sm_scale, void* out,
                                      int32_t out_dtype, void* workspace, size_t workspace_bytes,
                                      int32_t B, int32_t* d_status, void* stream) {
  int rc = check_cfg(cfg, true);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (out_dtype != KITTY_F32 && out_dtype != KITTY_BF16 && out_dtype != KITTY_F16)
    return KITTY_ERR_INVALID_ARG;
  if (B == 0) return KITTY_OK;
  if (B > 65535) return KITTY_ERR_UNSUPPORTED;
  if (!q || !out || !num_pages || (max_pages > 0 && (!block_table || !pool)) ||
      (pool && !aligned16(pool)) || ((tail_k == nullptr) != (tail_v == nullptr)) ||
      (tail_k && !tail_len) || !std::isfinite(sm_scale))
    return KITTY_ERR_INVALID_ARG;
  int sp, ch;
  plan(cfg, B, max_pages, &sp, &ch);
  size_t need = sp > 1 ? (size_t)B * cfg->num_q_heads * sp * kPartial * sizeof(float) : 0;
  if (workspace_bytes < need || (need > 0 && (!workspace || !aligned16(workspace))))
    return KITTY_ERR_WORKSPACE;
  DecodeParams p;
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
  p.pool_pages = pool_pages;
  p.max_pages = max_pages;
  p.out_dtype = out_dtype;
  p.splits = sp;
  p.chunk = ch;
  p.Hkv = cfg->num_kv_heads;
  p.Hq = cfg->num_q_heads;
  p.g = cfg->num_q_heads / cfg->num_kv_heads;
  p.n_hi = cfg->n_hi;
  p.blob = (int)blob_bytes(cfg->n_hi);
  p.in_dtype = cfg->in_dtype;
  const size_t smem = decode_smem(p.blob);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(sp, cfg->num_kv_heads, B);
  if (cfg->in_dtype == KITTY_BF16) {
    if (cudaFuncSetAttribute(decode_kernel<KITTY_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return KITTY_ERR_CUDA;
    decode_kernel<KITTY_BF16><<<grid, kDThreads, smem, s>>>(p);
  } else {
    if (cudaFuncSetAttribute(decode_kernel<KITTY_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return KITTY_ERR_CUDA;
    decode_kernel<KITTY_F16><<<grid, kDThreads, smem, s>>>(p);
  }
  if (sp > 1)
    combine_kernel<<<B * cfg->num_q_heads, kD, 0, s>>>(p.ws, num_pages, max_pages, ch, sp, cfg->num_q_heads, out, out_dtype, d_status);
  return cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
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
