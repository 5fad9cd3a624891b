// Kitty CPU oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-source C++17 restatement of what the Kitty hot path
// computes: per-page channel statistics, variance ranking with a top-k boost
// set, asymmetric min/max quantization of Keys (lo_bit codes; boosted channels
// hi_bit = 2*lo_bit, split into two uniform lo_bit planes; (hi_bit, lo_bit) =
// (4, 2) by default or (8, 4)) and Values (per-token groups of 32 channels,
// 2-bit, or 4-bit with 4-bit Key planes), the packed page format, the
// append/flush step, and fp64 decode attention over the dequantized pages.
//
// Only the test suite, the package's smoke check and the bench's CPU-baseline
// leg may load this library.  It shares no code with the CUDA path.  Build with
// -O2 -ffp-contract=off (no fused multiply-add): every fp32 operation below is
// one IEEE round-to-nearest-even operation, in the order written.
//
// Sources (by page title and section):
//  * "Kitty: Accurate and Efficient 2-bit KV Cache Quantization with Dynamic
//    Channel-wise Precision Boost" (arXiv 2511.18643), Abstract: channel
//    ranking with a small boosted fraction, each mixed-precision Key page
//    decomposed into two uniform 2-bit tensors, page-centric layout.
//  * "Kitty -- Dynamic Channel-wise Mixed-Precision Keys" (VeloxQuant-MLX docs),
//    How it works / Prefill phase steps 1-3 (per-channel variance, top
//    hi_fraction*D channels at hi_bit, asymmetric min/max groups of group_size
//    tokens), Decode phase step 2 (running variance formula), Effective
//    bit-width, Configuration reference, Tuning avg_bits (the (0.25, 8, 4) row:
//    8-bit boosted and 4-bit other Key channels; Values keep their 2-bit
//    format -- the table concerns Keys only, a reading).  The same paper's
//    Abstract names 4-bit KV quantization as the accuracy-preserving point
//    Kitty is measured against: with n_hi = 0, 4-bit Key planes and 4-bit
//    Values (v_bit = 4) this format is that uniform 4-bit KV cache (a reading:
//    the same per-channel Key and per-token Value groups at 15 levels).
//  * PagedAttention / FlashAttention (cited by the paper) for the block table
//    and softmax attention semantics.
// Readings where the pages are silent are stated next to the code that takes
// them.  Parity status of every function is pinned by the CPU test suite.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int D = 128;        // head_dim (the only supported value)
constexpr int P = 32;         // tokens per page = kitty_group_size
constexpr int VG = 32;        // channels per Value group

// ---------------------------------------------------------------- formats
// IEEE binary16 / bfloat16 <-> binary32, written out from the encodings.

float f16_to_f32(uint16_t h) {
  const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  const uint32_t e = (h >> 10) & 0x1Fu;
  const uint32_t m = h & 0x3FFu;
  uint32_t bits;
  if (e == 0) {
    if (m == 0) {
      bits = sign;
    } else {  // subnormal: m * 2^-24, exact in fp32
      float v = std::ldexp((float)m, -24);
      std::memcpy(&bits, &v, 4);
      bits |= sign;
    }
  } else if (e == 31) {
    bits = sign | 0x7F800000u | (m << 13);
  } else {
    bits = sign | ((e - 15 + 127) << 23) | (m << 13);
  }
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

float bf16_to_f32(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// binary32 -> binary16, round to nearest, ties to even, with subnormals.
uint16_t f32_to_f16(float f) {
  uint32_t x;
  std::memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  const uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x200u : 0u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);  // >= 65520 rounds to inf
  if (ax >= 0x38800000u) {                                     // normal half range
    const uint32_t e = (ax >> 23) - 127 + 15;
    const uint32_t mant = ax & 0x7FFFFFu;
    uint32_t h = (e << 10) | (mant >> 13);
    const uint32_t rem = mant & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;
    return (uint16_t)(sign | h);
  }
  if (ax < 0x33000000u) return (uint16_t)sign;  // below 2^-25: rounds to zero
  const uint32_t e = ax >> 23;                   // 102..112
  const uint32_t M = (ax & 0x7FFFFFu) | 0x800000u;
  const uint32_t s = 126 - e;                    // 14..24
  uint32_t m = M >> s;
  const uint32_t rem = M & ((1u << s) - 1u);
  const uint32_t half = 1u << (s - 1);
  if (rem > half || (rem == half && (m & 1u))) m++;
  return (uint16_t)(sign | m);
}

float in_to_f32(uint16_t v, int dtype) { return dtype == 1 ? bf16_to_f32(v) : f16_to_f32(v); }

// ---------------------------------------------------------------- page format
// The Key planes are w bits wide: w = lo_bit, and hi_bit = 2*w (a boosted code
// splits into two w-bit halves).  w = 2 is the paper's (4, 2) configuration,
// w = 4 the (8, 4) row of the avg_bits table.
// Byte layout of one (page, kv-head) blob, n_hi a multiple of 16 in [0, 128]:
//   Kbase  128*w B    w-bit codes, all D channels x 32 tokens (high halves of boosted codes)
//   Kextra n_hi*4*w B w-bit low halves of the boosted channels' 2w-bit codes
//   KS     256 B      fp16 step per channel, channel order (boosted: the base-plane step)
//   KM     256 B      fp16 minimum per channel, at km_pos(c)
//   Kch    n_hi B     boosted channel ids; row j of Kextra (the j-th smallest
//                     boosted channel) is stored at byte kch_pos(j)
//   Vbase  128*v B    v-bit codes (v = v_bit, 2 or 4), 32 tokens x D channels
//   VS     256 B      fp16 step per (group, token), at vmeta_pos(G, t)
//   VM     256 B      fp16 minimum per (group, token), at vmeta_pos(G, t)
struct Layout {
  int n_hi, w, vw;
  size_t kbase, kextra, ks, km, kch, vbase, vs, vm, bytes;
  Layout(int nh, int w_, int vw_) : n_hi(nh), w(w_), vw(vw_) {
    kbase = 0;
    kextra = (size_t)D * P * w / 8;
    ks = kextra + (size_t)nh * P * w / 8;
    km = ks + 256;
    kch = km + 256;
    vbase = kch + (size_t)nh;
    vs = vbase + (size_t)P * D * vw_ / 8;
    vm = vs + 256;
    bytes = vm + 256;
  }
};

// Position of one 2-bit code inside a plane: 32-bit little-endian word index
// and bit offset.  Each plane is stored in "fragment order": the 32 bytes (8
// words) of lane L hold exactly the codes that lane L of a 32-thread warp needs
// as 16x16 operand tiles, and inside a word the code of element (row, col) sits
// at bit 16*(col parity) + 8*(col half of the 16-wide tile) + 2*tau + 2,
// modulo 32, where tau names the row's 8-row block.  (Reading: the pages fix
// no bit layout.  The +2 -- every word rotated left by two bits against the
// plain order -- places a code, once masked out of its 16-bit half, in
// mantissa bits 2..9 of an fp16 subnormal rather than 0..7; on the GB300 the
// tensor cores keep measurably less of a product's low bits the further
// below the top of the mantissa its code sits.)  The mapping is a bijection
// (checked by tests).
//
// Key planes: row = token t, col = channel c (base) or boosted row j (extra).
struct BitPos { int word; int bit; };

// The rotation of a plane word's bit positions (see above).
int rot_bit(int b) { return (b + 2) & 31; }

BitPos key_pos(int col, int t, int words_per_lane) {
  const int ks = col >> 4, cc = col & 15;
  const int half = cc >> 3, qq = (cc & 7) >> 1, e = cc & 1;
  const int mt = t >> 4, rh = (t >> 3) & 1, r = t & 7;
  const int tau = 2 * mt + rh;
  const int lane = 4 * r + qq;
  return {lane * words_per_lane + ks, rot_bit(16 * e + 8 * half + 2 * tau)};
}

// 4-bit Key planes, same fragment order with nibbles: a lane holds two words
// per 16-column tile (one per 16-token block mt), and inside a word element
// (row, col) sits at bit 16*(col parity) + 8*(col half) + 4*(row's 8-row half)
// + 2, modulo 32 (a nibble may wrap from bit 31 to bit 0).
// words_per_lane = 2 * (columns / 16).
BitPos key_pos4(int col, int t, int words_per_lane) {
  const int ks = col >> 4, cc = col & 15;
  const int half = cc >> 3, qq = (cc & 7) >> 1, e = cc & 1;
  const int mt = t >> 4, rh = (t >> 3) & 1, r = t & 7;
  const int lane = 4 * r + qq;
  return {lane * words_per_lane + 2 * ks + mt, rot_bit(16 * e + 8 * half + 4 * rh)};
}

// Key code position for plane width w over `cols` columns (D or n_hi).
BitPos kpos(int w, int col, int t, int cols) {
  return w == 4 ? key_pos4(col, t, 2 * (cols / 16)) : key_pos(col, t, cols / 16);
}

// Value plane: row = channel c, col = token t (the transposed operand).
BitPos val_pos(int t, int c) {
  const int mc = c >> 4, rh = (c >> 3) & 1, r = c & 7;
  const int kt = t >> 4, half = (t >> 3) & 1, qq = (t & 7) >> 1, e = t & 1;
  const int tau = 2 * (mc & 1) + rh;
  const int lane = 4 * r + qq;
  return {lane * 8 + (mc >> 1) * 2 + kt, rot_bit(16 * e + 8 * half + 2 * tau)};
}

// 4-bit Value plane, same rows and columns with nibbles: a lane holds four
// words per 32-channel group G (16-token block kt, 16-channel tile parity), and
// inside a word element (row, col) sits at bit 16*(col parity) + 8*(col half) +
// 4*(row's 8-row half) + 2, modulo 32.
BitPos val_pos4(int t, int c) {
  const int mc = c >> 4, rh = (c >> 3) & 1, r = c & 7;
  const int kt = t >> 4, half = (t >> 3) & 1, qq = (t & 7) >> 1, e = t & 1;
  const int lane = 4 * r + qq;
  return {lane * 16 + (mc >> 1) * 4 + kt * 2 + (mc & 1), rot_bit(16 * e + 8 * half + 4 * rh)};
}

// Value code position for Value width vw.
BitPos vpos(int vw, int t, int c) { return vw == 4 ? val_pos4(t, c) : val_pos(t, c); }

// Metadata read by the decode in 16-byte pieces is stored in the same
// "fragment order" as the planes: the values lane group qq = (index % 8) / 2
// needs are contiguous.
//  km_pos(c):   channel c = 16j + 8h + 2qq + e  ->  ((qq*8 + j)*2 + h)*2 + e
int km_pos(int c) {
  const int j = c >> 4, h = (c >> 3) & 1, qq = (c >> 1) & 3, e = c & 1;
  return ((qq * 8 + j) * 2 + h) * 2 + e;
}
//  vmeta_pos(G, t): token t = 16kt + 8h + 2qq + e  ->  G*32 + qq*8 + kt*4 + h*2 + e
int vmeta_pos(int G, int t) {
  const int kt = t >> 4, h = (t >> 3) & 1, qq = (t >> 1) & 3, e = t & 1;
  return G * 32 + qq * 8 + kt * 4 + h * 2 + e;
}
//  kch_pos(j):  row j = 16js + 8h + 2qq + e  ->  js*16 + qq*4 + h*2 + e
int kch_pos(int j) {
  const int js = j >> 4, h = (j >> 3) & 1, qq = (j >> 1) & 3, e = j & 1;
  return js * 16 + qq * 4 + h * 2 + e;
}

// Write / read a `bits`-wide code at p; a code starting at bit 30 of a word
// continues at bit 0 of the same word.
uint32_t rotl32(uint32_t x, int k) { return k == 0 ? x : (x << k) | (x >> (32 - k)); }

void putb(uint8_t* plane, BitPos p, uint32_t code, int bits) {
  uint32_t w;
  std::memcpy(&w, plane + 4 * p.word, 4);
  w |= rotl32(code & ((1u << bits) - 1u), p.bit);
  std::memcpy(plane + 4 * p.word, &w, 4);
}

uint32_t getb(const uint8_t* plane, BitPos p, int bits) {
  uint32_t w;
  std::memcpy(&w, plane + 4 * p.word, 4);
  return rotl32(w, (32 - p.bit) & 31) & ((1u << bits) - 1u);
}


uint16_t rd16(const uint8_t* p, size_t i) { uint16_t v; std::memcpy(&v, p + 2 * i, 2); return v; }
void wr16(uint8_t* p, size_t i, uint16_t v) { std::memcpy(p + 2 * i, &v, 2); }

}  // namespace

// ---------------------------------------------------------------- status codes
// Same numbering as the library's public header; defined here on their own.
namespace {
constexpr int ST_OK = 0, ST_EMPTY = 1, ST_RANGE = 2, ST_NONFINITE = 3, ST_BAD_PAGE = 4,
              ST_BAD_LEN = 5, ST_TAIL_FULL = 6, ST_BAD_FLUSH = 7, ST_TABLE_FULL = 8,
              ST_BAD_SEQ = 9;

void note(int* st, int code) { if (*st == ST_OK) *st = code; }

int g_threads = 1;

// Run f(i) for i in [0, n) on g_threads std::threads (static interleaved split).
template <class F>
void parallel_for(int n, F f) {
  const int nt = std::max(1, std::min(g_threads, n));
  if (nt == 1) { for (int i = 0; i < n; ++i) f(i); return; }
  std::vector<std::thread> ts;
  for (int w = 0; w < nt; ++w)
    ts.emplace_back([=]() { for (int i = w; i < n; i += nt) f(i); });
  for (auto& t : ts) t.join();
}

// ---------------------------------------------------------------- statistics
// Pairwise tree sum of 32 fp32 values: fold the upper half onto the lower half
// 16, 8, 4, 2, 1 apart.  The pages fix no summation order; this one is chosen
// and stated so that a GPU warp reduction can reproduce it bit for bit.
float tree_sum(const float* x) {
  float a[32];
  for (int i = 0; i < 32; ++i) a[i] = x[i];
  for (int w = 16; w >= 1; w >>= 1)
    for (int i = 0; i < w; ++i) a[i] = a[i] + a[i + w];
  return a[0];
}

struct PageStats { float mn[D], mx[D], s1[D], s2[D]; };

// Minimum and maximum of a group of values.  The pages say "min/max" and no
// more; of two zeros, -0 is taken as the smaller (IEEE 754-2019 minimum and
// maximum), so the result does not depend on the order of the values.  Inputs
// are finite (others are reported, and their pages are not defined).
float min_of(float a, float b) {
  if (a == b) return std::signbit(a) ? a : b;
  return b < a ? b : a;
}
float max_of(float a, float b) {
  if (a == b) return std::signbit(a) ? b : a;
  return b > a ? b : a;
}

// Per channel over the 32 tokens of one Key page: min, max, sum and sum of
// squares (VeloxQuant-MLX docs, Prefill phase step 1 and step 5).
void page_stats(const float* xk, PageStats& st) {
  for (int c = 0; c < D; ++c) {
    float col[P], sq[P];
    float mn = xk[c], mx = xk[c];
    for (int t = 0; t < P; ++t) {
      const float x = xk[t * D + c];
      col[t] = x;
      sq[t] = x * x;
      mn = min_of(mn, x);
      mx = max_of(mx, x);
    }
    st.mn[c] = mn;
    st.mx[c] = mx;
    st.s1[c] = tree_sum(col);
    st.s2[c] = tree_sum(sq);
  }
}

// Running-variance estimate sigma^2 = (sum k^2)/n - ((sum k)/n)^2
// (VeloxQuant-MLX docs, Decode phase step 2), three divisions/products and one
// subtraction, each rounded once.
float variance(float sum, float sumsq, float n) {
  const float a = sumsq / n;
  const float b = sum / n;
  const float bb = b * b;
  return a - bb;
}

// Top-k boost set (VeloxQuant-MLX docs, Prefill phase step 2): the n_hi
// channels of largest variance; among equal variances the lower channel index
// ranks first (reading).  rank_c counts the channels that beat channel c.
void top_k(const float* var, int n_hi, bool* boosted) {
  for (int c = 0; c < D; ++c) {
    int rank = 0;
    for (int o = 0; o < D; ++o)
      if (var[o] > var[c] || (var[o] == var[c] && o < c)) ++rank;
    boosted[c] = rank < n_hi;
  }
}

// Stored step of a group: the smallest fp16 value that is >= s and whose
// significand has at most 7 bits (s >= 0).  First s is rounded up to 7
// significant bits (s = m * 2^e with m in [1/2, 1): ceil(m * 2^7) / 2^7 * 2^e),
// then up to the fp16 grid, which changes it only below the fp16 normal range.
// Reading: the pages fix neither the precision of the metadata nor its
// rounding.  Seven bits let a 4-bit half of a query or probability multiply the
// step exactly in fp16 (4 + 7 = 11 significant bits); rounding up keeps the
// step >= (max - min) / levels, so no value lies above the top level.
uint16_t step_f16(float s) {
  if (s == 0.0f) return 0;
  int e = 0;
  const double m = std::frexp((double)s, &e);
  const float v = (float)std::ldexp(std::ceil(std::ldexp(m, 7)), e - 7);
  uint16_t h = f32_to_f16(v);
  if (f16_to_f32(h) < v) ++h;  // positive fp16: the next pattern is the next value up
  return h;
}

// Asymmetric min/max quantization of one group (VeloxQuant-MLX docs, Prefill
// phase step 3).  Readings: the minimum is stored as fp16 (nearest), the step
// as step_f16 above, and the codes are computed against the STORED values, so
// encoder and decoder agree.  The code is the integer nearest to
// (x - M) * (1 / u), each of the subtraction, the reciprocal and the product
// rounded to nearest fp32 (integer ties to even), clamped to [0, 2^b - 1]:
// "round((x - min) / scale)" with the division done as a multiplication by the
// reciprocal of the step, as quantizers are commonly written.  It picks the
// level nearest to the exact quotient except where that quotient lies within
// about 2^-22 (relative) of a halfway point; there, and at exact halfway
// values, the rounding of the reciprocal decides between the two neighbours.  A boosted Key channel (2w-bit code) stores the step of its
// high w-bit plane, F = 2^w times its own step (F = 4 for the (4, 2)
// configuration, 16 for (8, 4)).
void quant_group(const float* x, int stride, int n, float mn, float mx, int levels,
                 bool boosted, uint16_t* S_out, uint16_t* M_out, uint16_t* code, float F = 4.0f) {
  const uint16_t M = f32_to_f16(mn);
  const float Mf = f16_to_f32(M);
  const float r = mx - mn;
  const float s = r / (float)levels;
  uint16_t S;
  float u;
  if (boosted) {
    S = step_f16(F * s);
    u = f16_to_f32(S) * (1.0f / F);
  } else {
    S = step_f16(s);
    u = f16_to_f32(S);
  }
  const float ru = u == 0.0f ? 0.0f : 1.0f / u;
  for (int i = 0; i < n; ++i) {
    if (u == 0.0f) { code[i] = 0; continue; }
    const float d = x[i * stride] - Mf;
    const float y = d * ru;
    float q = std::nearbyint(y);
    if (q < 0.0f) q = 0.0f;
    if (q > (float)levels) q = (float)levels;
    code[i] = (uint16_t)q;
  }
  *S_out = S;
  *M_out = M;
}

// Input range rule: fp16 metadata must hold the values, so |x| <= 65504.
int check_range(const float* x, int n) {
  for (int i = 0; i < n; ++i) {
    if (!std::isfinite(x[i])) return ST_NONFINITE;
    if (std::fabs(x[i]) > 65504.0f) return ST_RANGE;
  }
  return ST_OK;
}

// Encode one (page, kv-head): Key planes with the given boost set, Value
// plane, metadata and channel list, into `blob` (Layout(n_hi, w, vw).bytes bytes).
void encode_blob(const float* xk, const float* xv, const PageStats& st, const bool* boosted,
                 int n_hi, int w, int vw, uint8_t* blob) {
  const Layout lay(n_hi, w, vw);
  std::memset(blob, 0, lay.bytes);
  uint8_t* kbase = blob + lay.kbase;
  uint8_t* kextra = blob + lay.kextra;
  uint8_t* vbase = blob + lay.vbase;
  int row_of[D];
  int j = 0;
  for (int c = 0; c < D; ++c) {
    row_of[c] = -1;
    if (boosted[c]) { blob[lay.kch + kch_pos(j)] = (uint8_t)c; row_of[c] = j++; }
  }
  const int Lw = (1 << w) - 1, Lhi = (1 << (2 * w)) - 1;
  for (int c = 0; c < D; ++c) {
    uint16_t S, M;
    uint16_t code[P];
    const bool b = boosted[c];
    quant_group(xk + c, D, P, st.mn[c], st.mx[c], b ? Lhi : Lw, b, &S, &M, code, (float)(1 << w));
    wr16(blob + lay.ks, c, S);
    wr16(blob + lay.km, km_pos(c), M);
    for (int t = 0; t < P; ++t) {
      if (b) {
        // 2w-bit code = 2^w*hi + lo: hi joins the uniform base plane, lo the
        // extra plane row of this channel (two uniform w-bit tensors).
        putb(kbase, kpos(w, c, t, D), code[t] >> w, w);
        putb(kextra, kpos(w, row_of[c], t, n_hi), code[t] & (uint32_t)Lw, w);
      } else {
        putb(kbase, kpos(w, c, t, D), code[t], w);
      }
    }
  }
  for (int t = 0; t < P; ++t) {
    for (int g = 0; g < D / VG; ++g) {
      const float* x = xv + t * D + g * VG;
      float mn = x[0], mx = x[0];
      for (int i = 1; i < VG; ++i) { mn = min_of(mn, x[i]); mx = max_of(mx, x[i]); }
      uint16_t S, M;
      uint16_t code[VG];
      quant_group(x, 1, VG, mn, mx, (1 << vw) - 1, false, &S, &M, code);
      wr16(blob + lay.vs, vmeta_pos(g, t), S);
      wr16(blob + lay.vm, vmeta_pos(g, t), M);
      for (int i = 0; i < VG; ++i) putb(vbase, vpos(vw, t, g * VG + i), code[i], vw);
    }
  }
}

// Quantize one page-head from fp32 token-major tiles xk, xv [32][D].  In
// running mode the (sequence, head) accumulators are updated with this page's
// sums before it is ranked; in page mode the page ranks on its own 32 tokens.
int quantize_one(const float* xk, const float* xv, int n_hi, int w, int vw, int running,
                 float* rsum, float* rsq, int* rcount, uint8_t* blob) {
  int st = check_range(xk, P * D);
  if (st == ST_OK) st = check_range(xv, P * D);
  PageStats ps;
  page_stats(xk, ps);
  float var[D];
  if (running) {
    *rcount += P;
    const float n = (float)*rcount;
    for (int c = 0; c < D; ++c) {
      rsum[c] = rsum[c] + ps.s1[c];
      rsq[c] = rsq[c] + ps.s2[c];
      var[c] = variance(rsum[c], rsq[c], n);
    }
  } else {
    for (int c = 0; c < D; ++c) var[c] = variance(ps.s1[c], ps.s2[c], (float)P);
  }
  bool boosted[D];
  top_k(var, n_hi, boosted);
  encode_blob(xk, xv, ps, boosted, n_hi, w, vw, blob);
  return st;
}

// Sequence-wide ranking (VeloxQuant-MLX docs, Prefill phase steps 1-3 and 5):
// one boost set per (sequence, head), ranked on the variance over all of the
// sequence's pages, then every page quantized with that set.  The running
// accumulators end with the sequence totals (page sums added in page order).
// xk_pages/xv_pages: the pages' fp32 tiles in order; blobs: one per page.
int quantize_sequence(const std::vector<std::vector<float>>& xk_pages,
                      const std::vector<std::vector<float>>& xv_pages, int n_hi, int w, int vw,
                      float* rsum, float* rsq, int* rcount, const std::vector<uint8_t*>& blobs) {
  int st = ST_OK;
  std::vector<PageStats> ps(xk_pages.size());
  for (size_t p = 0; p < xk_pages.size(); ++p) {
    note(&st, check_range(xk_pages[p].data(), P * D));
    note(&st, check_range(xv_pages[p].data(), P * D));
    page_stats(xk_pages[p].data(), ps[p]);
    *rcount += P;
    for (int c = 0; c < D; ++c) {
      rsum[c] = rsum[c] + ps[p].s1[c];
      rsq[c] = rsq[c] + ps[p].s2[c];
    }
  }
  float var[D];
  const float n = (float)*rcount;
  for (int c = 0; c < D; ++c) var[c] = variance(rsum[c], rsq[c], n);
  bool boosted[D];
  top_k(var, n_hi, boosted);
  for (size_t p = 0; p < xk_pages.size(); ++p)
    encode_blob(xk_pages[p].data(), xv_pages[p].data(), ps[p], boosted, n_hi, w, vw, blobs[p]);
  return st;
}

}  // namespace

// ---------------------------------------------------------------- decode side
namespace {

// Dequantize one page-head in fp64: k = M + S*hi + [boosted]*(S/2^w)*lo and
// v = M + S*code, per the page format above.  Returns ST_BAD_PAGE if the
// channel list is not a strictly ascending list of valid channel ids.
int dequant(const uint8_t* blob, int n_hi, int w, int vw, double* kh, double* vh) {
  const Layout lay(n_hi, w, vw);
  int row_of[D];
  for (int c = 0; c < D; ++c) row_of[c] = -1;
  int prev = -1;
  for (int j = 0; j < n_hi; ++j) {
    const int ch = blob[lay.kch + kch_pos(j)];
    if (ch >= D || ch <= prev) return ST_BAD_PAGE;
    row_of[ch] = j;
    prev = ch;
  }
  const double F = (double)(1 << w);
  for (int c = 0; c < D; ++c) {
    const double S = f16_to_f32(rd16(blob + lay.ks, c));
    const double M = f16_to_f32(rd16(blob + lay.km, km_pos(c)));
    for (int t = 0; t < P; ++t) {
      double v = M + S * (double)getb(blob + lay.kbase, kpos(w, c, t, D), w);
      if (row_of[c] >= 0)
        v += (S / F) * (double)getb(blob + lay.kextra, kpos(w, row_of[c], t, n_hi), w);
      kh[t * D + c] = v;
    }
  }
  for (int t = 0; t < P; ++t)
    for (int c = 0; c < D; ++c) {
      const int g = c / VG;
      const double S = f16_to_f32(rd16(blob + lay.vs, vmeta_pos(g, t)));
      const double M = f16_to_f32(rd16(blob + lay.vm, vmeta_pos(g, t)));
      vh[t * D + c] = M + S * (double)getb(blob + lay.vbase, vpos(vw, t, c), vw);
    }
  return ST_OK;
}

struct AttnArgs {
  int Hkv, Hq, n_hi, w, vw, in_dtype;
  const uint16_t* q;
  const uint8_t* pool;
  int pool_pages;
  const int* block_table;
  int max_pages;
  const int* num_pages;
  const uint16_t* tail_k;
  const uint16_t* tail_v;
  const int* tail_len;
  double sm_scale;
};

// Softmax attention of the g query heads of kv head `kvh` of sequence b over
// every cached token: the pages in block-table order, then the unquantized tail
// (readings: no mask; grouped-query heads hq map to kv head hq / g).  fp64
// throughout.  out has g*D entries.
int attend_group(const AttnArgs& a, int b, int kvh, double* out) {
  const int g = a.Hq / a.Hkv;
  const Layout lay(a.n_hi, a.w, a.vw);
  const size_t page_stride = lay.bytes * (size_t)a.Hkv;
  const int np = a.num_pages[b];
  const int tl = a.tail_len[b];
  for (int i = 0; i < g * D; ++i) out[i] = 0.0;
  if (np < 0 || np > a.max_pages || tl < 0 || tl > P) return ST_BAD_LEN;
  const int ntok = np * P + tl;
  if (ntok == 0) return ST_EMPTY;
  std::vector<double> kh((size_t)ntok * D), vh((size_t)ntok * D);
  for (int p = 0; p < np; ++p) {
    const int id = a.block_table[(size_t)b * a.max_pages + p];
    if (id < 0 || id >= a.pool_pages) return ST_BAD_PAGE;
    const uint8_t* blob = a.pool + (size_t)id * page_stride + (size_t)kvh * lay.bytes;
    const int st = dequant(blob, a.n_hi, a.w, a.vw, &kh[(size_t)p * P * D], &vh[(size_t)p * P * D]);
    if (st != ST_OK) return st;
  }
  const size_t tail_base = ((size_t)b * a.Hkv + kvh) * P * D;
  for (int t = 0; t < tl; ++t)
    for (int c = 0; c < D; ++c) {
      kh[(size_t)(np * P + t) * D + c] = in_to_f32(a.tail_k[tail_base + (size_t)t * D + c], a.in_dtype);
      vh[(size_t)(np * P + t) * D + c] = in_to_f32(a.tail_v[tail_base + (size_t)t * D + c], a.in_dtype);
    }
  std::vector<double> s(ntok);
  for (int h = 0; h < g; ++h) {
    const int hq = kvh * g + h;
    double q[D];
    for (int c = 0; c < D; ++c) q[c] = in_to_f32(a.q[((size_t)b * a.Hq + hq) * D + c], a.in_dtype);
    double m = -INFINITY;
    for (int t = 0; t < ntok; ++t) {
      double dot = 0.0;
      for (int c = 0; c < D; ++c) dot += q[c] * kh[(size_t)t * D + c];
      s[t] = a.sm_scale * dot;
      m = std::max(m, s[t]);
    }
    double l = 0.0;
    for (int t = 0; t < ntok; ++t) { s[t] = std::exp(s[t] - m); l += s[t]; }
    for (int c = 0; c < D; ++c) {
      double acc = 0.0;
      for (int t = 0; t < ntok; ++t) acc += s[t] * vh[(size_t)t * D + c];
      out[h * D + c] = acc / l;
    }
  }
  return ST_OK;
}

bool valid_n_hi(int n_hi) { return n_hi >= 0 && n_hi <= D && n_hi % 16 == 0; }
// Key plane width: lo_bit 2 ((hi, lo) = (4, 2)) or 4 ((8, 4)); Value width:
// 2, or 4 with 4-bit Key planes.
bool valid_w(int w, int vw) { return (w == 2 || w == 4) && (vw == 2 || (vw == 4 && w == 4)); }

}  // namespace

// ---------------------------------------------------------------- C entry points
extern "C" {

int orc_abi_version() { return 1; }

void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

// Bytes of one (page, kv-head) blob; -1 for an unsupported n_hi, lo_bit or v_bit.
long orc_page_bytes(int n_hi, int lo_bit, int v_bit) {
  return valid_n_hi(n_hi) && valid_w(lo_bit, v_bit) ? (long)Layout(n_hi, lo_bit, v_bit).bytes : -1;
}

// Effective Key bits per element, codes only (VeloxQuant-MLX docs, Effective
// bit-width): hi_fraction*hi_bit + (1 - hi_fraction)*lo_bit.
double orc_avg_bits(double hi_fraction, int hi_bit, int lo_bit) {
  return hi_fraction * hi_bit + (1.0 - hi_fraction) * lo_bit;
}

uint16_t orc_f32_to_f16(float f) { return f32_to_f16(f); }
uint16_t orc_step_f16(float s) { return step_f16(s); }
float orc_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
float orc_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
float orc_tree_sum(const float* x) { return tree_sum(x); }
float orc_variance(float sum, float sumsq, float n) { return variance(sum, sumsq, n); }

void orc_top_k(const float* var, int n_hi, uint8_t* boosted) {
  bool b[D];
  top_k(var, n_hi, b);
  for (int c = 0; c < D; ++c) boosted[c] = b[c] ? 1 : 0;
}

void orc_key_pos(int col, int t, int words_per_lane, int* word, int* bit) {
  const BitPos p = key_pos(col, t, words_per_lane);
  *word = p.word;
  *bit = p.bit;
}

void orc_key_pos4(int col, int t, int words_per_lane, int* word, int* bit) {
  const BitPos p = key_pos4(col, t, words_per_lane);
  *word = p.word;
  *bit = p.bit;
}

void orc_val_pos(int t, int c, int* word, int* bit) {
  const BitPos p = val_pos(t, c);
  *word = p.word;
  *bit = p.bit;
}

void orc_val_pos4(int t, int c, int* word, int* bit) {
  const BitPos p = val_pos4(t, c);
  *word = p.word;
  *bit = p.bit;
}

// One page-head from fp32 tiles [32][D] (token-major).  running != 0 updates
// rsum/rsq [D] and *rcount before ranking.  Returns a status code.
int orc_quantize_page_f32(const float* xk, const float* xv, int n_hi, int running, float* rsum,
                          float* rsq, int* rcount, uint8_t* blob, int lo_bit, int v_bit) {
  if (!valid_n_hi(n_hi) || !valid_w(lo_bit, v_bit)) return -1;
  return quantize_one(xk, xv, n_hi, lo_bit, v_bit, running, rsum, rsq, rcount, blob);
}

// The boosted channel list of a blob in row order (ascending channel ids).
void orc_page_channels(const uint8_t* blob, int n_hi, int* out, int lo_bit) {
  const Layout lay(n_hi, lo_bit, 2);  // the list precedes the Value plane
  for (int j = 0; j < n_hi; ++j) out[j] = blob[lay.kch + kch_pos(j)];
}

void orc_meta_pos(int kind, int a, int b, int* pos) {
  *pos = kind == 0 ? km_pos(a) : kind == 1 ? vmeta_pos(a, b) : kch_pos(a);
}

void orc_dequant_page(const uint8_t* blob, int n_hi, double* kh, double* vh, int* status,
                      int lo_bit, int v_bit) {
  *status = valid_n_hi(n_hi) && valid_w(lo_bit, v_bit) ? dequant(blob, n_hi, lo_bit, v_bit, kh, vh)
                                                       : -1;
}

// Bulk quantization with the library's semantics.  k, v: [n_pages*32][Hkv][D]
// 16-bit values (in_dtype 0 = fp16, 1 = bf16).  Page i is written at
// pool + page_ids[i]*Hkv*blob.  rank_mode 0 = page, 1 = running, 2 = sequence;
// running and sequence modes need seq_of_page non-decreasing in [0, n_seqs) and
// accumulators run_sum/run_sumsq [n_seqs][Hkv][D], run_count [n_seqs][Hkv].
// Pages whose id is out of range are skipped (not counted, not written).
int orc_quantize_pages(int Hkv, int n_hi, int rank_mode, int in_dtype, const uint16_t* k,
                       const uint16_t* v, int n_pages, const int* page_ids, const int* seq_of_page,
                       int n_seqs, float* run_sum, float* run_sumsq, int* run_count, uint8_t* pool,
                       int pool_pages, int lo_bit, int v_bit) {
  if (!valid_n_hi(n_hi) || !valid_w(lo_bit, v_bit) || Hkv <= 0 || n_pages < 0) return -1;
  const int w = lo_bit, vw = v_bit;
  const Layout lay(n_hi, w, vw);
  const size_t page_stride = lay.bytes * (size_t)Hkv;
  int st = ST_OK;
  if (rank_mode == 1 || rank_mode == 2) {
    for (int i = 0; i < n_pages; ++i) {
      const int s = seq_of_page[i];
      if (s < 0 || s >= n_seqs || (i > 0 && s < seq_of_page[i - 1])) return ST_BAD_SEQ;
    }
  }
  auto tile = [&](int i, int h, std::vector<float>& xk, std::vector<float>& xv) {
    xk.assign(P * D, 0.f);
    xv.assign(P * D, 0.f);
    for (int t = 0; t < P; ++t)
      for (int c = 0; c < D; ++c) {
        const size_t src = (((size_t)i * P + t) * Hkv + h) * D + c;
        xk[t * D + c] = in_to_f32(k[src], in_dtype);
        xv[t * D + c] = in_to_f32(v[src], in_dtype);
      }
  };
  if (rank_mode == 2) {
    std::vector<int> sts2((size_t)Hkv * (n_seqs > 0 ? n_seqs : 1), ST_OK);
    parallel_for(Hkv * n_seqs, [&](int sh) {
      const int h = sh % Hkv, sq = sh / Hkv;
      std::vector<std::vector<float>> xk, xv;
      std::vector<uint8_t*> blobs;
      int bad = ST_OK;
      for (int i = 0; i < n_pages; ++i) {
        if (seq_of_page[i] != sq) continue;
        const int id = page_ids[i];
        if (id < 0 || id >= pool_pages) { bad = ST_BAD_PAGE; continue; }
        xk.emplace_back();
        xv.emplace_back();
        tile(i, h, xk.back(), xv.back());
        blobs.push_back(pool + (size_t)id * page_stride + (size_t)h * lay.bytes);
      }
      if (xk.empty()) { sts2[sh] = bad; return; }
      const size_t o = (size_t)sq * Hkv + h;
      int r = quantize_sequence(xk, xv, n_hi, w, vw, run_sum + o * D, run_sumsq + o * D,
                                run_count + o, blobs);
      sts2[sh] = r != ST_OK ? r : bad;
    });
    for (int x : sts2) note(&st, x);
    return st;
  }
  std::vector<int> sts(n_pages > 0 ? (size_t)n_pages * Hkv : 1, ST_OK);
  auto one = [&](int i, int h) {
    const int id = page_ids[i];
    if (id < 0 || id >= pool_pages) { sts[(size_t)i * Hkv + h] = ST_BAD_PAGE; return; }
    std::vector<float> xk(P * D), xv(P * D);
    for (int t = 0; t < P; ++t)
      for (int c = 0; c < D; ++c) {
        const size_t src = (((size_t)i * P + t) * Hkv + h) * D + c;
        xk[t * D + c] = in_to_f32(k[src], in_dtype);
        xv[t * D + c] = in_to_f32(v[src], in_dtype);
      }
    float* rs = nullptr;
    float* rq = nullptr;
    int* rc = nullptr;
    if (rank_mode == 1) {
      const size_t sh = (size_t)seq_of_page[i] * Hkv + h;
      rs = run_sum + sh * D;
      rq = run_sumsq + sh * D;
      rc = run_count + sh;
    }
    sts[(size_t)i * Hkv + h] = quantize_one(xk.data(), xv.data(), n_hi, w, vw, rank_mode == 1, rs, rq,
                                            rc, pool + (size_t)id * page_stride + (size_t)h * lay.bytes);
  };
  if (rank_mode == 1) {
    // Each head's accumulators see that head's pages strictly in input order.
    parallel_for(Hkv, [&](int h) { for (int i = 0; i < n_pages; ++i) one(i, h); });
  } else {
    parallel_for(n_pages * Hkv, [&](int ih) { one(ih / Hkv, ih % Hkv); });
  }
  for (int x : sts) note(&st, x);
  return st;
}

// Append one token per sequence (VeloxQuant-MLX docs, Decode phase), with the
// reading that a new token waits in an unquantized tail until 32 tokens form a
// page: the token goes to tail[tail_len]; when the tail becomes full and the
// caller named a page id for this sequence, the tail is quantized (running
// statistics updated first in running mode), written at that page id, the id
// is appended to the block table and the tail is emptied.
// k_new, v_new: [B][Hkv][D]; tail_k, tail_v: [B][Hkv][32][D];
// run_sum, run_sumsq: [B][Hkv][D]; run_count: [B][Hkv].
int orc_append_token(int Hkv, int n_hi, int rank_mode, int in_dtype, const uint16_t* k_new,
                     const uint16_t* v_new, uint16_t* tail_k, uint16_t* tail_v, int* tail_len,
                     float* run_sum, float* run_sumsq, int* run_count, const int* flush_page_ids,
                     int* block_table, int max_pages, int* num_pages, uint8_t* pool, int pool_pages,
                     int B, int lo_bit, int v_bit) {
  if (!valid_n_hi(n_hi) || !valid_w(lo_bit, v_bit) || Hkv <= 0 || B < 0) return -1;
  const Layout lay(n_hi, lo_bit, v_bit);
  const size_t page_stride = lay.bytes * (size_t)Hkv;
  std::vector<int> sts(B > 0 ? B : 1, ST_OK);
  parallel_for(B, [&](int b) {
    const int len = tail_len[b];
    if (len < 0 || len > P) { sts[b] = ST_BAD_LEN; return; }
    if (len == P) { sts[b] = ST_TAIL_FULL; return; }
    for (int h = 0; h < Hkv; ++h) {
      const size_t dst = (((size_t)b * Hkv + h) * P + len) * D;
      const size_t src = ((size_t)b * Hkv + h) * D;
      for (int c = 0; c < D; ++c) {
        tail_k[dst + c] = k_new[src + c];
        tail_v[dst + c] = v_new[src + c];
      }
    }
    const int n = len + 1;
    const int fid = flush_page_ids[b];
    if (fid >= 0 && n < P) { sts[b] = ST_BAD_FLUSH; tail_len[b] = n; return; }
    if (n < P || fid < 0) { tail_len[b] = n; return; }
    const int np = num_pages[b];
    if (np < 0 || np >= max_pages) { sts[b] = ST_TABLE_FULL; tail_len[b] = n; return; }
    if (fid >= pool_pages) { sts[b] = ST_BAD_PAGE; tail_len[b] = n; return; }
    int st = ST_OK;
    for (int h = 0; h < Hkv; ++h) {
      std::vector<float> xk(P * D), xv(P * D);
      const size_t base = ((size_t)b * Hkv + h) * P * D;
      for (int i = 0; i < P * D; ++i) {
        xk[i] = in_to_f32(tail_k[base + i], in_dtype);
        xv[i] = in_to_f32(tail_v[base + i], in_dtype);
      }
      const size_t sh = (size_t)b * Hkv + h;
      const bool running = rank_mode != 0;  // sequence mode continues with running statistics
      note(&st, quantize_one(xk.data(), xv.data(), n_hi, lo_bit, v_bit, running,
                             running ? run_sum + sh * D : nullptr,
                             running ? run_sumsq + sh * D : nullptr, running ? run_count + sh : nullptr,
                             pool + (size_t)fid * page_stride + (size_t)h * lay.bytes));
    }
    block_table[(size_t)b * max_pages + np] = fid;
    num_pages[b] = np + 1;
    tail_len[b] = 0;
    sts[b] = st;
  });
  int st = ST_OK;
  for (int x : sts) note(&st, x);
  return st;
}

// fp64 decode attention for every (sequence, query head); out: [B][Hq][D].
// sm_scale multiplies q.k (callers pass 1/sqrt(D) unless they want another).
int orc_decode_attention(int Hkv, int Hq, int n_hi, int in_dtype, const uint16_t* q,
                         const uint8_t* pool, int pool_pages, const int* block_table, int max_pages,
                         const int* num_pages, const uint16_t* tail_k, const uint16_t* tail_v,
                         const int* tail_len, float sm_scale, int B, double* out, int lo_bit,
                         int v_bit) {
  if (!valid_n_hi(n_hi) || !valid_w(lo_bit, v_bit) || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || B < 0)
    return -1;
  const AttnArgs a{Hkv, Hq, n_hi, lo_bit, v_bit, in_dtype, q, pool, pool_pages, block_table,
                   max_pages, num_pages, tail_k, tail_v, tail_len, (double)sm_scale};
  const int g = Hq / Hkv;
  std::vector<int> sts(B > 0 ? (size_t)B * Hkv : 1, ST_OK);
  parallel_for(B * Hkv, [&](int i) {
    const int b = i / Hkv, kvh = i % Hkv;
    sts[i] = attend_group(a, b, kvh, out + ((size_t)b * Hq + (size_t)kvh * g) * D);
  });
  int st = ST_OK;
  for (int x : sts) note(&st, x);
  return st;
}

// 16-bit paged KV baseline (the unquantized layout Kitty is compared against on
// one memory budget; paper: Abstract).  A (page, kv head) blob holds K [32][D]
// then V [32][D] in the input dtype; sequence b holds ctx_len[b] tokens, token
// t in slot t % 32 of page block_table[b][t / 32].  fp64 attention with no
// quantization: out[b][hq] = softmax_t(sm_scale * q.k_t) . v_t, query head hq
// reading kv head hq / (Hq / Hkv); an empty sequence gives 0 and ST_EMPTY.
int orc_decode_f16kv(int Hkv, int Hq, int in_dtype, const uint16_t* q, const uint16_t* pool,
                     int pool_pages, const int* block_table, int max_pages, const int* ctx_len,
                     float sm_scale, int B, double* out) {
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || B < 0) return -1;
  const int g = Hq / Hkv;
  const size_t blob = 2 * (size_t)P * D;  // 16-bit elements per (page, kv head)
  std::vector<int> sts(B > 0 ? (size_t)B * Hkv : 1, ST_OK);
  parallel_for(B * Hkv, [&](int i) {
    const int b = i / Hkv, kvh = i % Hkv;
    const int len = ctx_len[b];
    double* o = out + ((size_t)b * Hq + (size_t)kvh * g) * D;
    if (len < 0 || len > max_pages * P) { sts[i] = ST_BAD_LEN; return; }
    std::vector<const uint16_t*> krow(len), vrow(len);
    for (int t = 0; t < len; ++t) {
      const int pid = block_table[(size_t)b * max_pages + t / P];
      if (pid < 0 || pid >= pool_pages) { sts[i] = ST_BAD_PAGE; return; }
      const uint16_t* base = pool + ((size_t)pid * Hkv + kvh) * blob;
      krow[t] = base + (size_t)(t % P) * D;
      vrow[t] = base + (size_t)(P + t % P) * D;
    }
    for (int h = 0; h < g; ++h) {
      const uint16_t* qh = q + ((size_t)b * Hq + (size_t)kvh * g + h) * D;
      double* oh = o + (size_t)h * D;
      for (int c = 0; c < D; ++c) oh[c] = 0.0;
      if (len == 0) { sts[i] = ST_EMPTY; continue; }
      std::vector<double> sc(len);
      double mx = -INFINITY;
      for (int t = 0; t < len; ++t) {
        double acc = 0.0;
        for (int c = 0; c < D; ++c)
          acc += (double)in_to_f32(qh[c], in_dtype) * (double)in_to_f32(krow[t][c], in_dtype);
        sc[t] = acc * (double)sm_scale;
        mx = std::max(mx, sc[t]);
      }
      double den = 0.0;
      for (int t = 0; t < len; ++t) {
        sc[t] = std::exp(sc[t] - mx);
        den += sc[t];
      }
      for (int t = 0; t < len; ++t)
        for (int c = 0; c < D; ++c) oh[c] += sc[t] / den * (double)in_to_f32(vrow[t][c], in_dtype);
    }
  });
  int st = ST_OK;
  for (int x : sts) note(&st, x);
  return st;
}

// The g query heads of one (sequence, kv head) only; out: [g][D].  For sampled
// checks on workloads too large to run whole.
int orc_decode_attention_one(int Hkv, int Hq, int n_hi, int in_dtype, const uint16_t* q,
                             const uint8_t* pool, int pool_pages, const int* block_table,
                             int max_pages, const int* num_pages, const uint16_t* tail_k,
                             const uint16_t* tail_v, const int* tail_len, float sm_scale, int b,
                             int kvh, double* out, int lo_bit, int v_bit) {
  if (!valid_n_hi(n_hi) || !valid_w(lo_bit, v_bit) || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return -1;
  const AttnArgs a{Hkv, Hq, n_hi, lo_bit, v_bit, in_dtype, q, pool, pool_pages, block_table,
                   max_pages, num_pages, tail_k, tail_v, tail_len, (double)sm_scale};
  return attend_group(a, b, kvh, out);
}

}  // extern "C"
