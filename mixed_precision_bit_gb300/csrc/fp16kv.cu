// 16-bit paged KV cache: the unquantized layout that Kitty's memory budget and
// throughput are compared against (paper: Abstract, "up to 8x larger batches
// and 2.1x-4.1x higher throughput under the same memory budget").  Keys and
// Values are kept in the input dtype (fp16 or bf16), 32 tokens per page.
//
// Page blob of one (page, kv head): K [32 tokens][128] then V [32][128], 16-bit,
// 16 KB; a page holds Hkv blobs in head order.  A sequence of L tokens uses
// pages block_table[b][0 .. ceil(L / 32)); token t sits in slot t % 32 of page
// t / 32 (there is no separate tail).
//
// Decode: one CTA per (sequence, kv head, split), 4 warps, each warp streaming
// every 4th half page (16 tokens) of the split, two CTAs per SM.  A warp stages
// a half page's 32 rows (16 Key, 16 Value) with one 256-byte bulk copy per
// lane into rows padded to 272 bytes (conflict-free ldmatrix), then
//   scores  S[t][n] = sum_c K[t][c] q[c][n] on the tensor cores (K from
//           ldmatrix, B = the query of head n/2; the two columns of a head
//           carry the same score),
//   softmax fp32 online, and
//   PV      O^T[c][n] = sum_t V[t][c] P[t][n], V^T from transposing ldmatrix,
//           P as a (high, rest) pair in the 16-bit type per head.
// Splits are merged by a second kernel in split order.
#include "kitty_common.cuh"
#include "host_common.h"

#include <algorithm>
#include <atomic>

namespace kitty {
namespace {

constexpr int kFWarps = 4;
constexpr int kFBlocks = 2;                   // resident CTAs per SM
constexpr int kFStages = 3;                   // staged half pages per warp
constexpr int kHalf = kPage / 2;              // tokens per work item
constexpr int kRowB = kD * 2;                 // bytes of one token row
constexpr int kRowPad = kRowB + 16;           // staged row stride
constexpr int kFBlob = 2 * kPage * kRowB;     // 16384: K then V of one (page, kv head)
constexpr int kFStage = 2 * kHalf * kRowPad;  // 8704: one staged half page (K rows, V rows)
constexpr int kFPartial = kD + 4;             // split partial: m, l, 2 unused, o[128]
constexpr uint32_t kFWaitLimit = 1u << 22;
constexpr int kFMaxSplits = 64;

struct F16Params {
  const uint16_t* q;
  const uint8_t* pool;
  const int32_t* block_table;
  const int32_t* ctx_len;
  void* out;
  float* ws;
  int32_t* d_status;
  float sm_log2;
  int pool_pages, max_pages, out_dtype, splits, pps, Hkv, Hq, g;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void store_o(void* out, int dt, size_t i, float v) {
  if (dt == KITTY_F32) static_cast<float*>(out)[i] = v;
  else if (dt == KITTY_BF16) static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else static_cast<__half*>(out)[i] = __float2half_rn(v);
}

template <int DT>
__global__ void __launch_bounds__(kFWarps * 32, kFBlocks) f16kv_decode_kernel(const F16Params p) {
  extern __shared__ __align__(128) uint8_t fsm[];
  const int u = blockIdx.x, s = blockIdx.y;
  const int b = u / p.Hkv, kvh = u - b * p.Hkv;
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qq = lane & 3;
  int len = p.ctx_len[b];
  if (len < 0 || len > p.max_pages * kPage) {
    if (tid == 0 && s == 0 && kvh == 0) set_status(p.d_status, KITTY_ST_BAD_LEN);
    len = 0;
  }
  const int np = (len + kPage - 1) / kPage;
  const int pbeg = s * p.pps, pend = min(np, pbeg + p.pps);
  const size_t row0 = (size_t)b * p.Hq + (size_t)kvh * p.g;
  if (pbeg >= pend && s > 0) {  // no pages here: an empty partial
    if (tid < p.g) p.ws[((row0 + tid) * p.splits + s) * kFPartial] = -INFINITY;
    return;
  }
  uint8_t* stages = fsm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(fsm + kFWarps * kFStages * kFStage);
  uint16_t* qsm = reinterpret_cast<uint16_t*>(bars + kFWarps * kFStages);  // [4][128]
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint16_t v = 0;
    if (h < p.g) {
      v = p.q[(row0 + h) * kD + tid];
      const uint32_t m = v & 0x7FFFu;
      if (s == 0 && m >= (DT == KITTY_BF16 ? 0x7F80u : 0x7C00u))
        set_status(p.d_status, KITTY_ST_NONFINITE);
    }
    qsm[h * kD + tid] = v;
  }
  // work items are half pages: item x = (page x / 2, tokens 16 (x % 2) .. + 15)
  const int first = 2 * pbeg + wid;
  const int npw = 2 * pend > first ? (2 * pend - first + kFWarps - 1) / kFWarps : 0;
  uint8_t* wst = stages + (size_t)wid * kFStages * kFStage;
  uint64_t* wbar = bars + wid * kFStages;
  if (lane == 0) {
    for (int st = 0; st < kFStages; ++st) mbar_init(&wbar[st], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages;
  const size_t page_stride = (size_t)p.Hkv * kFBlob;
  const uint8_t* head_base = p.pool + (size_t)kvh * kFBlob;
  const uint32_t stage0 = smem_u32(wst), bar0 = smem_u32(wbar);
  uint32_t valid = 0;  // bit st: stage st holds a valid page
  // item i of this warp into stage i % kFStages: lane l < 16 copies Key row l of
  // the half page, lane 16 + l its Value row l
  auto issue = [&](int i) {
    const int x = first + i * kFWarps;
    const int pid = bt[x >> 1];
    const int st = i % kFStages;
    const bool ok = pid >= 0 && pid < p.pool_pages;
    const uint32_t bar = bar0 + 8 * st;
    if (ok) {
      if (lane == 0) mbar_arrive_expect_tx_s(bar, (uint32_t)(2 * kHalf * kRowB));
      __syncwarp();
      const int row = (lane >> 4) * kPage + (x & 1) * kHalf + (lane & 15);  // row of the blob
      bulk_g2s_s(stage0 + st * kFStage + lane * kRowPad,
                 head_base + (size_t)pid * page_stride + (size_t)row * kRowB, (uint32_t)kRowB, bar);
      valid |= 1u << st;
    } else {
      if (lane == 0) {
        set_status(p.d_status, KITTY_ST_BAD_PAGE);
        mbar_arrive_s(bar);
      }
      valid &= ~(1u << st);
    }
  };
  const int pro = min(npw, kFStages);
  for (int i = 0; i < pro; ++i) issue(i);

  // query B fragments: column n = lane/4 holds head n/2 (both columns of a head)
  uint32_t qf[8][2];
  {
    const uint16_t* qh = qsm + (lane >> 3) * kD;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qf[j][0] = *reinterpret_cast<const uint32_t*>(qh + 16 * j + 2 * qq);
      qf[j][1] = *reinterpret_cast<const uint32_t*>(qh + 16 * j + 2 * qq + 8);
    }
  }
  float acc[8][4];
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mc][i] = 0.f;
  float m = -1.0e30f, l = 0.f;
  bool timed_out = false;
  const int mtx = lane >> 3, mrow = lane & 7;  // ldmatrix: this lane's matrix and row
  for (int i = 0; i < npw; ++i) {
    const int st = i % kFStages;
    bool done = false;
    for (uint32_t it = 0;; ++it) {
      done = done || mbar_test_s(bar0 + 8 * st, (uint32_t)(i / kFStages) & 1u);
      if (__all_sync(0xFFFFFFFFu, done) || it >= kFWaitLimit) break;
      if (it > 64) __nanosleep(32);
    }
    if (!__all_sync(0xFFFFFFFFu, done)) {
      timed_out = true;
      if (lane == 0) {
        set_status(p.d_status, KITTY_ST_TIMEOUT);
        for (int k = i; k < min(npw, i + kFStages); ++k)
          mbar_wait_bounded(&wbar[k % kFStages], (uint32_t)(k / kFStages) & 1u, kFWaitLimit);
      }
      __syncwarp();
      break;
    }
    const int x = first + i * kFWarps;
    const int nvalid = ((valid >> st) & 1u) ? min(kHalf, len - x * kHalf) : 0;
    if (nvalid <= 0) {  // a bad page id, or past the sequence's end (warp-uniform)
      __syncwarp();
      if (i + kFStages < npw) issue(i + kFStages);
      continue;
    }
    const uint32_t sk = stage0 + st * kFStage, sv = sk + kHalf * kRowPad;
    // ---- scores of the 16 tokens
    float cs[4] = {};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t a[4];
      ldsm_x4(sk + ((mtx & 1) * 8 + mrow) * kRowPad + (16 * j + (mtx >> 1) * 8) * 2, a);
      mma16<DT>(cs, a, qf[j][0], qf[j][1]);
    }
    float sc[2];
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) sc[rh] = 8 * rh + r < nvalid ? cs[2 * rh] * p.sm_log2 : -INFINITY;
    // ---- online softmax (head qq over the 8 lanes of its column)
    float pm = fmaxf(sc[0], sc[1]);
    pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
    const float nm = fmaxf(m, pm);
    if (__any_sync(0xFFFFFFFFu, nm > m)) {
      const float a = ex2f(m - nm);
#pragma unroll
      for (int mc = 0; mc < 8; ++mc)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[mc][k] *= a;
      l *= a;
      m = nm;
    }
    uint32_t T[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float pr = ex2f(sc[k] - m);
      l += pr;
      T[k] = movmatrix_t(prob_pair<DT>(pr));
    }
    // ---- PV: A = V^T (channels x tokens) by transposing ldmatrix
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      uint32_t a[4];
      ldsm_x4_t(sv + ((mtx >> 1) * 8 + mrow) * kRowPad + (16 * mc + (mtx & 1) * 8) * 2, a);
      mma16<DT>(acc[mc], a, T[0], T[1]);
    }
    __syncwarp();
    if (i + kFStages < npw) issue(i + kFStages);
  }
  (void)timed_out;
  // ---- merge the 4 warps through shared memory (the stage buffers are idle now)
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 4);
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
  __syncthreads();
  float* mw = reinterpret_cast<float*>(fsm) + wid * (kD * 4 + 8);  // O[128][4], m[4], l[4]
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh)
      mw[(16 * mc + 8 * rh + r) * 4 + qq] = acc[mc][2 * rh] + acc[mc][2 * rh + 1];
  if (r == 0) {
    mw[kD * 4 + qq] = m;
    mw[kD * 4 + 4 + qq] = l;
  }
  __syncthreads();
  const int c = tid;
  const float* m0 = reinterpret_cast<const float*>(fsm);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    if (h >= p.g) break;
    float ms = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kFWarps; ++ww) ms = fmaxf(ms, m0[ww * (kD * 4 + 8) + kD * 4 + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int ww = 0; ww < kFWarps; ++ww) {
      const float* base = m0 + ww * (kD * 4 + 8);
      const float mm = base[kD * 4 + h];
      const float e = (ms == -INFINITY || mm == -INFINITY) ? 0.f : ex2f(mm - ms);
      L += base[kD * 4 + 4 + h] * e;
      O += base[c * 4 + h] * e;
    }
    const size_t row = row0 + h;
    if (p.splits == 1) {
      store_o(p.out, p.out_dtype, row * kD + c, L > 0.f ? O / L : 0.f);
      if (c == 0 && !(L > 0.f)) set_status(p.d_status, KITTY_ST_EMPTY);
    } else {
      float* part = p.ws + (row * p.splits + s) * kFPartial;
      part[4 + c] = O;
      if (c == 0) { part[0] = L > 0.f ? ms : -INFINITY; part[1] = L; }
    }
  }
}

// Split merge: one 128-thread CTA per (sequence, query head), splits in order.
__global__ void __launch_bounds__(128) f16kv_combine_kernel(const F16Params p) {
  const size_t row = blockIdx.x;
  const int c = threadIdx.x;
  const float* base = p.ws + row * p.splits * kFPartial;
  float ms = -INFINITY;
  for (int s = 0; s < p.splits; ++s) ms = fmaxf(ms, base[s * kFPartial]);
  float L = 0.f, O = 0.f;
  if (ms != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float m = base[s * kFPartial];
      if (m == -INFINITY) continue;
      const float e = ex2f(m - ms);
      L += base[s * kFPartial + 1] * e;
      O += base[s * kFPartial + 4 + c] * e;
    }
  }
  store_o(p.out, p.out_dtype, row * kD + c, L > 0.f ? O / L : 0.f);
  if (c == 0 && !(L > 0.f)) set_status(p.d_status, KITTY_ST_EMPTY);
}

// Copy full pages of token-major K, V [n_pages*32][Hkv][128] into the pool:
// one CTA per (input page, kv head), 16-byte loads and stores.
__global__ void __launch_bounds__(128) f16kv_write_kernel(const uint16_t* __restrict__ k,
                                                          const uint16_t* __restrict__ v,
                                                          const int32_t* page_ids, int Hkv,
                                                          uint8_t* pool, int pool_pages,
                                                          int32_t* d_status) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int pid = page_ids[i];
  if (pid < 0 || pid >= pool_pages) {
    if (threadIdx.x == 0) set_status(d_status, KITTY_ST_BAD_PAGE);
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(pool + ((size_t)pid * Hkv + h) * kFBlob);
  for (int e = threadIdx.x; e < 2 * kPage * (kD / 8); e += 128) {
    const int kv = e / (kPage * (kD / 8)), rem = e - kv * kPage * (kD / 8);
    const int t = rem / (kD / 8), ch = (rem % (kD / 8)) * 8;
    const uint16_t* src = (kv ? v : k) + ((size_t)(i * kPage + t) * Hkv + h) * kD + ch;
    dst[e] = *reinterpret_cast<const uint4*>(src);
  }
}

// Append one token per sequence: token len goes to slot len % 32 of page
// len / 32; a token that starts a page takes new_page_ids[b] (the caller's
// allocation), which is stored in the block table.  One CTA per (sequence, kv
// head), one thread per channel.  Lengths are advanced afterwards.
__global__ void __launch_bounds__(128) f16kv_append_kernel(const uint16_t* __restrict__ k_new,
                                                           const uint16_t* __restrict__ v_new,
                                                           uint8_t* pool, int pool_pages,
                                                           const int32_t* block_table,
                                                           int max_pages, const int32_t* ctx_len,
                                                           const int32_t* new_page_ids, int Hkv,
                                                           int32_t* d_status) {
  const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int len = ctx_len[b];
  if (len < 0 || len >= max_pages * kPage) {
    if (c == 0) set_status(d_status, len < 0 ? KITTY_ST_BAD_LEN : KITTY_ST_TABLE_FULL);
    return;
  }
  const int slot = len % kPage, pidx = len / kPage;
  const int pid = slot == 0 ? new_page_ids[b] : block_table[(size_t)b * max_pages + pidx];
  if (pid < 0 || pid >= pool_pages) {
    if (c == 0) set_status(d_status, KITTY_ST_BAD_PAGE);
    return;
  }
  uint16_t* blob = reinterpret_cast<uint16_t*>(pool + ((size_t)pid * Hkv + h) * kFBlob);
  const size_t sh = (size_t)b * Hkv + h;
  blob[slot * kD + c] = k_new[sh * kD + c];
  blob[(kPage + slot) * kD + c] = v_new[sh * kD + c];
}

__global__ void f16kv_append_finalize(int32_t* block_table, int max_pages, int32_t* ctx_len,
                                      const int32_t* new_page_ids, int pool_pages, int B) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int len = ctx_len[b];
  if (len < 0 || len >= max_pages * kPage) return;
  if (len % kPage == 0) {
    const int pid = new_page_ids[b];
    if (pid < 0 || pid >= pool_pages) return;
    block_table[(size_t)b * max_pages + len / kPage] = pid;
  }
  ctx_len[b] = len + 1;
}

size_t f16kv_smem() {
  return (size_t)kFWarps * kFStages * kFStage + kFWarps * kFStages * sizeof(uint64_t) + 4 * kD * 2;
}

// Equal splits: enough CTAs for about four waves at kFBlocks CTAs per SM, at
// least 8 pages a split, at most kFMaxSplits splits.
void f16kv_plan(int units, int max_pages, int* splits, int* pps) {
  if (max_pages <= 0) { *splits = 1; *pps = 1; return; }
  const int want = std::max(1, (4 * kFBlocks * sm_count() + units - 1) / std::max(units, 1));
  int sp = std::min({want, kFMaxSplits, std::max(1, max_pages / 8)});
  const int c = (max_pages + sp - 1) / sp;
  *pps = c;
  *splits = (max_pages + c - 1) / c;
}

template <int DT>
cudaError_t launch_f16kv(dim3 grid, cudaStream_t s, const F16Params& p) {
  static std::atomic<uint64_t> opted_in{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  const size_t smem = f16kv_smem();
  if (bit == 0 || (opted_in.load() & bit) == 0) {
    cudaError_t e = cudaFuncSetAttribute(f16kv_decode_kernel<DT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit);
  }
  f16kv_decode_kernel<DT><<<grid, kFWarps * 32, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace kitty

using namespace kitty;

extern "C" int kitty_f16kv_page_bytes(const kitty_cfg* cfg, size_t* per_head_blob,
                                      size_t* per_page) {
  const int rc = check_cfg(cfg);
  if (rc != KITTY_OK) return rc;
  if (per_head_blob) *per_head_blob = kFBlob;
  if (per_page) *per_page = (size_t)kFBlob * cfg->num_kv_heads;
  return KITTY_OK;
}

extern "C" int kitty_f16kv_write_pages(const kitty_cfg* cfg, const void* k, const void* v,
                                       int32_t n_pages, const int32_t* page_ids, void* pool,
                                       int32_t pool_pages, int32_t* d_status, void* stream) {
  const int rc = check_cfg(cfg);
  if (rc != KITTY_OK) return rc;
  if (n_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (n_pages == 0) return KITTY_OK;
  if (!k || !v || !page_ids || !pool || !aligned16(k) || !aligned16(v) || !aligned16(pool))
    return KITTY_ERR_INVALID_ARG;
  if (n_pages > 65535 * 1024) return KITTY_ERR_UNSUPPORTED;
  dim3 grid(n_pages, cfg->num_kv_heads);
  f16kv_write_kernel<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), page_ids,
      cfg->num_kv_heads, static_cast<uint8_t*>(pool), pool_pages, d_status);
  return cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
}

extern "C" int kitty_f16kv_append(const kitty_cfg* cfg, const void* k_new, const void* v_new,
                                  void* pool, int32_t pool_pages, int32_t* block_table,
                                  int32_t max_pages, int32_t* ctx_len,
                                  const int32_t* new_page_ids, int32_t B, int32_t* d_status,
                                  void* stream) {
  const int rc = check_cfg(cfg);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (B == 0) return KITTY_OK;
  if (!k_new || !v_new || !pool || !block_table || !ctx_len || !new_page_ids || !aligned16(pool))
    return KITTY_ERR_INVALID_ARG;
  if (B > 65535) return KITTY_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  f16kv_append_kernel<<<dim3(B, cfg->num_kv_heads), 128, 0, s>>>(
      static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
      static_cast<uint8_t*>(pool), pool_pages, block_table, max_pages, ctx_len, new_page_ids,
      cfg->num_kv_heads, d_status);
  f16kv_append_finalize<<<(B + 127) / 128, 128, 0, s>>>(block_table, max_pages, ctx_len,
                                                        new_page_ids, pool_pages, B);
  return cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
}

extern "C" int kitty_f16kv_workspace_bytes(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                           size_t* bytes) {
  const int rc = check_cfg(cfg, 4);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || !bytes) return KITTY_ERR_INVALID_ARG;
  int splits = 1, pps = 1;
  f16kv_plan(B * cfg->num_kv_heads, max_pages, &splits, &pps);
  *bytes = splits > 1 ? (size_t)B * cfg->num_q_heads * splits * kFPartial * sizeof(float) : 0;
  return KITTY_OK;
}

extern "C" int kitty_f16kv_decode(const kitty_cfg* cfg, const void* q, const void* pool,
                                  int32_t pool_pages, const int32_t* block_table,
                                  int32_t max_pages, const int32_t* ctx_len, float sm_scale,
                                  void* out, int32_t out_dtype, void* workspace,
                                  size_t workspace_bytes, int32_t B, int32_t* d_status,
                                  void* stream) {
  const int rc = check_cfg(cfg, 4);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (out_dtype != KITTY_F32 && out_dtype != KITTY_BF16 && out_dtype != KITTY_F16)
    return KITTY_ERR_INVALID_ARG;
  if (B == 0) return KITTY_OK;
  if (B > 65535) return KITTY_ERR_UNSUPPORTED;
  if (!q || !out || !ctx_len || (max_pages > 0 && (!block_table || !pool)) ||
      (pool && !aligned16(pool)) || !std::isfinite(sm_scale))
    return KITTY_ERR_INVALID_ARG;
  F16Params p = {};
  f16kv_plan(B * cfg->num_kv_heads, max_pages, &p.splits, &p.pps);
  const size_t need =
      p.splits > 1 ? (size_t)B * cfg->num_q_heads * p.splits * kFPartial * sizeof(float) : 0;
  if (workspace_bytes < need || (need > 0 && (!workspace || !aligned16(workspace))))
    return KITTY_ERR_WORKSPACE;
  p.q = static_cast<const uint16_t*>(q);
  p.pool = static_cast<const uint8_t*>(pool);
  p.block_table = block_table;
  p.ctx_len = ctx_len;
  p.out = out;
  p.ws = static_cast<float*>(workspace);
  p.d_status = d_status;
  p.sm_log2 = sm_scale * 1.4426950408889634f;
  p.pool_pages = pool_pages;
  p.max_pages = max_pages;
  p.out_dtype = out_dtype;
  p.Hkv = cfg->num_kv_heads;
  p.Hq = cfg->num_q_heads;
  p.g = cfg->num_q_heads / cfg->num_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)B * cfg->num_kv_heads, p.splits);
  const cudaError_t e = cfg->in_dtype == KITTY_BF16 ? launch_f16kv<KITTY_BF16>(grid, s, p)
                                                    : launch_f16kv<KITTY_F16>(grid, s, p);
  if (e != cudaSuccess) return KITTY_ERR_CUDA;
  if (p.splits > 1) f16kv_combine_kernel<<<(unsigned)B * cfg->num_q_heads, 128, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
}
