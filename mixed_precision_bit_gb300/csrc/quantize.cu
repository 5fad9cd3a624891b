// Kitty page quantization for GB300 (sm_103a): channel statistics, variance
// top-k boost selection, asymmetric min/max quantization of Keys (2-bit, boosted
// channels 4-bit split into two 2-bit planes) and Values (2-bit per-token groups
// of 32 channels), packed into the page-centric blob.
//
// Paper: "Kitty: Accurate and Efficient 2-bit KV Cache Quantization with
// Dynamic Channel-wise Precision Boost", Abstract.  Steps: "Kitty -- Dynamic
// Channel-wise Mixed-Precision Keys" (VeloxQuant-MLX docs), How it works,
// Prefill phase steps 1-3 and 5, Decode phase steps 1-3.
//
// Every fp32 step uses an explicitly rounded intrinsic (no contraction), in the
// order that defines the page bytes, so the packed pages are bit-exact with a
// plain sequential implementation.  One CTA of 128 threads quantizes one
// (page, kv-head): thread c owns Key channel c; thread 4t+G owns Value group G
// of token t.
//
// Device-side quantizer: quant_tile.cuh.
#include "quant_tile.cuh"
#include "host_common.h"

namespace kitty {
namespace {

// Page mode: one CTA per (input page i, kv head h).
template <int DT, int W, int V>
__global__ void __launch_bounds__(kQThreads, 8) quantize_pages_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, const int32_t* page_ids,
    int n_hi, int Hkv, uint8_t* pool, int pool_pages, int32_t* d_status) {
  __shared__ QuantSmem sm;
  const int i = blockIdx.x, h = blockIdx.y;
  const int pid = page_ids[i];
  if (pid < 0 || pid >= pool_pages) {
    if (threadIdx.x == 0) set_status(d_status, KITTY_ST_BAD_PAGE);
    return;
  }
  const BlobLayout lay(n_hi, W, V);
  const size_t stride = (size_t)Hkv * kD;
  const size_t src = (size_t)i * kPage * stride + (size_t)h * kD;
  float dummy_s = 0.f, dummy_q = 0.f;
  int dummy_c = 0;
  quantize_tile<DT, W, V>(sm, k + src, v + src, stride, n_hi, false, dummy_s, dummy_q, dummy_c,
                    pool + ((size_t)pid * Hkv + h) * lay.bytes, d_status);
}

__global__ void check_seq_kernel(const int32_t* seq_of_page, int n_pages, int n_seqs,
                                 int32_t* d_status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_pages) return;
  const int s = seq_of_page[i];
  if (s < 0 || s >= n_seqs || (i > 0 && s < seq_of_page[i - 1])) set_status(d_status, KITTY_ST_BAD_SEQ);
}

// Running and sequence modes, in three launches.  Only the fp32 accumulation
// over a sequence's pages is sequential, so:
//  A. page_sums_kernel (one CTA per (page, kv head)): the page's tree-ordered
//     channel sums S1, S2, parked in the page's own output blob (scratch);
//  B. seq_scan_kernel (one CTA per (sequence, kv head)): the same fp32 adds in
//     page order as a sequential walk.  Running mode writes each page's
//     running totals (including that page) back into its blob; sequence mode
//     ranks once on the totals and writes the boost flags into every blob.
//     The final totals go to run_sum / run_sumsq / run_count;
//  C. quantize_given_kernel (one CTA per (page, kv head)): reads its blob's
//     totals or flags, then overwrites the blob with the quantized page.
// Every fp32 operation and its order are those of a one-page-at-a-time walk,
// so the pages and accumulators are bit-identical to it.  Pages are distinct
// pool pages (the caller's ids), so blobs do not collide.
//
// Scratch words in a blob: running mode S1/R1 [0,128), S2/R2 [128,256), count
// [256]; sequence mode boost flags [0,128).

// Top-k boost flag of channel threadIdx.x for a variance given per thread, in
// shared arrays key[128] and boost[4].  Called by all 128 threads.
__device__ __forceinline__ bool topk_flag(uint32_t* key, uint32_t* boost, float var, int n_hi) {
  key[threadIdx.x] = var_key(var);
  __syncthreads();
  if (threadIdx.x < 32) topk_masks(key, boost, n_hi);
  __syncthreads();
  return (boost[threadIdx.x >> 5] >> (threadIdx.x & 31)) & 1u;
}

__device__ __forceinline__ int first_page_of(const int32_t* seq_of_page, int n_pages, int s) {
  int lo = 0, hi = n_pages;
  while (lo < hi) { const int m = (lo + hi) >> 1; if (seq_of_page[m] < s) lo = m + 1; else hi = m; }
  return lo;
}

template <int DT>
__global__ void __launch_bounds__(kQThreads, 8) page_sums_kernel(
    const uint16_t* __restrict__ k, const int32_t* page_ids, const int32_t* seq_of_page,
    int n_seqs, int Hkv, uint8_t* pool, int pool_pages, int blob) {
  __shared__ QuantSmem sm;
  const int i = blockIdx.x, h = blockIdx.y;
  const int sq = seq_of_page[i];
  const int pid = page_ids[i];
  // a bad id is reported by pass C; a bad sequence by check_seq_kernel
  if (pid < 0 || pid >= pool_pages || sq < 0 || sq >= n_seqs) return;
  const size_t stride = (size_t)Hkv * kD;
  float s1, s2;
  tile_stats<DT>(sm, k + (size_t)i * kPage * stride + (size_t)h * kD, stride, s1, s2);
  float* sc = reinterpret_cast<float*>(pool + ((size_t)pid * Hkv + h) * blob);
  sc[threadIdx.x] = s1;
  sc[kD + threadIdx.x] = s2;
}

// Thread c = channel c.  Pages are read 32 at a time ahead of the adds.
__global__ void __launch_bounds__(kQThreads) seq_scan_kernel(
    const int32_t* page_ids, const int32_t* seq_of_page, int n_pages, int Hkv, float* run_sum,
    float* run_sumsq, int32_t* run_count, uint8_t* pool, int pool_pages, int blob, int n_hi,
    int sequence_mode) {
  __shared__ uint32_t key[kD], boost[kD / 32];  // sequence-mode ranking
  const int s = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int p0 = first_page_of(seq_of_page, n_pages, s);
  const int p1 = first_page_of(seq_of_page, n_pages, s + 1);
  if (p0 >= p1) return;
  const size_t sh = (size_t)s * Hkv + h;
  float rs = run_sum[sh * kD + c];
  float rq = run_sumsq[sh * kD + c];
  int rc = run_count[sh];
  constexpr int kAhead = 32;  // pages whose sums are loaded ahead of the adds (a long chain is latency-bound)
  for (int i0 = p0; i0 < p1; i0 += kAhead) {
    float a1[kAhead], a2[kAhead];
    float* sc[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int i = i0 + u;
      const int pid = i < p1 ? page_ids[i] : -1;
      sc[u] = pid >= 0 && pid < pool_pages
                  ? reinterpret_cast<float*>(pool + ((size_t)pid * Hkv + h) * blob) : nullptr;
      a1[u] = sc[u] ? sc[u][c] : 0.f;
      a2[u] = sc[u] ? sc[u][kD + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      if (sc[u] == nullptr) continue;  // invalid page: not counted
      rs = __fadd_rn(rs, a1[u]);
      rq = __fadd_rn(rq, a2[u]);
      rc += kPage;
      if (!sequence_mode) {
        sc[u][c] = rs;
        sc[u][kD + c] = rq;
        if (c == 0) reinterpret_cast<int*>(sc[u])[2 * kD] = rc;
      }
    }
  }
  if (sequence_mode) {
    const int flag = topk_flag(key, boost, running_var(rs, rq, __int2float_rn(rc)), n_hi) ? 1 : 0;
    for (int i = p0; i < p1; ++i) {
      const int pid = page_ids[i];
      if (pid >= 0 && pid < pool_pages)
        reinterpret_cast<int*>(pool + ((size_t)pid * Hkv + h) * blob)[c] = flag;
    }
  }
  run_sum[sh * kD + c] = rs;
  run_sumsq[sh * kD + c] = rq;
  if (c == 0) run_count[sh] = rc;
}

// Passes A and B in one launch, for batches with many (sequence, kv head)
// chains: one CTA per chain streams its pages' Key tiles through a two-stage
// cp.async ring (16 bytes a thread, 4 per page) and computes each page's
// tree-ordered sums on arrival; the running totals take the same fp32 adds in
// page order as seq_scan_kernel, so the scratch words, the final totals and the
// sequence-mode flags are bit-identical to passes A and B.  Thread c = channel c.
constexpr int kWalkStages = 2;

template <int DT>
__global__ void __launch_bounds__(kQThreads) seq_walk_kernel(
    const uint16_t* __restrict__ k, const int32_t* page_ids, const int32_t* seq_of_page,
    int n_pages, int Hkv, float* run_sum, float* run_sumsq, int32_t* run_count, uint8_t* pool,
    int pool_pages, int blob, int n_hi, int sequence_mode) {
  __shared__ __align__(16) uint16_t tile[kWalkStages][kPage][kD];
  __shared__ uint32_t key[kD];
  __shared__ uint32_t boost[kD / 32];
  const int s = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int p0 = first_page_of(seq_of_page, n_pages, s);
  const int p1 = first_page_of(seq_of_page, n_pages, s + 1);
  if (p0 >= p1) return;
  const size_t sh = (size_t)s * Hkv + h;
  const size_t stride = (size_t)Hkv * kD;
  float rs = run_sum[sh * kD + c];
  float rq = run_sumsq[sh * kD + c];
  int rc = run_count[sh];
  auto issue = [&](int i) {  // page i's Key tile into stage i % kWalkStages
    const uint16_t* src = k + (size_t)i * kPage * stride + (size_t)h * kD;
    const uint32_t dst = smem_u32(&tile[(i - p0) % kWalkStages][0][0]);
#pragma unroll
    for (int it = 0; it < kPage * (kD / 8) / kQThreads; ++it) {
      const int idx = c + it * kQThreads;
      const int t = idx >> 4, ch = (idx & 15) * 8;
      cp_async16(dst + (uint32_t)(t * kD + ch) * 2, src + (size_t)t * stride + ch);
    }
  };
  for (int j = 0; j < kWalkStages - 1; ++j) {
    if (p0 + j < p1) issue(p0 + j);
    cp_async_commit();
  }
  for (int i = p0; i < p1; ++i) {
    if (i + kWalkStages - 1 < p1) issue(i + kWalkStages - 1);
    cp_async_commit();  // one group per iteration, empty near the end
    cp_async_wait<kWalkStages - 1>();
    __syncthreads();  // page i's tile complete for every thread
    const int pid = page_ids[i];
    if (pid >= 0 && pid < pool_pages) {  // an invalid page is not counted (pass C reports it)
      const int st = (i - p0) % kWalkStages;
      float a[kPage], b[kPage];
#pragma unroll
      for (int t = 0; t < kPage; ++t) a[t] = bits16_to_f32(tile[st][t][c], DT);
#pragma unroll
      for (int t = 0; t < kPage; t += 2) mul2_rn(b[t], b[t + 1], a[t], a[t + 1], a[t], a[t + 1]);
      const float s1 = tree32(a), s2 = tree32(b);
      rs = __fadd_rn(rs, s1);
      rq = __fadd_rn(rq, s2);
      rc += kPage;
      if (!sequence_mode) {
        float* sc = reinterpret_cast<float*>(pool + ((size_t)pid * Hkv + h) * blob);
        sc[c] = rs;
        sc[kD + c] = rq;
        if (c == 0) reinterpret_cast<int*>(sc)[2 * kD] = rc;
      }
    }
    __syncthreads();  // every thread is done with this stage before it is refilled
  }
  if (sequence_mode) {
    // the boost set of the whole sequence (the page quantizer's ranking)
    const int flag = topk_flag(key, boost, running_var(rs, rq, __int2float_rn(rc)), n_hi) ? 1 : 0;
    for (int i = p0; i < p1; ++i) {
      const int pid = page_ids[i];
      if (pid >= 0 && pid < pool_pages)
        reinterpret_cast<int*>(pool + ((size_t)pid * Hkv + h) * blob)[c] = flag;
    }
  }
  run_sum[sh * kD + c] = rs;
  run_sumsq[sh * kD + c] = rq;
  if (c == 0) run_count[sh] = rc;
}

template <int DT, int W, int V>
__global__ void __launch_bounds__(kQThreads, 8) quantize_given_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, const int32_t* page_ids,
    const int32_t* seq_of_page, int n_seqs, int n_hi, int Hkv, uint8_t* pool, int pool_pages,
    int sequence_mode, int32_t* d_status) {
  __shared__ QuantSmem sm;
  const int i = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int sq = seq_of_page[i];
  if (sq < 0 || sq >= n_seqs) return;  // no sequence scanned it (KITTY_ST_BAD_SEQ is set)
  const int pid = page_ids[i];
  if (pid < 0 || pid >= pool_pages) {
    if (c == 0) set_status(d_status, KITTY_ST_BAD_PAGE);
    return;
  }
  const BlobLayout lay(n_hi, W, V);
  uint8_t* dst = pool + ((size_t)pid * Hkv + h) * lay.bytes;
  const size_t stride = (size_t)Hkv * kD;
  const size_t src = (size_t)i * kPage * stride + (size_t)h * kD;
  const float* sc = reinterpret_cast<const float*>(dst);
  float rs = 0.f, rq = 0.f;
  int rc = 0, fixed;
  if (sequence_mode) {
    fixed = reinterpret_cast<const int*>(sc)[c] != 0 ? 1 : 0;
  } else {
    rs = sc[c];
    rq = sc[kD + c];
    rc = reinterpret_cast<const int*>(sc)[2 * kD];
    fixed = -2;  // rank on these totals
  }
  // quantize_tile reads the scratch values above before it overwrites the blob
  // (its only global write, after its last barrier)
  quantize_tile<DT, W, V>(sm, k + src, v + src, stride, n_hi, false, rs, rq, rc, dst, d_status, fixed);
}

// Append, part 1: one CTA per (sequence b, kv head h) writes the token into the
// tail and, when the tail fills and a page id is given, quantizes the tail.
template <int DT, int W, int V>
__global__ void __launch_bounds__(kQThreads) append_heads_kernel(
    const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new, uint16_t* tail_k,
    uint16_t* tail_v, const int32_t* tail_len, float* run_sum, float* run_sumsq,
    int32_t* run_count, const int32_t* flush_page_ids, int max_pages, const int32_t* num_pages,
    uint8_t* pool, int pool_pages, int n_hi, int Hkv, int running, int32_t* d_status) {
  __shared__ QuantSmem sm;
  const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int len = tail_len[b];
  if (len < 0 || len > kPage) { if (c == 0) set_status(d_status, KITTY_ST_BAD_LEN); return; }
  if (len == kPage) { if (c == 0) set_status(d_status, KITTY_ST_TAIL_FULL); return; }
  const size_t sh = (size_t)b * Hkv + h;
  tail_k[(sh * kPage + len) * kD + c] = k_new[sh * kD + c];
  tail_v[(sh * kPage + len) * kD + c] = v_new[sh * kD + c];
  const int n = len + 1;
  const int fid = flush_page_ids[b];
  if (fid >= 0 && n < kPage) { if (c == 0) set_status(d_status, KITTY_ST_BAD_FLUSH); return; }
  if (n < kPage || fid < 0) return;
  const int np = num_pages[b];
  if (np < 0 || np >= max_pages) { if (c == 0) set_status(d_status, KITTY_ST_TABLE_FULL); return; }
  if (fid >= pool_pages) { if (c == 0) set_status(d_status, KITTY_ST_BAD_PAGE); return; }
  __syncthreads();  // the new token row is visible to the whole CTA
  const BlobLayout lay(n_hi, W, V);
  float rs = 0.f, rq = 0.f;
  int rc = 0;
  if (running) {
    rs = run_sum[sh * kD + c];
    rq = run_sumsq[sh * kD + c];
    rc = run_count[sh];
  }
  quantize_tile<DT, W, V>(sm, tail_k + sh * kPage * kD, tail_v + sh * kPage * kD, kD, n_hi, running != 0,
                    rs, rq, rc, pool + ((size_t)fid * Hkv + h) * lay.bytes, d_status);
  if (running) {
    run_sum[sh * kD + c] = rs;
    run_sumsq[sh * kD + c] = rq;
    if (c == 0) run_count[sh] = rc;
  }
}

// Append, part 2: per-sequence bookkeeping (tail length, block table, page
// count), after every head of the sequence has used the old values.
__global__ void append_finalize_kernel(int32_t* tail_len, const int32_t* flush_page_ids,
                                       int32_t* block_table, int max_pages, int32_t* num_pages,
                                       int pool_pages, int B) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  append_finalize_one(b, tail_len, flush_page_ids, block_table, max_pages, num_pages, pool_pages);
}

// Calls f(KernelTag<DT, W, V>{}) for the configuration's input dtype, Key plane
// width (lo_bit) and Value code width (v_bit; 4 only with 4-bit Key planes).
template <int DT_, int W_, int V_>
struct KernelTag {
  static constexpr int DT = DT_, W = W_, V = V_;
};

template <class F>
void dispatch(const kitty_cfg* cfg, F f) {
  const int v = v_bits(cfg);
  if (cfg->in_dtype == KITTY_BF16) {
    if (cfg->lo_bit == 4 && v == 4) f(KernelTag<KITTY_BF16, 4, 4>{});
    else if (cfg->lo_bit == 4) f(KernelTag<KITTY_BF16, 4, 2>{});
    else f(KernelTag<KITTY_BF16, 2, 2>{});
  } else {
    if (cfg->lo_bit == 4 && v == 4) f(KernelTag<KITTY_F16, 4, 4>{});
    else if (cfg->lo_bit == 4) f(KernelTag<KITTY_F16, 4, 2>{});
    else f(KernelTag<KITTY_F16, 2, 2>{});
  }
}

}  // namespace
}  // namespace kitty

using namespace kitty;

extern "C" int kitty_quantize_pages(const kitty_cfg* cfg, const void* k, const void* v,
                                    int32_t n_pages, const int32_t* page_ids,
                                    const int32_t* seq_of_page, int32_t n_seqs, float* run_sum,
                                    float* run_sumsq, int32_t* run_count, void* pool,
                                    int32_t pool_pages, int32_t* d_status, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != KITTY_OK) return rc;
  if (n_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (n_pages == 0) return KITTY_OK;
  if (!k || !v || !page_ids || !pool || !aligned16(k) || !aligned16(v) || !aligned16(pool))
    return KITTY_ERR_INVALID_ARG;
  const bool running = cfg->rank_mode != KITTY_RANK_PAGE;  // running or sequence mode
  if (running && (!seq_of_page || n_seqs <= 0 || !run_sum || !run_sumsq || !run_count))
    return KITTY_ERR_INVALID_ARG;
  if (n_pages > 65535 * 1024) return KITTY_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Hkv = cfg->num_kv_heads;
  const auto* k16 = static_cast<const uint16_t*>(k);
  const auto* v16 = static_cast<const uint16_t*>(v);
  auto* p8 = static_cast<uint8_t*>(pool);
  if (!running) {
    dim3 grid(n_pages, Hkv);
    dispatch(cfg, [&](auto tag) {
      using T = decltype(tag);
      quantize_pages_kernel<T::DT, T::W, T::V><<<grid, kQThreads, 0, s>>>(k16, v16, page_ids, cfg->n_hi, Hkv, p8, pool_pages, d_status);
    });
  } else {
    check_seq_kernel<<<(n_pages + 255) / 256, 256, 0, s>>>(seq_of_page, n_pages, n_seqs, d_status);
    const int blob = (int)blob_bytes(cfg->n_hi, cfg->lo_bit, v_bits(cfg));
    const int seq = cfg->rank_mode == KITTY_RANK_SEQUENCE ? 1 : 0;
    dim3 pages(n_pages, Hkv), seqs(n_seqs, Hkv);
    if ((long)n_seqs * Hkv >= 3L * sm_count()) {
      // many chains: passes A and B fused, Key tiles read once
      if (cfg->in_dtype == KITTY_BF16)
        seq_walk_kernel<KITTY_BF16><<<seqs, kQThreads, 0, s>>>(k16, page_ids, seq_of_page, n_pages, Hkv, run_sum, run_sumsq, run_count, p8, pool_pages, blob, cfg->n_hi, seq);
      else
        seq_walk_kernel<KITTY_F16><<<seqs, kQThreads, 0, s>>>(k16, page_ids, seq_of_page, n_pages, Hkv, run_sum, run_sumsq, run_count, p8, pool_pages, blob, cfg->n_hi, seq);
    } else {
      if (cfg->in_dtype == KITTY_BF16)
        page_sums_kernel<KITTY_BF16><<<pages, kQThreads, 0, s>>>(k16, page_ids, seq_of_page, n_seqs, Hkv, p8, pool_pages, blob);
      else
        page_sums_kernel<KITTY_F16><<<pages, kQThreads, 0, s>>>(k16, page_ids, seq_of_page, n_seqs, Hkv, p8, pool_pages, blob);
      seq_scan_kernel<<<seqs, kQThreads, 0, s>>>(page_ids, seq_of_page, n_pages, Hkv, run_sum, run_sumsq,
                                                 run_count, p8, pool_pages, blob, cfg->n_hi, seq);
    }
    dispatch(cfg, [&](auto tag) {
      using T = decltype(tag);
      quantize_given_kernel<T::DT, T::W, T::V><<<pages, kQThreads, 0, s>>>(k16, v16, page_ids, seq_of_page, n_seqs, cfg->n_hi, Hkv, p8, pool_pages, seq, d_status);
    });
  }
  return cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
}

extern "C" int kitty_append_token(const kitty_cfg* cfg, const void* k_new, const void* v_new,
                                  void* tail_k, void* tail_v, int32_t* tail_len, float* run_sum,
                                  float* run_sumsq, int32_t* run_count,
                                  const int32_t* flush_page_ids, int32_t* block_table,
                                  int32_t max_pages, int32_t* num_pages, void* pool,
                                  int32_t pool_pages, int32_t B, int32_t* d_status, void* stream) {
  int rc = check_cfg(cfg);
  if (rc != KITTY_OK) return rc;
  if (B < 0 || max_pages < 0 || pool_pages < 0) return KITTY_ERR_INVALID_ARG;
  if (B == 0) return KITTY_OK;
  if (!k_new || !v_new || !tail_k || !tail_v || !tail_len || !flush_page_ids || !block_table ||
      !num_pages || !pool || !aligned16(tail_k) || !aligned16(tail_v) || !aligned16(pool))
    return KITTY_ERR_INVALID_ARG;
  const bool running = cfg->rank_mode != KITTY_RANK_PAGE;  // sequence mode appends as running
  if (running && (!run_sum || !run_sumsq || !run_count)) return KITTY_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Hkv = cfg->num_kv_heads;
  dim3 grid(B, Hkv);
  auto* tk = static_cast<uint16_t*>(tail_k);
  auto* tv = static_cast<uint16_t*>(tail_v);
  const auto* kn = static_cast<const uint16_t*>(k_new);
  const auto* vn = static_cast<const uint16_t*>(v_new);
  auto* p8 = static_cast<uint8_t*>(pool);
  dispatch(cfg, [&](auto tag) {
    using T = decltype(tag);
    append_heads_kernel<T::DT, T::W, T::V><<<grid, kQThreads, 0, s>>>(kn, vn, tk, tv, tail_len, run_sum, run_sumsq, run_count, flush_page_ids, max_pages, num_pages, p8, pool_pages, cfg->n_hi, Hkv, running ? 1 : 0, d_status);
  });
  append_finalize_kernel<<<(B + 127) / 128, 128, 0, s>>>(tail_len, flush_page_ids, block_table, max_pages, num_pages, pool_pages, B);
  return cudaGetLastError() == cudaSuccess ? KITTY_OK : KITTY_ERR_CUDA;
}
