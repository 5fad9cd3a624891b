/* kitty.h -- C ABI of the Kitty GB300 library (libkitty.so).
 *
 * Kitty keeps a paged KV cache at ~2 bits per element.  Key pages rank their
 * channels by variance and store the top n_hi at 4 bits, split into two 2-bit
 * planes, so every Key page is two uniform 2-bit tensors plus a channel list;
 * Values use 2-bit per-token groups of 32 channels (4-bit as an option, for the
 * uniform 4-bit KV comparison layout).  Decode attention reads the
 * packed pages through a block table and dequantizes them in registers.
 *
 * Sources: "Kitty: Accurate and Efficient 2-bit KV Cache Quantization with
 * Dynamic Channel-wise Precision Boost" (arXiv 2511.18643), Abstract; and
 * "Kitty -- Dynamic Channel-wise Mixed-Precision Keys" (VeloxQuant-MLX docs),
 * sections "How it works" (Prefill phase, Decode phase), "Effective bit-width"
 * and "Configuration reference".
 *
 * Conventions for every entry point:
 *  - Return value: KITTY_OK (0) or a negative KITTY_ERR_* code.  Arguments are
 *    checked on the host before anything is launched; on an error nothing is
 *    launched and no memory is touched.
 *  - Device pointers are raw CUDA device addresses owned by the caller (the
 *    library allocates no device memory and keeps no global state, apart from
 *    the fixed scratch array of kitty_decode_attention_noalloc).  Work is
 *    enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronizing.
 *  - `d_status` (optional, may be NULL) is a caller-owned device int32.  Data
 *    errors found on the device (bad page id, bad lengths, out-of-range input,
 *    wait timeout) store a KITTY_ST_* code there if it still holds 0 (first
 *    error wins); the affected work item is skipped.  The library never traps.
 *  - 16-bit inputs are fp16 or bf16 per cfg->in_dtype.  Layouts are dense,
 *    row-major, with the shapes given below.
 */
#ifndef KITTY_H_
#define KITTY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes */
#define KITTY_OK 0
#define KITTY_ERR_INVALID_ARG -1 /* null pointer, bad size, misaligned pointer */
#define KITTY_ERR_UNSUPPORTED -2 /* a configuration the kernels do not cover */
#define KITTY_ERR_CUDA -3        /* a CUDA runtime call or launch failed */
#define KITTY_ERR_WORKSPACE -4   /* workspace smaller than kitty_decode_workspace_bytes */
#define KITTY_ERR_OOM -5         /* page allocator has too few free pages */

/* device status codes (written to *d_status) */
#define KITTY_ST_OK 0
#define KITTY_ST_EMPTY 1      /* a sequence with no cached token: its output is 0 */
#define KITTY_ST_RANGE 2      /* |input| > 65504: fp16 metadata cannot hold it */
#define KITTY_ST_NONFINITE 3  /* NaN or Inf input */
#define KITTY_ST_BAD_PAGE 4   /* page id outside [0, pool_pages) or corrupt page */
#define KITTY_ST_BAD_LEN 5    /* num_pages outside [0, max_pages] or tail_len outside [0, 32] */
#define KITTY_ST_TAIL_FULL 6  /* append to a tail that already holds 32 tokens */
#define KITTY_ST_BAD_FLUSH 7  /* flush page id given although the tail did not fill */
#define KITTY_ST_TABLE_FULL 8 /* flush with num_pages == max_pages */
#define KITTY_ST_BAD_SEQ 9    /* seq_of_page not non-decreasing in [0, n_seqs) */
#define KITTY_ST_TIMEOUT 10   /* a bounded wait on an in-flight copy gave up */

#define KITTY_F16 0
#define KITTY_BF16 1
#define KITTY_F32 2 /* output only */

#define KITTY_RANK_PAGE 0    /* rank each page on its own 32 tokens */
#define KITTY_RANK_RUNNING 1 /* rank on running sum / sum of squares per (seq, head) */
#define KITTY_RANK_SEQUENCE 2 /* bulk quantize: one ranking per (seq, head) over all its
                                 pages (prefill); appends then continue as running mode */

/* Configuration.  The parameters follow the VeloxQuant-MLX docs,
 * "Configuration reference": kitty_hi_fraction (as n_hi = round(hf * D)),
 * kitty_hi_bit, kitty_lo_bit, kitty_group_size, head_dim. */
typedef struct {
  int32_t head_dim;     /* D; must be 128 */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t num_q_heads;  /* Hq, a multiple of Hkv.  Decode attention takes
                           Hq/Hkv <= 32 (groups above 4 run as CTAs of 4
                           query heads over the same pages); the fused append
                           + decode and the 16-bit baseline take Hq/Hkv <= 4 */
  int32_t page_tokens;  /* tokens per page = Key quantization group; must be 32 */
  int32_t n_hi;         /* boosted Key channels per page: 0, 16, 32, ..., 128 */
  int32_t hi_bit;       /* (hi_bit, lo_bit) = (4, 2): Key channels 2-bit, boosted 4-bit as */
  int32_t lo_bit;       /* two 2-bit planes; or (8, 4): 4-bit, boosted 8-bit as two 4-bit
                           planes (VeloxQuant-MLX docs, "Tuning avg_bits"); Values are
                           2-bit in both */
  int32_t v_group;      /* channels per Value group; must be 32 */
  int32_t rank_mode;    /* KITTY_RANK_PAGE, KITTY_RANK_RUNNING or KITTY_RANK_SEQUENCE */
  int32_t in_dtype;     /* KITTY_F16 or KITTY_BF16 for K, V, Q and the tails */
  int32_t decode_pages_per_split; /* split-K: 0 = library's schedule (split sizes
                                   shrinking towards the end of the grid), > 0 =
                                   splits of this many pages, raised to
                                   ceil(max_pages / 256) if smaller */
  int32_t decode_total_pages;     /* optional planning hint for the library's split
                                   schedule: the batch's total page count
                                   (sum of num_pages); 0 = unknown.  Any value
                                   gives correct results; it only shapes the
                                   splits (and so the workspace size) */
  int32_t decode_max_pages;       /* optional planning hint: the largest num_pages
                                   of the batch; 0 = unknown (max_pages is
                                   assumed).  Splits are sized over this many
                                   pages, and the last one still reaches
                                   max_pages, so any value gives correct
                                   results */
  int32_t decode_wait_polls;      /* bound of the decode page loop's waits for a
                                   staged page, in polls of its barrier;
                                   0 = the library's bound (2^22 polls, about
                                   0.1-1 s).  A wait that runs out sets
                                   KITTY_ST_TIMEOUT, waits (with the library's
                                   bound) for the CTA's copies still in flight
                                   and ends the CTA's page loop; its outputs are
                                   then undefined.  A small value makes ordinary
                                   copies outlast the wait, which is how the
                                   timeout path is tested */
  int32_t v_bit;                  /* Value code width: 2 (0 = 2) or 4.  4-bit
                                   Values need lo_bit = 4; with n_hi = 0 that
                                   is a uniform 4-bit KV cache (per-channel
                                   4-bit Keys, per-token 4-bit Value groups),
                                   the accuracy-preserving point the paper's
                                   Abstract names ("4-bit KV quantization") */
} kitty_cfg;

/* Library ABI version (this header: 5; kitty_cfg gained decode_total_pages in
 * version 2, decode_max_pages in version 3, decode_wait_polls in version 4 and
 * v_bit in version 5). */
int kitty_abi_version(void);

/* Packed page size.  A page holds Hkv blobs, one per kv head, in head order;
 * physical page p starts at byte p * per_page of the pool.  Blob of one
 * (page, kv head), in order, with w = lo_bit and v = v_bit: Key base plane
 * 512*w B, Key extra plane 4*w*n_hi B, Key step fp16[128], Key minimum
 * fp16[128], channel list uint8[n_hi] (ascending), Value plane 512*v B, Value
 * step fp16[4][32], Value minimum fp16[4][32] (group-major).  = 3072 + 9*n_hi
 * bytes at (4, 2) (3360 at n_hi=32), 4096 + 17*n_hi at (8, 4), 5120 + 17*n_hi
 * at (8, 4) with 4-bit Values.  Inside the planes, codes sit in "fragment
 * order": the 32*w (Keys) or 32*v (Values) bytes at offset 32*w*L (32*v*L) of
 * a plane hold what lane L of a warp takes as its tensor-core operand
 * fragments (the oracle's key_pos, key_pos4, val_pos and val_pos4 index
 * functions spell the maps out).  Paper: Abstract
 * (page-centric layout, two uniform 2-bit tensors per Key page). */
int kitty_page_bytes(const kitty_cfg* cfg, size_t* per_head_blob, size_t* per_page);

/* Effective Key bits per element, codes only: hf*hi_bit + (1-hf)*lo_bit with
 * hf = n_hi/D (VeloxQuant-MLX docs, "Effective bit-width").  <0 on a bad cfg. */
float kitty_avg_bits(const kitty_cfg* cfg);

/* ---------------------------------------------------------------- page allocator
 * Host-side free list of physical page ids [0, num_pages) (PagedAttention-style
 * block table, cited by the paper).  LIFO and deterministic: a fresh allocator
 * hands out 0, 1, 2, ...  Not thread-safe; one allocator per pool. */
typedef struct kitty_alloc kitty_alloc;
int kitty_alloc_create(int32_t num_pages, kitty_alloc** out);
/* n ids into ids_out, all or nothing: KITTY_ERR_OOM if fewer than n are free. */
int kitty_alloc_pages(kitty_alloc* a, int32_t n, int32_t* ids_out);
/* Return ids; KITTY_ERR_INVALID_ARG (nothing freed) on an id out of range or
 * not currently allocated. */
int kitty_free_pages(kitty_alloc* a, int32_t n, const int32_t* ids);
int32_t kitty_alloc_free_count(const kitty_alloc* a);
void kitty_alloc_destroy(kitty_alloc* a);

/* ---------------------------------------------------------------- quantize
 * Quantize n_pages pages of 32 tokens into the pool.  Paper: Abstract (Dynamic
 * Channel-wise Precision Boost, two-plane Key page); VeloxQuant-MLX docs,
 * Prefill phase steps 1-3 and 5.
 *   k, v        device [n_pages*32][Hkv][128] 16-bit; page i = tokens 32i..32i+31
 *   page_ids    device int32 [n_pages]: page i is written at pool page page_ids[i];
 *               the ids must be distinct (repeated ids give undefined pages;
 *               running and sequence modes use each page's own blob as scratch
 *               before writing it); out-of-range ids are skipped with
 *               KITTY_ST_BAD_PAGE
 *   Page mode: each page ranks its channels on its own 32 tokens; seq_of_page,
 *   run_* may be NULL and n_seqs is ignored.
 *   Running mode: seq_of_page device int32 [n_pages], non-decreasing, in
 *   [0, n_seqs); run_sum, run_sumsq device f32 [n_seqs][Hkv][128] and run_count
 *   device int32 [n_seqs][Hkv] are updated with each page's sums (in page order)
 *   before that page is ranked.
 *   Sequence mode (same arguments): the accumulators take all of a sequence's
 *   page sums first, the channels are ranked once on that variance, and every
 *   page of the sequence is quantized with that one boost set (VeloxQuant-MLX
 *   docs, Prefill phase: one ranking per head over the prompt).
 *   Both modes keep the fp32 additions in page order, so they give the same
 *   bytes as quantizing one page at a time.  With at least 3 (sequence, kv
 *   head) chains per SM they run in two launches (a per-chain walk that reads
 *   each Key tile once and keeps the running totals, then quantization in
 *   parallel); with fewer chains in three (page sums in parallel, a
 *   per-(sequence, head) scan, quantization in parallel).
 *   Pages whose seq_of_page entry is outside [0, n_seqs) are not written
 *   (KITTY_ST_BAD_SEQ).
 *   pool        device, pool_pages * per_page bytes, 16-byte aligned. */
int kitty_quantize_pages(const kitty_cfg* cfg, const void* k, const void* v, int32_t n_pages,
                         const int32_t* page_ids, const int32_t* seq_of_page, int32_t n_seqs,
                         float* run_sum, float* run_sumsq, int32_t* run_count, void* pool,
                         int32_t pool_pages, int32_t* d_status, void* stream);

/* ---------------------------------------------------------------- append
 * Append one token per sequence (VeloxQuant-MLX docs, Decode phase).  The token
 * goes to tail[b][h][tail_len[b]]; when the tail becomes full (32 tokens) and
 * flush_page_ids[b] >= 0, the tail is quantized as one page (running mode:
 * accumulators updated first) into pool page flush_page_ids[b], that id is
 * stored at block_table[b][num_pages[b]], num_pages[b] is incremented and the
 * tail emptied.  The caller knows every tail length, so it prepares
 * flush_page_ids without reading device memory.
 *   k_new, v_new   device [B][Hkv][128] 16-bit
 *   tail_k, tail_v device [B][Hkv][32][128] 16-bit
 *   tail_len, num_pages device int32 [B]; block_table device int32 [B][max_pages]
 *   run_sum, run_sumsq device f32 [B][Hkv][128], run_count int32 [B][Hkv]
 *   (running mode only; may be NULL in page mode)
 *   flush_page_ids device int32 [B], -1 = no flush for that sequence */
int kitty_append_token(const kitty_cfg* cfg, const void* k_new, const void* v_new, void* tail_k,
                       void* tail_v, int32_t* tail_len, float* run_sum, float* run_sumsq,
                       int32_t* run_count, const int32_t* flush_page_ids, int32_t* block_table,
                       int32_t max_pages, int32_t* num_pages, void* pool, int32_t pool_pages,
                       int32_t B, int32_t* d_status, void* stream);

/* ---------------------------------------------------------------- decode attention
 * Workspace needed by kitty_decode_attention for this batch shape (0 when a
 * single split suffices). */
int kitty_decode_workspace_bytes(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                 size_t* bytes);

/* Split-K paged decode attention (paper: Abstract, page dequantization with a
 * coalesced page-centric layout; FlashAttention-style online softmax).  For
 * query head hq of sequence b (kv head hq / (Hq/Hkv)):
 *   out[b][hq] = softmax_t(sm_scale * q.k_t) . v_t over the num_pages[b] pages
 *   listed in block_table[b][0..num_pages[b]) followed by the tail_len[b] tail
 *   tokens; an empty sequence gives 0 and KITTY_ST_EMPTY.
 *   q       device [B][Hq][128] 16-bit (in_dtype).  The tensor cores take the
 *           query as fp16: a bf16 query element with |q| > 65504 sets
 *           KITTY_ST_RANGE (NaN or Inf: KITTY_ST_NONFINITE), and the outputs of
 *           its kv head's query group are then undefined
 *   pool    device, 16-byte aligned, pool_pages pages
 *   tail_k, tail_v device [B][Hkv][32][128] 16-bit, 16-byte aligned; may be NULL
 *           if all tails are 0
 *   out     device [B][Hq][128] of out_dtype (KITTY_F32, KITTY_BF16, KITTY_F16)
 *   workspace device, >= kitty_decode_workspace_bytes, 16-byte aligned (may be
 *   NULL when that size is 0).
 * Query groups: Hq/Hkv <= 32.  A group above 4 heads runs as ceil(g/8) CTAs of
 * up to 8 query heads each in the (4, 2) format with 2-bit Values, else as
 * ceil(g/4) CTAs of up to 4 query heads each, over the same pages.
 * Launches, in stream order: the decode kernel, then (with more than one split)
 * the split combine as a programmatic dependent launch, which may start while
 * the decode grid drains and waits for it before reading the partials (32
 * threads per (sequence, query head) row up to 8 splits; above that, a
 * 128-thread CTA per row).  Both
 * can be captured in a CUDA graph, also as the first call on a device (that
 * call sets the kernel's shared-memory attributes, which is allowed during
 * capture). */
int kitty_decode_attention(const kitty_cfg* cfg, const void* q, const void* pool,
                           int32_t pool_pages, const int32_t* block_table, int32_t max_pages,
                           const int32_t* num_pages, const void* tail_k, const void* tail_v,
                           const int32_t* tail_len, float sm_scale, void* out, int32_t out_dtype,
                           void* workspace, size_t workspace_bytes, int32_t B, int32_t* d_status,
                           void* stream);

/* One decode step of a layer in one launch (plus the split combine): exactly
 * kitty_append_token followed by kitty_decode_attention on the updated cache,
 * with the same arguments, layouts, workspace size and status codes as those
 * two calls.  The new token goes into the tail; a sequence whose tail fills
 * and whose flush_page_ids entry is a page id gets that page quantized from
 * its tail (paper: Abstract, page-centric layout; VeloxQuant-MLX docs, Decode
 * phase steps 1-3) and attended from on-chip memory in the same launch; block
 * table, page counts and tail lengths are updated after every head has read
 * the old ones.  Invalid lengths (KITTY_ST_BAD_LEN) append nothing.
 *   tail_k, tail_v device [B][Hkv][32][128], 16-byte aligned (required here)
 *   workspace      >= kitty_decode_workspace_bytes(cfg, B, max_pages) */
int kitty_append_decode(const kitty_cfg* cfg, const void* k_new, const void* v_new, const void* q,
                        void* tail_k, void* tail_v, int32_t* tail_len, float* run_sum,
                        float* run_sumsq, int32_t* run_count, const int32_t* flush_page_ids,
                        int32_t* block_table, int32_t max_pages, int32_t* num_pages, void* pool,
                        int32_t pool_pages, float sm_scale, void* out, int32_t out_dtype,
                        void* workspace, size_t workspace_bytes, int32_t B, int32_t* d_status,
                        void* stream);

/* Decode attention that allocates nothing and takes no workspace.  The paper has
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory while they run -- e.g. a serving process that reserved all of
 * the GPU's memory for its page pool up front, or a host language runtime with
 * no access to a CUDA allocator.  It computes exactly what
 * kitty_decode_attention computes, with the split-K partials kept in a
 * file-scope device array of KITTY_NOALLOC_SCRATCH_BYTES (8 MiB) that every
 * GPU loading this library holds until the process exits.
 *  - Returns KITTY_ERR_WORKSPACE, launching nothing, when this batch shape
 *    needs more split-K scratch than that (kitty_decode_workspace_bytes tells).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - All calls on a device share the one array and every call overwrites the
 *    partials it reads, so nothing needs clearing between calls; calls whose
 *    kernels overlap on the GPU (different streams, no ordering) race on it.
 *  Arguments are those of kitty_decode_attention without the workspace. */
#define KITTY_NOALLOC_SCRATCH_BYTES (8u << 20)
int kitty_decode_attention_noalloc(const kitty_cfg* cfg, const void* q, const void* pool,
                                   int32_t pool_pages, const int32_t* block_table,
                                   int32_t max_pages, const int32_t* num_pages,
                                   const void* tail_k, const void* tail_v,
                                   const int32_t* tail_len, float sm_scale, void* out,
                                   int32_t out_dtype, int32_t B, int32_t* d_status, void* stream);

/* ---------------------------------------------------------------- 16-bit paged baseline
 * The unquantized paged KV cache that Kitty's memory budget and throughput are
 * compared against (paper: Abstract, "up to 8x larger batches and 2.1x-4.1x
 * higher throughput under the same memory budget").  Keys and Values stay in
 * the input dtype (cfg->in_dtype); cfg's quantization fields are ignored.
 * A (page, kv head) blob is K [32 tokens][128] followed by V [32][128], 16 KB; a
 * page holds Hkv blobs in head order.  Sequence b holds ctx_len[b] tokens, token
 * t in slot t % 32 of pool page block_table[b][t / 32]; there is no tail.
 * Conventions (status codes, streams, ownership) are those above. */
int kitty_f16kv_page_bytes(const kitty_cfg* cfg, size_t* per_head_blob, size_t* per_page);

/* Write n_pages full pages: page i of k, v (device [n_pages*32][Hkv][128],
 * 16-byte aligned) goes to pool page page_ids[i] (out-of-range ids are skipped
 * with KITTY_ST_BAD_PAGE). */
int kitty_f16kv_write_pages(const kitty_cfg* cfg, const void* k, const void* v, int32_t n_pages,
                            const int32_t* page_ids, void* pool, int32_t pool_pages,
                            int32_t* d_status, void* stream);

/* Append one token per sequence (k_new, v_new device [B][Hkv][128]) at position
 * ctx_len[b]; a token that starts a page (ctx_len[b] % 32 == 0) goes to the
 * caller's page new_page_ids[b], which is stored in the block table.  Then
 * ctx_len[b] is incremented.  A full table gives KITTY_ST_TABLE_FULL. */
int kitty_f16kv_append(const kitty_cfg* cfg, const void* k_new, const void* v_new, void* pool,
                       int32_t pool_pages, int32_t* block_table, int32_t max_pages,
                       int32_t* ctx_len, const int32_t* new_page_ids, int32_t B,
                       int32_t* d_status, void* stream);

/* Split-K workspace of kitty_f16kv_decode for this batch shape (0: one split). */
int kitty_f16kv_workspace_bytes(const kitty_cfg* cfg, int32_t B, int32_t max_pages,
                                size_t* bytes);

/* Decode attention over the 16-bit pages: for query head hq of sequence b,
 * out[b][hq] = softmax_t(sm_scale * q.k_t) . v_t over its ctx_len[b] tokens
 * (kv head hq / (Hq/Hkv)); an empty sequence gives 0 and KITTY_ST_EMPTY.  q
 * device [B][Hq][128] in_dtype; out [B][Hq][128] of out_dtype; workspace
 * >= kitty_f16kv_workspace_bytes, 16-byte aligned. */
int kitty_f16kv_decode(const kitty_cfg* cfg, const void* q, const void* pool, int32_t pool_pages,
                       const int32_t* block_table, int32_t max_pages, const int32_t* ctx_len,
                       float sm_scale, void* out, int32_t out_dtype, void* workspace,
                       size_t workspace_bytes, int32_t B, int32_t* d_status, void* stream);

/* Launch shape that kitty_decode_attention uses for this batch shape: number of
 * splits per (sequence, kv head, head group) (at most 256) and the pages in the
 * largest split (for reporting and tests).  Split s covers block-table positions [start_s,
 * start_(s+1)), from position 0 upwards with the largest split first.  A
 * sequence shorter than max_pages leaves its later splits without pages: they
 * write an empty partial, which the merge skips.  Split 0 always runs; it also
 * takes the tail tokens. */
int kitty_decode_plan(const kitty_cfg* cfg, int32_t B, int32_t max_pages, int32_t* splits,
                      int32_t* pages_per_split);

#ifdef __cplusplus
}
#endif

#endif /* KITTY_H_ */
