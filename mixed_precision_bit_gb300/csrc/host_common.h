// Host-side argument checks shared by the Kitty entry points.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "kitty.h"

namespace kitty {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks the fixed parameters; max_group > 0 also bounds the query group Hq/Hkv
// (the calls that attend).
inline int check_cfg(const kitty_cfg* c, int max_group = 0) {
  if (c == nullptr) return KITTY_ERR_INVALID_ARG;
  if (c->num_kv_heads <= 0 || c->num_q_heads <= 0 || c->num_q_heads % c->num_kv_heads != 0)
    return KITTY_ERR_INVALID_ARG;
  if (c->n_hi < 0 || c->n_hi > 128) return KITTY_ERR_INVALID_ARG;
  // Key planes: (hi_bit, lo_bit) = (4, 2), two 2-bit planes, or (8, 4), two 4-bit planes
  const bool bits_ok = (c->hi_bit == 4 && c->lo_bit == 2) || (c->hi_bit == 8 && c->lo_bit == 4);
  if (c->head_dim != 128 || c->page_tokens != 32 || !bits_ok || c->v_group != 32 ||
      c->n_hi % 16 != 0)
    return KITTY_ERR_UNSUPPORTED;
  // Value codes: 2-bit (0 = the default), or 4-bit with 4-bit Key planes
  if (c->v_bit != 0 && c->v_bit != 2 && !(c->v_bit == 4 && c->lo_bit == 4))
    return KITTY_ERR_UNSUPPORTED;
  if (c->rank_mode != KITTY_RANK_PAGE && c->rank_mode != KITTY_RANK_RUNNING &&
      c->rank_mode != KITTY_RANK_SEQUENCE)
    return KITTY_ERR_INVALID_ARG;
  if (c->in_dtype != KITTY_F16 && c->in_dtype != KITTY_BF16) return KITTY_ERR_INVALID_ARG;
  if (c->decode_pages_per_split < 0 || c->decode_total_pages < 0 || c->decode_max_pages < 0 ||
      c->decode_wait_polls < 0)
    return KITTY_ERR_INVALID_ARG;
  if (max_group > 0 && c->num_q_heads / c->num_kv_heads > max_group) return KITTY_ERR_UNSUPPORTED;
  return KITTY_OK;
}

#ifdef __CUDACC__
// Streaming multiprocessors of the current device (148 if it cannot be read);
// for the CUDA translation units (host.cpp is built without the CUDA headers).
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}
#endif

// Value code width of a configuration: 2 or 4.
inline int v_bits(const kitty_cfg* c) { return c->v_bit == 4 ? 4 : 2; }

// Bytes of one (page, kv-head) blob; w = lo_bit (Key plane width, 2 or 4),
// v = Value code width (2 or 4).
inline size_t blob_bytes(int n_hi, int w, int v) {
  return 512u * (size_t)w + 4u * (size_t)w * (size_t)n_hi + (size_t)n_hi + 512u * (size_t)v + 1024u;
}

}  // namespace kitty
