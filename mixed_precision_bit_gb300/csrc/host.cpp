// Host-side parts of the Kitty library: version, page sizes, effective bits and
// the physical page allocator (a PagedAttention-style free list of page ids).
#include <new>
#include <vector>

#include "host_common.h"
#include "kitty.h"

using kitty::blob_bytes;
using kitty::check_cfg;

struct kitty_alloc {
  int32_t num_pages;
  std::vector<int32_t> free_list;  // stack: back() is handed out next
  std::vector<uint8_t> in_use;
};

extern "C" int kitty_abi_version(void) { return 5; }

extern "C" int kitty_page_bytes(const kitty_cfg* cfg, size_t* per_head_blob, size_t* per_page) {
  const int rc = check_cfg(cfg);
  if (rc != KITTY_OK) return rc;
  const size_t b = blob_bytes(cfg->n_hi, cfg->lo_bit, kitty::v_bits(cfg));
  if (per_head_blob) *per_head_blob = b;
  if (per_page) *per_page = b * (size_t)cfg->num_kv_heads;
  return KITTY_OK;
}

// hi_fraction * hi_bit + (1 - hi_fraction) * lo_bit, hi_fraction = n_hi / D.
extern "C" float kitty_avg_bits(const kitty_cfg* cfg) {
  if (check_cfg(cfg) != KITTY_OK) return -1.0f;
  const double hf = (double)cfg->n_hi / cfg->head_dim;
  return (float)(hf * cfg->hi_bit + (1.0 - hf) * cfg->lo_bit);
}

extern "C" int kitty_alloc_create(int32_t num_pages, kitty_alloc** out) {
  if (num_pages < 0 || out == nullptr) return KITTY_ERR_INVALID_ARG;
  kitty_alloc* a = new (std::nothrow) kitty_alloc;
  if (a == nullptr) return KITTY_ERR_OOM;
  a->num_pages = num_pages;
  a->free_list.resize(num_pages);
  for (int32_t i = 0; i < num_pages; ++i) a->free_list[i] = num_pages - 1 - i;
  a->in_use.assign(num_pages, 0);
  *out = a;
  return KITTY_OK;
}

extern "C" int kitty_alloc_pages(kitty_alloc* a, int32_t n, int32_t* ids_out) {
  if (a == nullptr || n < 0 || (n > 0 && ids_out == nullptr)) return KITTY_ERR_INVALID_ARG;
  if ((size_t)n > a->free_list.size()) return KITTY_ERR_OOM;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = a->free_list.back();
    a->free_list.pop_back();
    a->in_use[id] = 1;
    ids_out[i] = id;
  }
  return KITTY_OK;
}

extern "C" int kitty_free_pages(kitty_alloc* a, int32_t n, const int32_t* ids) {
  if (a == nullptr || n < 0 || (n > 0 && ids == nullptr)) return KITTY_ERR_INVALID_ARG;
  std::vector<uint8_t> seen(a->num_pages, 0);
  for (int32_t i = 0; i < n; ++i) {  // validate everything before changing anything
    const int32_t id = ids[i];
    if (id < 0 || id >= a->num_pages || !a->in_use[id] || seen[id]) return KITTY_ERR_INVALID_ARG;
    seen[id] = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    a->in_use[ids[i]] = 0;
    a->free_list.push_back(ids[i]);
  }
  return KITTY_OK;
}

extern "C" int32_t kitty_alloc_free_count(const kitty_alloc* a) {
  return a == nullptr ? -1 : (int32_t)a->free_list.size();
}

extern "C" void kitty_alloc_destroy(kitty_alloc* a) { delete a; }
