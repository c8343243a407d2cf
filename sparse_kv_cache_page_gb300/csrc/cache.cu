// KV cache manager around the page-retrieval path.
//
// WorldAttention (review page), HKV section and Fig. 2: the KV of past chunks
// lives in pages of 8 frames; L1 (GPU HBM) holds the pages in use plus the
// page summaries and prompt embeddings ("page indices"), L2 (CPU DRAM) the
// pages not in use; frequently used pages stay on the GPU, the rest are
// offloaded, so HBM occupancy stays bounded however long the video grows.
// Inferix (summary page), KV Cache Manager: append a clean block's KV, range
// (window) access, index-based selective fetch, offload to main memory.
//
// Host-side runtime (no kernels of its own):
//   * page table: logical page p (chunk p / ppc) -> tier (HBM / DRAM) and slot;
//   * HBM tier: one device pool of hbm_pages page slots (K and V); DRAM tier:
//     one pinned pool of host_pages slots; summaries [max pages][H][d] and
//     prompt embeddings [max chunks][prompt_dim] stay in HBM for every page;
//   * append: the chunk's pages go to free HBM slots; when none is free the
//     least recently used resident page moves to the DRAM tier (copy engine);
//     page summaries are computed at insert (wa_page_summarize on the chunk);
//   * retrieve: prompt stage + page stage over the summaries (wa_select_pages),
//     the K_p indices to the host (one stream synchronisation), each selected
//     page copied into the caller's buffer from its tier; a page fetched from
//     DRAM is promoted back to HBM, swapping with the least recently used page
//     not selected in this retrieval;
//   * window: the last n tokens of the sequence, contiguous, from either tier.
// The least-recently-used clock ticks once per append and per retrieval.
// dry_run caches do no CUDA work at all: moves are planned and counted, so
// the placement policy can be exercised without a GPU.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "wa_internal.cuh"

struct wa_cache {
  wa_cache_config cfg;
  size_t page_bytes = 0;          // one tensor (K or V) of one page
  int n_pages = 0, n_chunks = 0;
  unsigned long long clock = 0;
  struct Entry {
    int tier;                     // 0 HBM, 1 DRAM
    int slot;
    unsigned long long last_use;
  };
  std::vector<Entry> table;       // by logical page
  std::vector<int> hbm_owner;     // slot -> page or -1
  std::vector<int> host_owner;
  char* hbm_k = nullptr;
  char* hbm_v = nullptr;
  char* host_k = nullptr;
  char* host_v = nullptr;
  float* kbar = nullptr;          // [max_pages][H][d]
  float* prompts = nullptr;       // [max_chunks][prompt_dim]
  int32_t* idx_dev = nullptr;     // [k_p max]
  int32_t* idx_host = nullptr;    // pinned
  int idx_cap = 0;
  wa_cache_stats stats{};
};

namespace {

using wa::cuda_status;

inline bool dt_ok(wa_dtype dt) { return dt == WA_BF16 || dt == WA_F32; }
inline size_t dt_size(wa_dtype dt) { return dt == WA_BF16 ? 2 : 4; }

int free_slot(const std::vector<int>& owner) {
  for (size_t s = 0; s < owner.size(); ++s)
    if (owner[s] < 0) return (int)s;
  return -1;
}

// Least recently used page in `tier`, skipping pages marked in `keep`
// (ties to the lower page number).
int lru_page(const wa_cache* c, int tier, const std::vector<char>* keep) {
  int best = -1;
  for (int p = 0; p < c->n_pages; ++p) {
    const wa_cache::Entry& e = c->table[p];
    if (e.tier != tier || (keep && (*keep)[p])) continue;
    if (best < 0 || e.last_use < c->table[best].last_use) best = p;
  }
  return best;
}

char* tier_ptr(wa_cache* c, int tier, int slot, bool v) {
  char* base = tier == 0 ? (v ? c->hbm_v : c->hbm_k) : (v ? c->host_v : c->host_k);
  return base + (size_t)slot * c->page_bytes;
}

wa_status copy_page(wa_cache* c, void* dst, const void* src, cudaMemcpyKind kind, cudaStream_t s) {
  if (c->cfg.dry_run) return WA_OK;
  return cuda_status(cudaMemcpyAsync(dst, src, c->page_bytes, kind, s));
}

void count_bytes(wa_cache* c, cudaMemcpyKind kind, size_t bytes) {
  if (kind == cudaMemcpyHostToDevice) c->stats.bytes_h2d += (long long)bytes;
  else if (kind == cudaMemcpyDeviceToHost) c->stats.bytes_d2h += (long long)bytes;
  else c->stats.bytes_d2d += (long long)bytes;
}

// Move page p from HBM to a free DRAM slot (K and V).
wa_status offload(wa_cache* c, int p, cudaStream_t s) {
  const int hs = free_slot(c->host_owner);
  if (hs < 0) return WA_ERR_OOM;
  wa_cache::Entry& e = c->table[p];
  for (int t = 0; t < 2; ++t) {
    wa_status rc = copy_page(c, tier_ptr(c, 1, hs, t), tier_ptr(c, 0, e.slot, t),
                             cudaMemcpyDeviceToHost, s);
    if (rc != WA_OK) return rc;
    count_bytes(c, cudaMemcpyDeviceToHost, c->page_bytes);
  }
  c->hbm_owner[e.slot] = -1;
  c->host_owner[hs] = p;
  e.tier = 1;
  e.slot = hs;
  c->stats.offloads++;
  return WA_OK;
}

// A free HBM slot, offloading the least recently used resident page (not in
// `keep`) when none is free.
wa_status hbm_slot(wa_cache* c, const std::vector<char>* keep, cudaStream_t s, int* slot) {
  int hs = free_slot(c->hbm_owner);
  if (hs < 0) {
    const int victim = lru_page(c, 0, keep);
    if (victim < 0) return WA_ERR_OOM;
    const int vslot = c->table[victim].slot;
    wa_status rc = offload(c, victim, s);
    if (rc != WA_OK) return rc;
    hs = vslot;
  }
  *slot = hs;
  return WA_OK;
}

// Promote page p (in DRAM) into HBM: the least recently used resident page
// not in `keep` moves to DRAM first when HBM is full.  When the page's K and V
// are already on the device (from_k, from_v: the caller's retrieval buffer,
// filled earlier on the same stream) its DRAM slot is released first, so the
// evicted page can take it (a swap); otherwise the page is copied from DRAM.
wa_status promote(wa_cache* c, int p, const std::vector<char>& keep, const char* from_k,
                  const char* from_v, cudaStream_t s) {
  wa_cache::Entry& e = c->table[p];
  const int old_host = e.slot;
  const bool on_device = (from_k && from_v) || c->cfg.dry_run;
  if (on_device) c->host_owner[old_host] = -1;
  int hs = -1;
  wa_status rc = hbm_slot(c, &keep, s, &hs);
  if (rc != WA_OK) return rc;
  for (int t = 0; t < 2; ++t) {
    const char* src = on_device ? (t ? from_v : from_k) : tier_ptr(c, 1, old_host, t);
    const cudaMemcpyKind kind = on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    rc = copy_page(c, tier_ptr(c, 0, hs, t), src, kind, s);
    if (rc != WA_OK) return rc;
    count_bytes(c, kind, c->page_bytes);
  }
  if (!on_device) c->host_owner[old_host] = -1;
  c->hbm_owner[hs] = p;
  e.tier = 0;
  e.slot = hs;
  c->stats.promotions++;
  return WA_OK;
}

void release(wa_cache* c) {
  if (!c->cfg.dry_run) {
    cudaFree(c->hbm_k);
    cudaFree(c->hbm_v);
    cudaFreeHost(c->host_k);
    cudaFreeHost(c->host_v);
    cudaFree(c->kbar);
    cudaFree(c->prompts);
    cudaFree(c->idx_dev);
    cudaFreeHost(c->idx_host);
  }
  delete c;
}

}  // namespace

extern "C" {

wa_status wa_cache_create(const wa_cache_config* cfg, wa_cache** out) {
  if (!cfg || !out) return WA_ERR_INVALID_ARG;
  *out = nullptr;
  const wa_cache_config& g = *cfg;
  if (!dt_ok(g.dtype)) return WA_ERR_DTYPE;
  if (g.n_heads <= 0 || g.head_dim <= 0 || g.page_tokens <= 0 || g.pages_per_chunk <= 0 ||
      g.hbm_pages <= 0 || g.host_pages < 0 || g.max_chunks <= 0 || g.prompt_dim < 0)
    return WA_ERR_INVALID_ARG;
  if (((long long)g.n_heads * g.head_dim * dt_size(g.dtype)) % 16 != 0) return WA_ERR_SHAPE;
  wa_cache* c = new (std::nothrow) wa_cache();
  if (!c) return WA_ERR_OOM;
  c->cfg = g;
  c->page_bytes = (size_t)g.page_tokens * g.n_heads * g.head_dim * dt_size(g.dtype);
  c->hbm_owner.assign(g.hbm_pages, -1);
  c->host_owner.assign(g.host_pages, -1);
  c->table.reserve((size_t)g.max_chunks * g.pages_per_chunk);
  if (!g.dry_run) {
    const size_t max_pages = (size_t)g.max_chunks * g.pages_per_chunk;
    bool ok = cudaMalloc(&c->hbm_k, c->page_bytes * g.hbm_pages) == cudaSuccess &&
              cudaMalloc(&c->hbm_v, c->page_bytes * g.hbm_pages) == cudaSuccess &&
              cudaMalloc(&c->kbar, max_pages * g.n_heads * g.head_dim * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&c->prompts, (size_t)g.max_chunks * (g.prompt_dim > 0 ? g.prompt_dim : 1) *
                                          sizeof(float)) == cudaSuccess;
    if (ok && g.host_pages > 0)
      ok = cudaHostAlloc((void**)&c->host_k, c->page_bytes * g.host_pages, cudaHostAllocDefault) ==
               cudaSuccess &&
           cudaHostAlloc((void**)&c->host_v, c->page_bytes * g.host_pages, cudaHostAllocDefault) ==
               cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      release(c);
      return WA_ERR_OOM;
    }
  }
  *out = c;
  return WA_OK;
}

wa_status wa_cache_destroy(wa_cache* c) {
  if (!c) return WA_ERR_INVALID_ARG;
  if (!c->cfg.dry_run) cudaDeviceSynchronize();
  release(c);
  return WA_OK;
}

wa_status wa_cache_reset(wa_cache* c) {
  if (!c) return WA_ERR_INVALID_ARG;
  if (!c->cfg.dry_run) cudaDeviceSynchronize();   // no copy may still read or write a slot
  c->table.clear();
  std::fill(c->hbm_owner.begin(), c->hbm_owner.end(), -1);
  std::fill(c->host_owner.begin(), c->host_owner.end(), -1);
  c->n_pages = 0;
  c->n_chunks = 0;
  c->clock = 0;
  c->stats = wa_cache_stats{};
  return WA_OK;
}

wa_status wa_cache_append_chunk(wa_cache* c, const void* k, const void* v, const float* prompt,
                                wa_stream_t stream) {
  if (!c) return WA_ERR_INVALID_ARG;
  const wa_cache_config& g = c->cfg;
  if (!g.dry_run && (!k || !v)) return WA_ERR_INVALID_ARG;
  if (g.prompt_dim > 0 && !g.dry_run && !prompt) return WA_ERR_INVALID_ARG;
  if (c->n_chunks >= g.max_chunks) return WA_ERR_OOM;
  if ((long long)c->n_pages + g.pages_per_chunk > (long long)g.hbm_pages + g.host_pages)
    return WA_ERR_OOM;
  cudaStream_t s = (cudaStream_t)stream;
  c->clock++;
  const int p0 = c->n_pages;
  if (!g.dry_run) {
    // summaries at insert, straight from the appended chunk (page-major, contiguous)
    wa_status rc = wa_page_summarize(k, g.dtype, g.pages_per_chunk, g.page_tokens, g.n_heads,
                                     g.head_dim, c->kbar + (size_t)p0 * g.n_heads * g.head_dim,
                                     stream);
    if (rc != WA_OK) return rc;
    if (g.prompt_dim > 0 &&
        cudaMemcpyAsync(c->prompts + (size_t)c->n_chunks * g.prompt_dim, prompt,
                        (size_t)g.prompt_dim * sizeof(float), cudaMemcpyDeviceToDevice,
                        s) != cudaSuccess)
      return WA_ERR_CUDA;
  }
  // the new chunk's pages are the most recent: none of them is an eviction victim
  std::vector<char> keep(p0 + g.pages_per_chunk, 0);
  for (int j = 0; j < g.pages_per_chunk; ++j) {
    const int p = p0 + j;
    c->table.push_back({-1, -1, c->clock});
    c->n_pages = p + 1;
    keep[p] = 1;
    int hs = -1;
    wa_status rc = hbm_slot(c, &keep, s, &hs);
    if (rc != WA_OK) return rc;
    for (int t = 0; t < 2; ++t) {
      const char* src = static_cast<const char*>(t ? v : k);
      rc = copy_page(c, tier_ptr(c, 0, hs, t), src ? src + (size_t)j * c->page_bytes : nullptr,
                     cudaMemcpyDeviceToDevice, s);
      if (rc != WA_OK) return rc;
      count_bytes(c, cudaMemcpyDeviceToDevice, c->page_bytes);
    }
    c->hbm_owner[hs] = p;
    c->table[p].tier = 0;
    c->table[p].slot = hs;
  }
  c->n_chunks++;
  return WA_OK;
}

// Mark pages as used by one retrieval: LRU update, and pages in DRAM promoted to HBM.
static wa_status use_pages(wa_cache* c, const int32_t* pages, int n, const char* const* dev_k,
                           const char* const* dev_v, cudaStream_t s) {
  c->clock++;
  std::vector<char> keep(c->n_pages, 0);
  for (int i = 0; i < n; ++i) {
    if (pages[i] < 0 || pages[i] >= c->n_pages) return WA_ERR_INDEX;
    keep[pages[i]] = 1;
  }
  for (int i = 0; i < n; ++i) {
    wa_cache::Entry& e = c->table[pages[i]];
    e.last_use = c->clock;
    if (e.tier == 1) {
      wa_status rc = promote(c, pages[i], keep, dev_k ? dev_k[i] : nullptr,
                             dev_v ? dev_v[i] : nullptr, s);
      if (rc != WA_OK) return rc;
    }
  }
  return WA_OK;
}

wa_status wa_cache_touch(wa_cache* c, const int32_t* pages, int n) {
  if (!c || (!pages && n > 0) || n < 0) return WA_ERR_INVALID_ARG;
  if (!c->cfg.dry_run) return WA_ERR_INVALID_ARG;
  return use_pages(c, pages, n, nullptr, nullptr, nullptr);
}

wa_status wa_cache_retrieve(wa_cache* c, const void* q, int n_q, const float* prompt_cur, int k_p,
                            void* k_buf, void* v_buf, int32_t* idx_out, wa_stream_t stream) {
  if (!c || !q || !k_buf || !v_buf || !idx_out || n_q <= 0 || k_p <= 0) return WA_ERR_INVALID_ARG;
  if (c->cfg.dry_run) return WA_ERR_INVALID_ARG;
  const wa_cache_config& g = c->cfg;
  if (c->n_pages == 0) return WA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (c->idx_cap < k_p) {
    if (c->idx_dev) {
      cudaFree(c->idx_dev);
      cudaFreeHost(c->idx_host);
      c->idx_dev = nullptr;
      c->idx_host = nullptr;
    }
    if (cudaMalloc(&c->idx_dev, k_p * sizeof(int32_t)) != cudaSuccess ||
        cudaHostAlloc((void**)&c->idx_host, k_p * sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess) {
      cudaGetLastError();
      c->idx_cap = 0;
      return WA_ERR_OOM;
    }
    c->idx_cap = k_p;
  }
  const bool prompts = g.prompt_dim > 0 && prompt_cur;
  wa_status rc = wa_select_pages(q, g.dtype, n_q, g.n_heads, g.head_dim, c->kbar, c->n_pages,
                                 prompts ? prompt_cur : nullptr, prompts ? c->prompts : nullptr,
                                 prompts ? c->n_chunks : 0, g.prompt_dim, g.pages_per_chunk, k_p,
                                 c->idx_dev, nullptr, nullptr, stream);
  if (rc != WA_OK) return rc;
  if (cudaMemcpyAsync(c->idx_host, c->idx_dev, k_p * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return WA_ERR_CUDA;
  memcpy(idx_out, c->idx_host, k_p * sizeof(int32_t));
  std::vector<const char*> dk(k_p), dv(k_p);
  for (int i = 0; i < k_p; ++i) {
    const int p = idx_out[i];
    if (p < 0 || p >= c->n_pages) return WA_ERR_INDEX;
    const wa_cache::Entry& e = c->table[p];
    char* dst_k = static_cast<char*>(k_buf) + (size_t)i * c->page_bytes;
    char* dst_v = static_cast<char*>(v_buf) + (size_t)i * c->page_bytes;
    const cudaMemcpyKind kind = e.tier == 0 ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    rc = copy_page(c, dst_k, tier_ptr(c, e.tier, e.slot, false), kind, s);
    if (rc == WA_OK) rc = copy_page(c, dst_v, tier_ptr(c, e.tier, e.slot, true), kind, s);
    if (rc != WA_OK) return rc;
    count_bytes(c, kind, 2 * c->page_bytes);
    dk[i] = dst_k;
    dv[i] = dst_v;
  }
  // pages that came from DRAM are promoted from the caller's buffer (device to device)
  return use_pages(c, idx_out, k_p, dk.data(), dv.data(), s);
}

wa_status wa_cache_window(wa_cache* c, int n_tokens, void* k_out, void* v_out, wa_stream_t stream) {
  if (!c || !k_out || !v_out || n_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (c->cfg.dry_run) return WA_ERR_INVALID_ARG;
  const wa_cache_config& g = c->cfg;
  const long long total = (long long)c->n_pages * g.page_tokens;
  if (n_tokens > total) return WA_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t row = c->page_bytes / g.page_tokens;
  long long first = total - n_tokens;                 // first token of the window
  size_t out_off = 0;
  for (int p = (int)(first / g.page_tokens); p < c->n_pages; ++p) {
    const long long t0 = std::max(first, (long long)p * g.page_tokens) - (long long)p * g.page_tokens;
    const size_t bytes = (size_t)(g.page_tokens - t0) * row;
    const wa_cache::Entry& e = c->table[p];
    const cudaMemcpyKind kind = e.tier == 0 ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    for (int t = 0; t < 2; ++t) {
      if (cudaMemcpyAsync(static_cast<char*>(t ? v_out : k_out) + out_off,
                          tier_ptr(c, e.tier, e.slot, t) + (size_t)t0 * row, bytes, kind, s) !=
          cudaSuccess)
        return WA_ERR_CUDA;
    }
    count_bytes(c, kind, 2 * bytes);
    out_off += bytes;
  }
  return WA_OK;
}

wa_status wa_cache_page_location(const wa_cache* c, int page, int* tier, int* slot) {
  if (!c || !tier || !slot) return WA_ERR_INVALID_ARG;
  if (page < 0 || page >= c->n_pages) return WA_ERR_INDEX;
  *tier = c->table[page].tier;
  *slot = c->table[page].slot;
  return WA_OK;
}

wa_status wa_cache_get_stats(const wa_cache* c, wa_cache_stats* out) {
  if (!c || !out) return WA_ERR_INVALID_ARG;
  *out = c->stats;
  out->n_pages = c->n_pages;
  out->n_chunks = c->n_chunks;
  out->in_hbm = 0;
  out->in_host = 0;
  for (int p = 0; p < c->n_pages; ++p) (c->table[p].tier == 0 ? out->in_hbm : out->in_host)++;
  return WA_OK;
}

}  // extern "C"
