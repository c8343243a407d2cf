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
// Host-side runtime around a few kernels of the library:
//   * page table: logical page p (chunk p / ppc) -> HBM slot and/or DRAM slot.
//     The DRAM tier is inclusive: pages never change once appended, so a
//     page's DRAM copy stays valid after it is promoted back to HBM, and
//     evicting such a page again moves no bytes;
//   * HBM tier: one device pool of hbm_pages page slots (K and V); DRAM tier:
//     one pinned, device-mapped pool of host_pages slots, holding the cache's
//     dtype, FP8 E4M3 codes plus per-(token, head) scales, or NVFP4 (E2M1 codes,
//     E4M3 scales per 16 values, fp32 row scales) -- dram_format, the
//     compressed tier: 1.9x or 3.4x fewer bytes across the CPU-GPU link;
//     summaries [max pages][H][d] and prompt embeddings [max chunks][prompt_dim]
//     stay in HBM for every page;
//   * append: the chunk's pages go to free HBM slots; when none is free the
//     least recently used resident page leaves HBM -- with no copy when it
//     already has a DRAM copy, else offloaded to a free DRAM slot (or to one
//     reclaimed from the most recently used page that holds both copies);
//     page summaries are computed at insert (wa_page_summarize on the chunk);
//   * offloads overlap the caller's work: the victim is copied (or FP8-encoded)
//     into a device staging ring on the caller's stream, which then reuses the
//     HBM slot at once, and an internal copy stream moves the staging slot to
//     DRAM.  Events order every reuse: a staging slot is rewritten only after
//     its copy to DRAM finished, a DRAM slot is read only after its copy
//     landed, and each copy to DRAM starts after the caller's stream reached
//     the staging write (so after every earlier read of the DRAM slot);
//   * retrieve: prompt stage + page stage over the summaries (wa_select_pages),
//     the K_p indices written to mapped host memory (one stream
//     synchronisation, no copy-engine transfer to queue behind offloads), each selected
//     page copied into the caller's buffer from its tier (compressed DRAM pages
//     first copied whole by the copy engine, then decoded from HBM); a page
//     found only in DRAM is promoted to HBM from the caller's buffer;
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
  size_t page_bytes = 0;          // one tensor (K or V) of one page in HBM
  size_t host_page_bytes = 0;     // the same in the DRAM tier (slot stride)
  size_t code_bytes = 0;          // compressed tier: codes of one page tensor, then
  size_t bs_off = 0, rs_off = 0;  // (NVFP4) block scales and row scales at these offsets
  int n_pages = 0, n_chunks = 0;
  unsigned long long clock = 0;
  struct Entry {
    int hbm;                      // HBM slot or -1
    int host;                     // DRAM slot or -1
    unsigned long long last_use;
  };
  std::vector<Entry> table;       // by logical page
  std::vector<int> hbm_owner;     // slot -> page or -1
  std::vector<int> host_owner;
  char* hbm_k = nullptr;
  char* hbm_v = nullptr;
  char* host_k = nullptr;         // pinned, device-mapped
  char* host_v = nullptr;
  char* host_k_dev = nullptr;     // their device addresses
  char* host_v_dev = nullptr;
  char* stage_k = nullptr;        // staging ring [n_stage][host_page_bytes]
  char* stage_v = nullptr;
  int n_stage = 0, next_stage = 0;
  cudaStream_t copy = nullptr;    // staging -> DRAM copies
  cudaEvent_t filled = nullptr;   // caller's stream passed a staging write
  cudaEvent_t drained = nullptr;  // copy stream passed its latest copy
  std::vector<cudaEvent_t> stage_done;  // staging slot's last copy out finished
  std::vector<cudaEvent_t> host_ready;  // DRAM slot's last copy in finished
  std::vector<char> stage_pending, host_pending;
  bool copies_issued = false;
  float* kbar = nullptr;          // [max_pages][H][d]
  float* prompts = nullptr;       // [max_chunks][prompt_dim]
  char* fetch = nullptr;          // device copies of compressed DRAM slots being decoded
  size_t fetch_cap = 0;
  int32_t* idx_host = nullptr;    // [k_p max], pinned and device-mapped
  int32_t* idx_dev = nullptr;     // its device address
  int idx_cap = 0;
  wa_cache_stats stats{};
};

namespace {

using wa::cuda_status;
using wa::fault_mode;

inline bool dt_ok(wa_dtype dt) { return dt == WA_BF16 || dt == WA_F32; }
inline size_t dt_size(wa_dtype dt) { return dt == WA_BF16 ? 2 : 4; }
inline bool fp8(const wa_cache* c) { return c->cfg.dram_format == 1; }
inline bool nvfp4(const wa_cache* c) { return c->cfg.dram_format == 2; }
inline size_t pad16(size_t n) { return (n + 15) / 16 * 16; }

int free_slot(const std::vector<int>& owner) {
  for (size_t s = 0; s < owner.size(); ++s)
    if (owner[s] < 0) return (int)s;
  return -1;
}

// Least recently used page with an HBM copy, skipping pages marked in `keep`
// (ties to the lower page number).
int lru_resident(const wa_cache* c, const std::vector<char>* keep) {
  int best = -1;
  for (int p = 0; p < c->n_pages; ++p) {
    const wa_cache::Entry& e = c->table[p];
    if (e.hbm < 0 || (keep && (*keep)[p])) continue;
    if (best < 0 || e.last_use < c->table[best].last_use) best = p;
  }
  return best;
}

char* hbm_ptr(wa_cache* c, int slot, bool v) {
  return (v ? c->hbm_v : c->hbm_k) + (size_t)slot * c->page_bytes;
}
char* host_ptr(wa_cache* c, int slot, bool v, bool device_address) {
  char* base = device_address ? (v ? c->host_v_dev : c->host_k_dev) : (v ? c->host_v : c->host_k);
  return base + (size_t)slot * c->host_page_bytes;
}

void count_bytes(wa_cache* c, cudaMemcpyKind kind, size_t bytes) {
  if (kind == cudaMemcpyHostToDevice) c->stats.bytes_h2d += (long long)bytes;
  else if (kind == cudaMemcpyDeviceToHost) c->stats.bytes_d2h += (long long)bytes;
  else c->stats.bytes_d2d += (long long)bytes;
}

// Bytes of `rows` (token, head) rows in the DRAM tier's format.
size_t host_row_bytes(const wa_cache* c, size_t rows) {
  const size_t d = (size_t)c->cfg.head_dim;
  if (fp8(c)) return rows * (d + sizeof(float));
  if (nvfp4(c)) return rows * (d / 2 + d / 16 + sizeof(float));
  return rows * d * dt_size(c->cfg.dtype);
}

// Make `s` wait until DRAM slot x holds its latest copy.
wa_status wait_host_slot(wa_cache* c, int x, cudaStream_t s) {
  if (c->cfg.dry_run || !c->host_pending[x]) return WA_OK;
  return cuda_status(cudaStreamWaitEvent(s, c->host_ready[x], 0));
}

// A DRAM slot for an offload: a free one, else one reclaimed from the most
// recently used page holding both copies (ties: lower page), else (for a
// promotion whose data is already on the device) the promoted page's own.
int acquire_host_slot(wa_cache* c, int self_page) {
  int x = free_slot(c->host_owner);
  if (x >= 0) return x;
  int w = -1;
  for (int p = 0; p < c->n_pages; ++p) {
    const wa_cache::Entry& e = c->table[p];
    if (e.hbm >= 0 && e.host >= 0 && (w < 0 || e.last_use > c->table[w].last_use)) w = p;
  }
  if (w < 0 && self_page >= 0 && c->table[self_page].host >= 0) w = self_page;
  if (w < 0) return -1;
  x = c->table[w].host;
  c->table[w].host = -1;
  c->host_owner[x] = -1;
  c->stats.reclaims++;
  return x;
}

// Copy page v (HBM only) to DRAM slot x through the staging ring.
wa_status offload(wa_cache* c, int v, int x, cudaStream_t s) {
  wa_cache::Entry& e = c->table[v];
  if (!c->cfg.dry_run) {
    const int r = c->next_stage;
    c->next_stage = (r + 1) % c->n_stage;
    if (c->stage_pending[r] && cudaStreamWaitEvent(s, c->stage_done[r], 0) != cudaSuccess)
      return WA_ERR_CUDA;
    const size_t rows = (size_t)c->cfg.page_tokens * c->cfg.n_heads;
    for (int t = 0; t < 2; ++t) {
      char* st = (t ? c->stage_v : c->stage_k) + (size_t)r * c->host_page_bytes;
      wa_status rc;
      if (fp8(c))
        rc = wa::launch_fp8_encode(hbm_ptr(c, e.hbm, t), rows, c->cfg.head_dim, st,
                                   reinterpret_cast<float*>(st + c->code_bytes), s);
      else if (nvfp4(c))
        rc = wa::launch_nvfp4_encode(hbm_ptr(c, e.hbm, t), rows, c->cfg.head_dim, st,
                                     st + c->bs_off, reinterpret_cast<float*>(st + c->rs_off), s);
      else
        rc = cuda_status(cudaMemcpyAsync(st, hbm_ptr(c, e.hbm, t), c->page_bytes,
                                         cudaMemcpyDeviceToDevice, s));
      if (rc != WA_OK) return rc;
    }
    if (cudaEventRecord(c->filled, s) != cudaSuccess ||
        cudaStreamWaitEvent(c->copy, c->filled, 0) != cudaSuccess)
      return WA_ERR_CUDA;
    for (int t = 0; t < 2; ++t) {
      const char* st = (t ? c->stage_v : c->stage_k) + (size_t)r * c->host_page_bytes;
      if (cudaMemcpyAsync(host_ptr(c, x, t, false), st, c->host_page_bytes,
                          cudaMemcpyDeviceToHost, c->copy) != cudaSuccess)
        return WA_ERR_CUDA;
    }
    if (cudaEventRecord(c->stage_done[r], c->copy) != cudaSuccess ||
        cudaEventRecord(c->host_ready[x], c->copy) != cudaSuccess)
      return WA_ERR_CUDA;
    c->stage_pending[r] = 1;
    c->host_pending[x] = 1;
    c->copies_issued = true;
  }
  count_bytes(c, cudaMemcpyDeviceToHost, 2 * c->host_page_bytes);
  c->host_owner[x] = v;
  e.host = x;
  c->stats.offloads++;
  return WA_OK;
}

// Take page v out of HBM (its slot is then free).
wa_status evict(wa_cache* c, int v, int self_page, cudaStream_t s) {
  wa_cache::Entry& e = c->table[v];
  if (e.host >= 0) {
    c->stats.evictions++;
  } else {
    const int x = acquire_host_slot(c, self_page);
    if (x < 0) return WA_ERR_OOM;
    wa_status rc = offload(c, v, x, s);
    if (rc != WA_OK) return rc;
  }
  c->hbm_owner[e.hbm] = -1;
  e.hbm = -1;
  return WA_OK;
}

// A free HBM slot, evicting the least recently used resident page (not in
// `keep`) when none is free.
wa_status hbm_slot(wa_cache* c, const std::vector<char>* keep, int self_page, cudaStream_t s,
                   int* slot) {
  int hs = free_slot(c->hbm_owner);
  if (hs < 0) {
    const int victim = lru_resident(c, keep);
    if (victim < 0) return WA_ERR_OOM;
    hs = c->table[victim].hbm;
    wa_status rc = evict(c, victim, self_page, s);
    if (rc != WA_OK) return rc;
  }
  *slot = hs;
  return WA_OK;
}

// Promote page p (DRAM only) into HBM from its copy in the caller's buffer
// (from_k, from_v: filled earlier on the same stream).  Its DRAM copy stays.
wa_status promote(wa_cache* c, int p, const std::vector<char>& keep, const char* from_k,
                  const char* from_v, cudaStream_t s) {
  int hs = -1;
  wa_status rc = hbm_slot(c, &keep, p, s, &hs);
  if (rc != WA_OK) return rc;
  if (!c->cfg.dry_run) {
    for (int t = 0; t < 2; ++t)
      if (cudaMemcpyAsync(hbm_ptr(c, hs, t), t ? from_v : from_k, c->page_bytes,
                          cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return WA_ERR_CUDA;
  }
  count_bytes(c, cudaMemcpyDeviceToDevice, 2 * c->page_bytes);
  c->hbm_owner[hs] = p;
  c->table[p].hbm = hs;
  c->stats.promotions++;
  return WA_OK;
}

inline bool compressed(const wa_cache* c) { return fp8(c) || nvfp4(c); }

// A device buffer of at least `bytes` for compressed DRAM slots.
wa_status ensure_fetch(wa_cache* c, size_t bytes) {
  if (c->fetch_cap >= bytes) return WA_OK;
  if (fault_mode() == WA_FAULT_ALLOC) return WA_ERR_OOM;
  if (c->fetch) {
    cudaDeviceSynchronize();             // no decode may still read the old buffer
    cudaFree(c->fetch);
    c->fetch = nullptr;
    c->fetch_cap = 0;
  }
  if (cudaMalloc(&c->fetch, bytes) != cudaSuccess) {
    cudaGetLastError();
    return WA_ERR_OOM;
  }
  c->fetch_cap = bytes;
  return WA_OK;
}

// Copy the compressed DRAM slot of page p's K (v = 0) or V into fetch slot f.
wa_status fetch_slot(wa_cache* c, int p, bool v, int f, cudaStream_t s) {
  const wa_cache::Entry& e = c->table[p];
  wa_status rc = wait_host_slot(c, e.host, s);
  if (rc != WA_OK) return rc;
  count_bytes(c, cudaMemcpyHostToDevice, c->host_page_bytes);
  return cuda_status(cudaMemcpyAsync(c->fetch + (size_t)f * c->host_page_bytes,
                                     host_ptr(c, e.host, v, false), c->host_page_bytes,
                                     cudaMemcpyHostToDevice, s));
}

// Decode rows [r0, r0 + rows) of the compressed slot held in fetch slot f into dst.
wa_status decode_fetched(wa_cache* c, int f, size_t r0, size_t rows, char* dst, cudaStream_t s) {
  const size_t d = (size_t)c->cfg.head_dim;
  const char* base = c->fetch + (size_t)f * c->host_page_bytes;
  if (fp8(c))
    return wa::launch_fp8_decode(base + r0 * d, reinterpret_cast<const float*>(base + c->code_bytes) + r0,
                                 nullptr, 1, rows, rows, c->cfg.head_dim, dst, s);
  return wa::launch_nvfp4_decode(base + r0 * (d / 2), base + c->bs_off + r0 * (d / 16),
                                 reinterpret_cast<const float*>(base + c->rs_off) + r0, nullptr, 1,
                                 rows, rows, c->cfg.head_dim, dst, s);
}

// Copy `rows` (token, head) rows of page p, starting at row r0, into dst
// (K or V) from the page's HBM copy if it has one, else from DRAM (a
// compressed slot through fetch slot f).
wa_status read_page(wa_cache* c, int p, bool v, size_t r0, size_t rows, char* dst,
                    cudaStream_t s, int f = 0) {
  const wa_cache::Entry& e = c->table[p];
  const size_t row_bytes = (size_t)c->cfg.head_dim * dt_size(c->cfg.dtype);
  if (e.hbm >= 0) {
    count_bytes(c, cudaMemcpyDeviceToDevice, rows * row_bytes);
    return cuda_status(cudaMemcpyAsync(dst, hbm_ptr(c, e.hbm, v) + r0 * row_bytes,
                                       rows * row_bytes, cudaMemcpyDeviceToDevice, s));
  }
  if (compressed(c)) {
    wa_status rc = ensure_fetch(c, (size_t)(f + 1) * c->host_page_bytes);
    if (rc == WA_OK) rc = fetch_slot(c, p, v, f, s);
    if (rc == WA_OK) rc = decode_fetched(c, f, r0, rows, dst, s);
    return rc;
  }
  wa_status rc = wait_host_slot(c, e.host, s);
  if (rc != WA_OK) return rc;
  count_bytes(c, cudaMemcpyHostToDevice, host_row_bytes(c, rows));
  return cuda_status(cudaMemcpyAsync(dst, host_ptr(c, e.host, v, false) + r0 * row_bytes,
                                     rows * row_bytes, cudaMemcpyHostToDevice, s));
}

void release(wa_cache* c) {
  if (!c->cfg.dry_run) {
    cudaFree(c->hbm_k);
    cudaFree(c->hbm_v);
    cudaFree(c->stage_k);
    cudaFree(c->stage_v);
    cudaFreeHost(c->host_k);
    cudaFreeHost(c->host_v);
    cudaFree(c->kbar);
    cudaFree(c->prompts);
    cudaFree(c->fetch);
    cudaFreeHost(c->idx_host);
    for (cudaEvent_t ev : c->stage_done) cudaEventDestroy(ev);
    for (cudaEvent_t ev : c->host_ready) cudaEventDestroy(ev);
    if (c->filled) cudaEventDestroy(c->filled);
    if (c->drained) cudaEventDestroy(c->drained);
    if (c->copy) cudaStreamDestroy(c->copy);
  }
  delete c;
}

bool make_events(std::vector<cudaEvent_t>* evs, int n) {
  evs->reserve(n);
  for (int i = 0; i < n; ++i) {
    cudaEvent_t ev = nullptr;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return false;
    evs->push_back(ev);
  }
  return true;
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
  if (g.dram_format < 0 || g.dram_format > 2) return WA_ERR_INVALID_ARG;
  if (g.dram_format != 0) {
    if (g.dtype != WA_BF16) return WA_ERR_DTYPE;
    if (g.head_dim != 64 && g.head_dim != 128 && g.head_dim != 256) return WA_ERR_SHAPE;
  }
  wa_cache* c = new (std::nothrow) wa_cache();
  if (!c) return WA_ERR_OOM;
  c->cfg = g;
  const size_t rows = (size_t)g.page_tokens * g.n_heads;
  c->page_bytes = rows * g.head_dim * dt_size(g.dtype);
  if (g.dram_format == 1) {
    c->code_bytes = rows * g.head_dim;
    c->host_page_bytes = c->code_bytes + pad16(rows * sizeof(float));
  } else if (g.dram_format == 2) {
    c->code_bytes = rows * (g.head_dim / 2);
    c->bs_off = c->code_bytes;
    c->rs_off = c->bs_off + pad16(rows * (g.head_dim / 16));
    c->host_page_bytes = c->rs_off + pad16(rows * sizeof(float));
  } else {
    c->host_page_bytes = c->page_bytes;
  }
  c->hbm_owner.assign(g.hbm_pages, -1);
  c->host_owner.assign(g.host_pages, -1);
  c->table.reserve((size_t)g.max_chunks * g.pages_per_chunk);
  if (!g.dry_run) {
    const size_t max_pages = (size_t)g.max_chunks * g.pages_per_chunk;
    c->n_stage = g.host_pages > 0 ? g.pages_per_chunk + 4 : 0;
    bool ok = fault_mode() != WA_FAULT_ALLOC &&
              cudaMalloc(&c->hbm_k, c->page_bytes * g.hbm_pages) == cudaSuccess &&
              cudaMalloc(&c->hbm_v, c->page_bytes * g.hbm_pages) == cudaSuccess &&
              cudaMalloc(&c->kbar, max_pages * g.n_heads * g.head_dim * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&c->prompts, (size_t)g.max_chunks * (g.prompt_dim > 0 ? g.prompt_dim : 1) *
                                          sizeof(float)) == cudaSuccess &&
              cudaEventCreateWithFlags(&c->filled, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&c->drained, cudaEventDisableTiming) == cudaSuccess &&
              cudaStreamCreateWithFlags(&c->copy, cudaStreamNonBlocking) == cudaSuccess &&
              make_events(&c->stage_done, c->n_stage) && make_events(&c->host_ready, g.host_pages);
    if (ok && g.host_pages > 0)
      ok = cudaMalloc(&c->stage_k, c->host_page_bytes * c->n_stage) == cudaSuccess &&
           cudaMalloc(&c->stage_v, c->host_page_bytes * c->n_stage) == cudaSuccess &&
           cudaHostAlloc((void**)&c->host_k, c->host_page_bytes * g.host_pages,
                         cudaHostAllocMapped) == cudaSuccess &&
           cudaHostAlloc((void**)&c->host_v, c->host_page_bytes * g.host_pages,
                         cudaHostAllocMapped) == cudaSuccess &&
           cudaHostGetDevicePointer((void**)&c->host_k_dev, c->host_k, 0) == cudaSuccess &&
           cudaHostGetDevicePointer((void**)&c->host_v_dev, c->host_v, 0) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      release(c);
      return WA_ERR_OOM;
    }
    c->stage_pending.assign(c->n_stage, 0);
    c->host_pending.assign(g.host_pages, 0);
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
  if (!c->cfg.dry_run) {
    cudaDeviceSynchronize();   // no copy may still read or write a slot
    std::fill(c->stage_pending.begin(), c->stage_pending.end(), 0);
    std::fill(c->host_pending.begin(), c->host_pending.end(), 0);
    c->next_stage = 0;
    c->copies_issued = false;
  }
  c->table.clear();
  std::fill(c->hbm_owner.begin(), c->hbm_owner.end(), -1);
  std::fill(c->host_owner.begin(), c->host_owner.end(), -1);
  c->n_pages = 0;
  c->n_chunks = 0;
  c->clock = 0;
  c->stats = wa_cache_stats{};
  return WA_OK;
}

wa_status wa_cache_wait_copies(wa_cache* c, wa_stream_t stream) {
  if (!c) return WA_ERR_INVALID_ARG;
  if (c->cfg.dry_run || !c->copies_issued) return WA_OK;
  if (cudaEventRecord(c->drained, c->copy) != cudaSuccess) return WA_ERR_CUDA;
  return cuda_status(cudaStreamWaitEvent((cudaStream_t)stream, c->drained, 0));
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
    wa_status rc = hbm_slot(c, &keep, -1, s, &hs);
    if (rc != WA_OK) return rc;
    if (!g.dry_run) {
      for (int t = 0; t < 2; ++t) {
        const char* src = static_cast<const char*>(t ? v : k) + (size_t)j * c->page_bytes;
        if (cudaMemcpyAsync(hbm_ptr(c, hs, t), src, c->page_bytes, cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
          return WA_ERR_CUDA;
      }
    }
    count_bytes(c, cudaMemcpyDeviceToDevice, 2 * c->page_bytes);
    c->hbm_owner[hs] = p;
    c->table[p].hbm = hs;
  }
  c->n_chunks++;
  return WA_OK;
}

// Mark pages as used by one retrieval: LRU update, and pages found only in
// DRAM promoted to HBM from the caller's buffer (dev_k[i], dev_v[i]).
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
    if (e.hbm < 0) {
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
  // The selection kernel writes the indices straight into mapped host memory:
  // a device-to-host copy here would queue behind the offloads on the copy
  // engine, and the host waits for the indices.
  if (c->idx_cap < k_p) {
    if (fault_mode() == WA_FAULT_ALLOC) return WA_ERR_OOM;
    if (c->idx_host) {
      cudaFreeHost(c->idx_host);
      c->idx_host = nullptr;
      c->idx_dev = nullptr;
    }
    if (cudaHostAlloc((void**)&c->idx_host, k_p * sizeof(int32_t), cudaHostAllocMapped) !=
            cudaSuccess ||
        cudaHostGetDevicePointer((void**)&c->idx_dev, c->idx_host, 0) != cudaSuccess) {
      cudaGetLastError();
      if (c->idx_host) cudaFreeHost(c->idx_host);
      c->idx_host = nullptr;
      c->idx_dev = nullptr;
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
  if (cudaStreamSynchronize(s) != cudaSuccess) return WA_ERR_CUDA;
  memcpy(idx_out, c->idx_host, k_p * sizeof(int32_t));
  std::vector<const char*> dk(k_p), dv(k_p);
  const size_t rows = (size_t)g.page_tokens * g.n_heads;
  for (int i = 0; i < k_p; ++i)
    if (idx_out[i] < 0 || idx_out[i] >= c->n_pages) return WA_ERR_INDEX;
  // compressed DRAM pages: every copy first (the copy engine streams them back
  // to back), then the decodes from HBM
  if (compressed(c)) {
    int n_f = 0;
    for (int i = 0; i < k_p; ++i)
      if (c->table[idx_out[i]].hbm < 0) ++n_f;
    if (n_f > 0 && (rc = ensure_fetch(c, (size_t)2 * n_f * c->host_page_bytes)) != WA_OK) return rc;
  }
  int f = 0;
  std::vector<int> fslot(k_p, -1);
  for (int i = 0; i < k_p; ++i) {
    if (!compressed(c) || c->table[idx_out[i]].hbm >= 0) continue;
    fslot[i] = f;
    if ((rc = fetch_slot(c, idx_out[i], false, f, s)) != WA_OK ||
        (rc = fetch_slot(c, idx_out[i], true, f + 1, s)) != WA_OK)
      return rc;
    f += 2;
  }
  for (int i = 0; i < k_p; ++i) {
    const int p = idx_out[i];
    char* dst_k = static_cast<char*>(k_buf) + (size_t)i * c->page_bytes;
    char* dst_v = static_cast<char*>(v_buf) + (size_t)i * c->page_bytes;
    if (fslot[i] >= 0) {
      rc = decode_fetched(c, fslot[i], 0, rows, dst_k, s);
      if (rc == WA_OK) rc = decode_fetched(c, fslot[i] + 1, 0, rows, dst_v, s);
    } else {
      rc = read_page(c, p, false, 0, rows, dst_k, s);
      if (rc == WA_OK) rc = read_page(c, p, true, 0, rows, dst_v, s);
    }
    if (rc != WA_OK) return rc;
    dk[i] = dst_k;
    dv[i] = dst_v;
  }
  return use_pages(c, idx_out, k_p, dk.data(), dv.data(), s);
}

wa_status wa_cache_window(wa_cache* c, int n_tokens, void* k_out, void* v_out, wa_stream_t stream) {
  if (!c || !k_out || !v_out || n_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (c->cfg.dry_run) return WA_ERR_INVALID_ARG;
  const wa_cache_config& g = c->cfg;
  const long long total = (long long)c->n_pages * g.page_tokens;
  if (n_tokens > total) return WA_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t row_bytes = (size_t)g.n_heads * g.head_dim * dt_size(g.dtype);   // one token
  const long long first = total - n_tokens;            // first token of the window
  size_t out_off = 0;
  for (int p = (int)(first / g.page_tokens); p < c->n_pages; ++p) {
    const long long t0 = std::max(first, (long long)p * g.page_tokens) - (long long)p * g.page_tokens;
    const size_t toks = (size_t)(g.page_tokens - t0);
    for (int t = 0; t < 2; ++t) {
      wa_status rc = read_page(c, p, t, (size_t)t0 * g.n_heads, toks * g.n_heads,
                               static_cast<char*>(t ? v_out : k_out) + out_off, s);
      if (rc != WA_OK) return rc;
    }
    out_off += toks * row_bytes;
  }
  return WA_OK;
}

wa_status wa_cache_page_location(const wa_cache* c, int page, int* tier, int* slot) {
  if (!c || !tier || !slot) return WA_ERR_INVALID_ARG;
  if (page < 0 || page >= c->n_pages) return WA_ERR_INDEX;
  const wa_cache::Entry& e = c->table[page];
  *tier = e.hbm >= 0 ? 0 : 1;
  *slot = e.hbm >= 0 ? e.hbm : e.host;
  return WA_OK;
}

wa_status wa_cache_page_slots(const wa_cache* c, int page, int* hbm_slot, int* host_slot) {
  if (!c || !hbm_slot || !host_slot) return WA_ERR_INVALID_ARG;
  if (page < 0 || page >= c->n_pages) return WA_ERR_INDEX;
  *hbm_slot = c->table[page].hbm;
  *host_slot = c->table[page].host;
  return WA_OK;
}

wa_status wa_cache_get_stats(const wa_cache* c, wa_cache_stats* out) {
  if (!c || !out) return WA_ERR_INVALID_ARG;
  *out = c->stats;
  out->n_pages = c->n_pages;
  out->n_chunks = c->n_chunks;
  out->in_hbm = 0;
  out->in_host = 0;
  for (int p = 0; p < c->n_pages; ++p) {
    out->in_hbm += c->table[p].hbm >= 0;
    out->in_host += c->table[p].host >= 0;
  }
  return WA_OK;
}

}  // extern "C"
