// Gather of the retrieved pages into one contiguous KV buffer.
//
// WorldAttention (review page), Fig. 1 custom-kernels prong: retrieved pages
// are reorganised into a contiguous buffer so that attention reads dense
// memory; the page's Tab. 9 breakdown puts "KV reconstruction + contiguous
// copy" at 31% of HSA time.  Inferix (summary page), KV Cache Manager:
// index-based selective fetch of cached blocks.
//
// A page is one contiguous slab, so the gather is 2*k_p slab copies whose
// source addresses come from device memory (the indices never visit the
// host).  Each CTA moves one 64 KiB span of one slab with 16-byte loads,
// all loads of a thread issued before its stores.
#include "wa_internal.cuh"

namespace wa {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;                                    // 16 B vectors per thread per span
constexpr size_t kSpan = (size_t)kThreads * kUnroll * 16;     // 32 KiB per CTA iteration

__global__ void __launch_bounds__(kThreads)
k_gather_pages(const uint4* __restrict__ k_pages, const uint4* __restrict__ v_pages,
               size_t page_vecs, int n_pages, const int32_t* __restrict__ idx, int k_p,
               uint4* __restrict__ k_buf, uint4* __restrict__ v_buf, size_t spans_per_slab,
               Ctrl* ctrl) {
  pdl_wait();
  const int n_tensors = v_pages ? 2 : 1;
  const size_t total = spans_per_slab * (size_t)k_p * n_tensors;
  for (size_t w = blockIdx.x; w < total; w += gridDim.x) {
    const size_t span = w % spans_per_slab;
    const size_t rest = w / spans_per_slab;
    const int slot = (int)(rest % k_p);
    const int tensor = (int)(rest / k_p);
    const int page = __ldg(idx + slot);
    const uint4* src = tensor ? v_pages : k_pages;
    uint4* dst = (tensor ? v_buf : k_buf) + (size_t)slot * page_vecs;
    const size_t v0 = span * (kSpan / 16);
    if (page < 0 || page >= n_pages) {
      // bad index: zero this slot and record it (no trap)
      for (int u = 0; u < kUnroll; ++u) {
        const size_t v = v0 + (size_t)u * kThreads + threadIdx.x;
        if (v < page_vecs) dst[v] = make_uint4(0, 0, 0, 0);
      }
      if (threadIdx.x == 0 && span == 0) atomicOr(&ctrl->status, kStatusIndex);
      continue;
    }
    src += (size_t)page * page_vecs;
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t v = v0 + (size_t)u * kThreads + threadIdx.x;
      if (v < page_vecs) r[u] = __ldcs(src + v);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t v = v0 + (size_t)u * kThreads + threadIdx.x;
      if (v < page_vecs) dst[v] = r[u];
    }
  }
}

// Per-head page sets: head h's slice of buffer token s*P + t comes from page
// idx[h*k_p + s].  One CTA copies kPhRows token rows of one (tensor, slot);
// the slot's page for every head is read once into shared memory, and each
// thread walks its (row, vector) position by fixed increments, so the only
// arithmetic per 16-byte vector is an address.  A head row (d elements) is hv
// vectors of one page.
constexpr int kPhRows = 32;
constexpr int kMaxHeads = 1024;

__global__ void __launch_bounds__(kThreads)
k_gather_per_head(const uint4* __restrict__ k_pages, const uint4* __restrict__ v_pages,
                  int n_pages, int page_tokens, int n_heads, int hv, int hv_shift,
                  const int32_t* __restrict__ idx, int k_p, uint4* __restrict__ k_buf,
                  uint4* __restrict__ v_buf, Ctrl* ctrl) {
  __shared__ int pg[kMaxHeads];
  const int slot = blockIdx.y % k_p, tensor = blockIdx.y / k_p;
  for (int h = threadIdx.x; h < n_heads; h += kThreads) {
    const int p = __ldg(idx + h * k_p + slot);
    const bool bad = p < 0 || p >= n_pages;
    pg[h] = bad ? -1 : p;
    if (bad && blockIdx.x == 0) atomicOr(&ctrl->status, kStatusIndex);   // slot zeroed, recorded
  }
  __syncthreads();
  const uint4* src = tensor ? v_pages : k_pages;
  uint4* dst = tensor ? v_buf : k_buf;
  const int row_vecs = n_heads * hv;
  const size_t slab_vecs = (size_t)row_vecs * page_tokens;
  const int r0 = blockIdx.x * kPhRows;
  const int n = (min(page_tokens, r0 + kPhRows) - r0) * row_vecs;   // vectors of this chunk
  const int drow = kThreads / row_vecs, dvec = kThreads - drow * row_vecs;   // dvec < row_vecs
  int row = threadIdx.x / row_vecs, vec = threadIdx.x - row * row_vecs;
  for (int w = threadIdx.x; w < n; w += kThreads * kUnroll) {
    uint4 r[kUnroll];
    size_t at[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (w + u * kThreads < n) {
        const int h = hv_shift >= 0 ? (vec >> hv_shift) : vec / hv;
        const int p = pg[h];
        const size_t off = (size_t)(r0 + row) * row_vecs + vec;
        at[u] = (size_t)slot * slab_vecs + off;
        r[u] = p < 0 ? make_uint4(0, 0, 0, 0) : __ldcs(src + (size_t)p * slab_vecs + off);
      }
      row += drow;
      vec += dvec;
      if (vec >= row_vecs) {
        vec -= row_vecs;
        ++row;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (w + u * kThreads < n) dst[at[u]] = r[u];
  }
}

}  // namespace

wa_status launch_gather_device(const void* k_pages, const void* v_pages, size_t page_bytes,
                               int n_pages, const int32_t* idx_dev, int k_p, void* k_buf,
                               void* v_buf, cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const size_t page_vecs = page_bytes / 16;
  const size_t spans = (page_bytes + kSpan - 1) / kSpan;
  const size_t total = spans * (size_t)k_p * (v_pages ? 2 : 1);
  // 8 CTAs per SM, more than fit at once (late starters fill the SMs that
  // finish early: measured faster than the resident count), grid-stride over spans
  size_t grid = (size_t)sm_count() * 8;
  if (grid > total) grid = total;
  if (grid == 0) return WA_OK;
  return cuda_status(launch_pdl(k_gather_pages, dim3((unsigned)grid), dim3(kThreads), 0, s,
                                (const uint4*)k_pages, (const uint4*)v_pages, page_vecs, n_pages,
                                idx_dev, k_p, (uint4*)k_buf, (uint4*)v_buf, (size_t)spans, ctrl));
}

}  // namespace wa

namespace wa {

wa_status launch_gather_per_head(const void* k_pages, const void* v_pages, int n_pages,
                                 int page_tokens, int n_heads, size_t head_row_bytes,
                                 const int32_t* idx_dev, int k_p, void* k_buf, void* v_buf,
                                 cudaStream_t s) {
  const int hv = (int)(head_row_bytes / 16);
  if (n_heads > kMaxHeads || (long long)n_heads * hv > (1 << 20) || k_p > 32767) return WA_ERR_SHAPE;
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  int hv_shift = -1;
  if ((hv & (hv - 1)) == 0) {
    hv_shift = 0;
    while ((1 << hv_shift) < hv) ++hv_shift;
  }
  dim3 grid((unsigned)((page_tokens + kPhRows - 1) / kPhRows), (unsigned)(k_p * (v_pages ? 2 : 1)));
  k_gather_per_head<<<grid, kThreads, 0, s>>>((const uint4*)k_pages, (const uint4*)v_pages, n_pages,
                                              page_tokens, n_heads, hv, hv_shift, idx_dev, k_p,
                                              (uint4*)k_buf, (uint4*)v_buf, ctrl);
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa
