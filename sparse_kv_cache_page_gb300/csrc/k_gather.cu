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
// idx[h*k_p + s].  Each unit is one 16-byte vector of the destination, so
// stores stay contiguous; a head row (d elements) is hv vectors of one page.
__global__ void __launch_bounds__(kThreads)
k_gather_per_head(const uint4* __restrict__ k_pages, const uint4* __restrict__ v_pages,
                  int n_pages, int page_tokens, int n_heads, int hv,
                  const int32_t* __restrict__ idx, int k_p, uint4* __restrict__ k_buf,
                  uint4* __restrict__ v_buf, size_t vecs_per_tensor, Ctrl* ctrl) {
  const int n_tensors = v_pages ? 2 : 1;
  const size_t row_vecs = (size_t)n_heads * hv;            // one token row
  const size_t slab_vecs = row_vecs * page_tokens;         // one page
  const size_t total = vecs_per_tensor * n_tensors;
  const size_t step = (size_t)gridDim.x * kThreads * kUnroll;
  for (size_t base = (size_t)blockIdx.x * kThreads * kUnroll; base < total; base += step) {
    uint4 r[kUnroll];
    size_t dv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t w = base + (size_t)u * kThreads + threadIdx.x;
      dv[u] = w;
      if (w >= total) continue;
      const int tensor = w >= vecs_per_tensor;
      const size_t v = w - (tensor ? vecs_per_tensor : 0);
      const int slot = (int)(v / slab_vecs);
      const size_t in_slab = v % slab_vecs;
      const int h = (int)((in_slab % row_vecs) / hv);
      const int page = __ldg(idx + h * k_p + slot);
      if (page < 0 || page >= n_pages) {
        r[u] = make_uint4(0, 0, 0, 0);
        atomicOr(&ctrl->status, kStatusIndex);
      } else {
        r[u] = __ldcs((tensor ? v_pages : k_pages) + (size_t)page * slab_vecs + in_slab);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t w = dv[u];
      if (w >= total) continue;
      if (w >= vecs_per_tensor) v_buf[w - vecs_per_tensor] = r[u];
      else k_buf[w] = r[u];
    }
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
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t grid = (size_t)sms * 8;   // 8 resident CTAs per SM, grid-stride over spans
  if (grid > total) grid = total;
  k_gather_pages<<<(unsigned)grid, kThreads, 0, s>>>(
      (const uint4*)k_pages, (const uint4*)v_pages, page_vecs, n_pages, idx_dev, k_p,
      (uint4*)k_buf, (uint4*)v_buf, spans, ctrl);
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa

namespace wa {

wa_status launch_gather_per_head(const void* k_pages, const void* v_pages, int n_pages,
                                 int page_tokens, int n_heads, size_t head_row_bytes,
                                 const int32_t* idx_dev, int k_p, void* k_buf, void* v_buf,
                                 cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const int hv = (int)(head_row_bytes / 16);
  const size_t vecs = (size_t)k_p * page_tokens * n_heads * hv;
  const size_t total = vecs * (v_pages ? 2 : 1);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t grid = (size_t)sms * 8;
  const size_t need = (total + (size_t)kThreads * kUnroll - 1) / ((size_t)kThreads * kUnroll);
  if (grid > need) grid = need;
  k_gather_per_head<<<(unsigned)grid, kThreads, 0, s>>>(
      (const uint4*)k_pages, (const uint4*)v_pages, n_pages, page_tokens, n_heads, hv, idx_dev,
      k_p, (uint4*)k_buf, (uint4*)v_buf, vecs, ctrl);
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa
