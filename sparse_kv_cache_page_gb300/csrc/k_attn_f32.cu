// fp32 block attention on the CUDA cores (fp32 inputs, fp32 FMA, accurate
// expf/logf), the path for fp32 workloads that must agree with fp64 to 1e-5.
//
// Inferix (summary page), §3 Technical Approach, Step 3: the chunk's queries
// attend, with no mask, to [cached KV (+) the block's own KV].
//
// One warp per query row: lanes score 32 keys at a time (each lane one full
// dot product against the query row staged in shared memory), the warp keeps
// an online max / sum, and each lane accumulates its own output columns.
//
// Paged form (the gather in the same launch): buffer row r of head h is row
// r % P of page idx[idx_stride * h + r / P] of the page bank; a bad index
// reads as a row of zeros and is recorded, as the gather does.  The first
// warp of each head's first CTA reads every key and value row of its head,
// so it also writes them to the buffer (when one is given).
#include <math.h>

#include "wa_internal.cuh"

namespace wa {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct PagedF32 {
  const float* k_pages;
  const float* v_pages;
  int n_pages, page_tokens, idx_stride;
  const int32_t* idx;
  float* k_buf;      // NULL: no buffer written
  float* v_buf;
  int* status;
};

// Row of buffer position r (< n_main) of head h in the page bank, or NULL for
// a bad page index.
__device__ __forceinline__ size_t paged_row(const PagedF32& pg, int h, int r, size_t row, int d,
                                            bool& bad) {
  const int slot = r / pg.page_tokens;
  const int page = __ldg(pg.idx + (size_t)pg.idx_stride * h + slot);
  bad = page < 0 || page >= pg.n_pages;
  return bad ? 0 : ((size_t)page * pg.page_tokens + (r - slot * pg.page_tokens)) * row + (size_t)h * d;
}

template <bool kPaged>
__global__ void __launch_bounds__(kWarps * 32)
k_block_attn_f32(const float* __restrict__ q, int n_q, const float* __restrict__ k_main,
                 const float* __restrict__ v_main, int n_main, const float* __restrict__ k_loc,
                 const float* __restrict__ v_loc, int n_loc, int n_heads, int d, float scale,
                 float* __restrict__ o, float* __restrict__ lse, const PagedF32 pg) {
  __shared__ __align__(16) float qs[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int i = blockIdx.x * kWarps + warp;
  if (i >= n_q) return;
  const size_t row = (size_t)n_heads * d;
  for (int e = lane; e < d; e += 32) qs[warp][e] = q[(size_t)i * row + (size_t)h * d + e];
  __syncwarp();
  const int n = n_main + n_loc;
  // paged form: this warp also writes its head's buffer rows
  const bool writer = kPaged && pg.k_buf != nullptr && blockIdx.x == 0 && warp == 0;
  float m = -INFINITY, l = 0.f;
  float acc[kMaxD / 32];
#pragma unroll
  for (int c = 0; c < kMaxD / 32; ++c) acc[c] = 0.f;
  for (int k0 = 0; k0 < n; k0 += 32) {
    const int kk = k0 + lane;
    float s = -INFINITY;
    if (kk < n) {
      const float* kr;
      bool bad = false;
      if (kk >= n_main) {
        kr = k_loc + (size_t)(kk - n_main) * row + (size_t)h * d;
      } else if (kPaged) {
        kr = pg.k_pages + paged_row(pg, h, kk, row, d, bad);
        if (bad && writer) atomicOr(pg.status, kStatusIndex);
      } else {
        kr = k_main + (size_t)kk * row + (size_t)h * d;
      }
      float dot = 0.f;
      if (!bad) {
        for (int e = 0; e < d; e += 4) {
          const float4 kv = *reinterpret_cast<const float4*>(kr + e);
          dot = fmaf(qs[warp][e], kv.x, dot);
          dot = fmaf(qs[warp][e + 1], kv.y, dot);
          dot = fmaf(qs[warp][e + 2], kv.z, dot);
          dot = fmaf(qs[warp][e + 3], kv.w, dot);
        }
      }
      if (writer && kk < n_main) {
        float4* dst = reinterpret_cast<float4*>(pg.k_buf + (size_t)kk * row + (size_t)h * d);
        for (int e = 0; e < d; e += 4)
          dst[e / 4] = bad ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(kr + e);
      }
      s = dot * scale;
    }
    const float m_new = fmaxf(m, warp_max(s));
    const float corr = expf(m - m_new);   // 0 on the first batch (m = -inf)
    const float p = kk < n ? expf(s - m_new) : 0.f;
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c) acc[c] *= corr;
    const int nb = min(32, n - k0);
    for (int t = 0; t < nb; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
      const int kt = k0 + t;
      const float* vr;
      bool bad = false;
      if (kt >= n_main) {
        vr = v_loc + (size_t)(kt - n_main) * row + (size_t)h * d;
      } else if (kPaged) {
        vr = pg.v_pages + paged_row(pg, h, kt, row, d, bad);
      } else {
        vr = v_main + (size_t)kt * row + (size_t)h * d;
      }
#pragma unroll
      for (int c = 0; c < kMaxD / 32; ++c) {
        const int e = lane + 32 * c;
        if (e < d) {
          const float v = bad ? 0.f : vr[e];
          acc[c] = fmaf(pt, v, acc[c]);
          if (writer && kt < n_main) pg.v_buf[(size_t)kt * row + (size_t)h * d + e] = v;
        }
      }
    }
    m = m_new;
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int c = 0; c < kMaxD / 32; ++c) {
    const int e = lane + 32 * c;
    if (e < d) o[(size_t)i * row + (size_t)h * d + e] = acc[c] * inv;
  }
  if (lse && lane == 0) lse[(size_t)h * n_q + i] = m + logf(l);
}

}  // namespace

wa_status launch_attn_f32(const float* q, int n_q, const float* k_main, const float* v_main,
                          int n_main, const float* k_loc, const float* v_loc, int n_loc,
                          int n_heads, int head_dim, float scale, float* o, float* lse,
                          cudaStream_t s, const PagedKV* paged) {
  dim3 grid((n_q + kWarps - 1) / kWarps, n_heads);
  PagedF32 pg{};
  if (paged) {
    Ctrl* ctrl = nullptr;
    wa_status rc = get_ctrl(&ctrl);
    if (rc != WA_OK) return rc;
    pg.k_pages = static_cast<const float*>(paged->k_pages);
    pg.v_pages = static_cast<const float*>(paged->v_pages);
    pg.n_pages = paged->n_pages;
    pg.page_tokens = paged->page_tokens;
    pg.idx_stride = paged->idx_stride;
    pg.idx = paged->idx;
    pg.k_buf = const_cast<float*>(k_main);   // the buffer to write, or NULL
    pg.v_buf = const_cast<float*>(v_main);
    pg.status = &ctrl->status;
    k_block_attn_f32<true><<<grid, kWarps * 32, 0, s>>>(q, n_q, nullptr, nullptr, n_main, k_loc,
                                                        v_loc, n_loc, n_heads, head_dim, scale, o,
                                                        lse, pg);
  } else {
    k_block_attn_f32<false><<<grid, kWarps * 32, 0, s>>>(q, n_q, k_main, v_main, n_main, k_loc,
                                                         v_loc, n_loc, n_heads, head_dim, scale, o,
                                                         lse, pg);
  }
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa
