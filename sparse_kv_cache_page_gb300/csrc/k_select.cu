// Page summaries and two-stage page retrieval.
//
// WorldAttention (review page), HKV section (paper §3.1 HKV): every cached
// 8-frame page is summarised by its mean key; a chunk is scored through its
// mean query, alpha_{m,j} = Qbar^T Kbar_{m,j} / sqrt(d_k), after a prompt-
// stage top-1 chunk pick by cosine similarity; the top-K_p pages are kept.
//
// Both kernels are HBM-bound column sums over token rows: each thread owns
// one or more 16-byte column vectors of a token row and walks rows with
// several independent loads in flight; CTAs of one reduction meet through a
// "last CTA finishes" ticket (no spin-wait): every CTA stores its partial
// sums, fences, and takes a ticket; the CTA holding the last ticket adds the
// partials in a fixed order (deterministic) and runs the tail work.
#include <math.h>
#include <mutex>

#include "wa_internal.cuh"

namespace wa {
namespace {

constexpr int kThreads = 384;           // 2 x 192 16-byte vectors of a 1,536-element bf16 row
constexpr int kTargetCtas = 152 * 4;     // resident summarize CTAs: 152 SMs x 4
constexpr unsigned kSelectCounter = 4095;

template <typename T> struct VecOf;
template <> struct VecOf<__nv_bfloat16> { static constexpr int E = 8; };
template <> struct VecOf<float> { static constexpr int E = 4; };

__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&f)[8]) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load_vec(const float* p, float (&f)[4]) {
  float4 v = __ldg(reinterpret_cast<const float4*>(p));
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}

// Column sums of rows [r0, r1) of a matrix with rows `stride` elements apart,
// over the first row_elems columns, into red[0..row_elems).
// Thread layout: the first nvec*R threads; vec = tid % nvec, row phase = tid / nvec.
// VPT > 1 only when R == 1 (nvec > blockDim): thread handles vec, vec+256, ...
// kBatchTail: the rows left after the whole batches go as one more batch with
// every load in flight (rows past r1 skipped), else one row at a time (fewer
// registers: the page summaries, whose ranges are long, keep four CTAs per SM).
template <typename T, int VPT, bool kBatchTail = false>
__device__ void colsum_rows(const T* __restrict__ base, size_t stride, int row_elems, int nvec,
                            int R, int r0, int r1, float* red /* smem, R*row_elems floats */) {
  constexpr int E = VecOf<T>::E;
  constexpr int U = VPT == 1 ? 8 : (VPT == 2 ? 4 : 2);   // rows in flight
  const int tid = threadIdx.x;
  const bool active = tid < nvec * R || VPT > 1;
  const int vec = VPT > 1 ? tid : tid % nvec;
  const int rp = VPT > 1 ? 0 : tid / nvec;
  float acc[VPT][E];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[v][e] = 0.f;
  if (active) {
    int r = r0 + rp;
    for (; r + (U - 1) * R < r1; r += U * R) {
      float f[U][VPT][E];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int cv = vec + v * kThreads;
          if (VPT == 1 || cv < nvec)
            load_vec(base + (size_t)(r + u * R) * stride + (size_t)cv * E, f[u][v]);
          else
#pragma unroll
            for (int e = 0; e < E; ++e) f[u][v][e] = 0.f;
        }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < VPT; ++v)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[v][e] += f[u][v][e];
    }
    // the last (partial) batch: its loads all in flight, rows past r1 skipped
    if (kBatchTail && r < r1) {
      float f[U][VPT][E];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          const int cv = vec + v * kThreads;
          if (r + u * R < r1 && (VPT == 1 || cv < nvec))
            load_vec(base + (size_t)(r + u * R) * stride + (size_t)cv * E, f[u][v]);
        }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < VPT; ++v)
          if (r + u * R < r1 && (VPT == 1 || vec + v * kThreads < nvec))
#pragma unroll
            for (int e = 0; e < E; ++e) acc[v][e] += f[u][v][e];
    }
    for (; !kBatchTail && r < r1; r += R) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int cv = vec + v * kThreads;
        if (VPT == 1 || cv < nvec) {
          float f[E];
          load_vec(base + (size_t)r * stride + (size_t)cv * E, f);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[v][e] += f[e];
        }
      }
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int cv = vec + v * kThreads;
      if (VPT == 1 || cv < nvec)
#pragma unroll
        for (int e = 0; e < E; ++e) red[rp * row_elems + cv * E + e] = acc[v][e];
    }
  }
  __syncthreads();
  // fold the R row phases (fixed order)
  if (R > 1) {
    for (int c = tid; c < row_elems; c += blockDim.x) {
      float s = red[c];
      for (int p = 1; p < R; ++p) s += red[p * row_elems + c];
      red[c] = s;
    }
    __syncthreads();
  }
}

// Returns true in every thread of the CTA that took the last ticket.
__device__ bool last_ticket(unsigned* counter, unsigned n) {
  __shared__ unsigned s_ticket;
  // the CTA's writes are ordered before thread 0's fence by the barrier (a
  // fence is cumulative over what happens before it), so one fence suffices
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_ticket = atomicAdd(counter, 1u);
    if (s_ticket == n - 1) __threadfence();
  }
  __syncthreads();
  return s_ticket == n - 1;
}

// out[c] = scale * sum_{p < n} rows[p][c] for c < row_elems (row_elems % 4 == 0),
// p in increasing order; loads of 8 rows in flight per thread.
__device__ void sum_rows4(const float* rows, int n, int row_elems, float* out, float scale) {
  const int n4 = row_elems / 4;
  for (int c = threadIdx.x; c < n4; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int p = 0;
    for (; p + 8 <= n; p += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = __ldcg(reinterpret_cast<const float4*>(rows + (size_t)(p + u) * row_elems) + c);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
    for (; p < n; ++p) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(rows + (size_t)p * row_elems) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    reinterpret_cast<float4*>(out)[c] =
        make_float4(acc.x * scale, acc.y * scale, acc.z * scale, acc.w * scale);
  }
}

// out[c] = scale * sum_{p < n} rows[p * stride + c] for c < width (width and
// stride multiples of 4), p in increasing order; loads of 8 rows in flight.
__device__ void sum_rows4_strided(const float* rows, int n, int width, size_t stride, float* out,
                                  float scale) {
  const int n4 = width / 4;
  for (int c = threadIdx.x; c < n4; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int p = 0;
    for (; p + 8 <= n; p += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = __ldcg(reinterpret_cast<const float4*>(rows + (size_t)(p + u) * stride) + c);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
    for (; p < n; ++p) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(rows + (size_t)p * stride) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    reinterpret_cast<float4*>(out)[c] =
        make_float4(acc.x * scale, acc.y * scale, acc.z * scale, acc.w * scale);
  }
}

// ---------------------------------------------------------------------------
// page summaries
// ---------------------------------------------------------------------------
// One launch sums up to kMaxSegs independent row sets ("segments"), each cut
// into pages of page_tokens rows and each page into `splits` row ranges; CTAs
// [cta0, cta0 + n_pages * splits) belong to a segment.  A segment's arithmetic
// (its ranges and the fixed-order reduction of their partials) does not depend
// on the other segments in the launch.
constexpr int kMaxSegs = 3;
template <typename T>
struct SumSeg {
  const T* pages;
  float* kbar;         // [n_pages][row_elems] means
  float* partial;      // [n_pages][splits][row_elems] scratch (splits > 1)
  int page_tokens, n_rows, splits, rows_per_split, cta0, counter0;
};
template <typename T>
struct SumSegs {
  SumSeg<T> s[kMaxSegs];
  int n;
};

// Four resident CTAs per SM (at most 40 registers): five, which the compiler picks
// otherwise, stream about 8% slower.
template <typename T, int VPT>
__global__ void __launch_bounds__(kThreads, 4)
k_page_summarize(const SumSegs<T> segs, int row_elems, int cw, int n_cb, int nvec, int R,
                 Ctrl* ctrl) {
  extern __shared__ float red[];
  pdl_wait();
  // this CTA's segment (static indices: the table stays in parameter space)
  SumSeg<T> g = segs.s[0];
  if (segs.n > 1 && (int)blockIdx.x >= segs.s[1].cta0) g = segs.s[1];
  if (segs.n > 2 && (int)blockIdx.x >= segs.s[2].cta0) g = segs.s[2];
  // CTA order: column block fastest, so the CTAs reading one row range start together
  const int local = (int)blockIdx.x - g.cta0;
  const int cb = local % n_cb;
  const int js = local / n_cb;
  const int j = js / g.splits, s = js % g.splits;
  // page j holds rows [j P, j P + rows_j) of the n_rows; only the last may be short
  const int rows_j = min(g.page_tokens, g.n_rows - j * g.page_tokens);
  const int r0 = s * g.rows_per_split;
  const int r1 = min(rows_j, r0 + g.rows_per_split);
  const T* base = g.pages + (size_t)j * g.page_tokens * row_elems + (size_t)cb * cw;
  colsum_rows<T, VPT>(base, (size_t)row_elems, cw, nvec, R, r0, r1, red);
  const float inv = 1.0f / (float)rows_j;
  float* out = g.kbar + (size_t)j * row_elems + (size_t)cb * cw;
  if (g.splits == 1) {
    for (int c = threadIdx.x; c < cw; c += blockDim.x) out[c] = red[c] * inv;
    return;
  }
  float* mine = g.partial + ((size_t)j * g.splits + s) * row_elems + (size_t)cb * cw;
  for (int c = threadIdx.x; c < cw; c += blockDim.x) mine[c] = red[c];
  unsigned* counter = &ctrl->counters[g.counter0 + j * n_cb + cb];
  if (!last_ticket(counter, (unsigned)g.splits)) return;
  // the column block's partial sums in split order, then the mean
  sum_rows4_strided(g.partial + (size_t)j * g.splits * row_elems + (size_t)cb * cw, g.splits, cw,
                    (size_t)row_elems, out, inv);
  if (threadIdx.x == 0) *counter = 0u;
}

// ---------------------------------------------------------------------------
// select: mean query -> prompt top-1 -> page scores -> top-K_p
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Orderable key: ascending key = descending score, then ascending candidate.
__device__ __forceinline__ unsigned long long score_key(float a, unsigned c) {
  if (a == 0.f) a = 0.f;   // -0 ties +0
  unsigned u = __float_as_uint(a);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)(~u) << 32) | c;
}

// Ascending bitonic sort of 32 keys, one per lane, by shuffles.
__device__ __forceinline__ unsigned long long warp_sort32(unsigned long long key) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, j);
      const bool keep_min = ((lane & j) == 0) == ((lane & k) == 0);
      key = keep_min ? (other < key ? other : key) : (other > key ? other : key);
    }
  return key;
}

__device__ void bitonic_sort(unsigned long long* keys, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const unsigned long long a = keys[i], b = keys[ixj];
          if ((a > b) == up) { keys[i] = b; keys[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

// The selection kernel runs three kinds of CTAs at once:
//   * query tiles: CTA (column block cb, row block rb) sums query rows
//     [rb*rps, ...) over the columns of heads [cb*hpb, ...) (one head per block
//     when a head row is whole 16-byte vectors of at least 32 values, else all
//     heads in one block) and stores the partial sums; the last CTA of a column
//     block adds its n_rb partials in row-block order into the block's mean
//     query, then scores every page that can be a candidate on each of its heads,
//     alpha_part[h][j] = Qbar_h . Kbar[j][h];
//   * prompt CTAs: CTA m computes cos(prompt_cur, prompt_chunks[m]);
//   * the CTA that finishes last picks the chunk (largest cosine, lowest index on
//     ties), forms alpha_j = sum_h alpha_part[h][j] / sqrt(d) in head order (or
//     keeps alpha_part per head for a page set per head) and keeps the top k_p.
// Every sum runs in a fixed order, so the result does not depend on timing.
struct SelectArgs {
  int n_q, row_elems, head_dim, n_heads;
  int nvec, R;                 // phase-A thread layout over one column block
  int hpb, cw, n_cb;           // heads per column block, its width, column blocks
  int n_rb, rows_per_block;    // row blocks of the queries
  int n_alpha;                 // pages that can be candidates (scored per head)
  float* partial;              // [n_cb][n_rb][cw]
  float* alpha_part;           // [n_heads][n_alpha]
  float* cosv;                 // [n_chunks]
  const float* kbar;
  int n_pages;
  const float* prompt_cur;
  const float* prompt_chunks;
  int n_chunks, prompt_dim, ppc, k_p;
  int32_t* idx_out;
  float* scores_out;
  int32_t* chunk_out;
  Ctrl* ctrl;
  int n_cand_max2;   // power of two >= candidate count
  int per_head;      // 0: one page set scored over all heads; 1: a page set per head
  int stage_floats;  // shared memory past alpha and keys for staging partial scores
};

// Sum of a block-wide value over the CTA's warps in warp order (every thread
// gets the total); `scratch` holds 33 floats.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < nw ? scratch[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) scratch[32] = t;
  }
  __syncthreads();
  return scratch[32];
}

// Top k_p of n candidates (scores in alpha[0..n)) into out_idx / out_sc,
// ascending by candidate; ties to the lower candidate.  keys: n2 words of smem.
__device__ void select_topk(const float* alpha, int n, int n2, int k_p, int cand0,
                            unsigned long long* keys, int32_t* out_idx, float* out_sc) {
  const int tid = threadIdx.x;
  if (n <= 32) {
    if (tid < 32) {
      unsigned long long key = tid < n ? score_key(alpha[tid], (unsigned)tid) : ~0ull;
      key = warp_sort32(key);
      unsigned long long sel = tid < k_p ? (key & 0xffffffffull) : ~0ull;
      sel = warp_sort32(sel);
      if (tid < k_p) {
        const int c = (int)(sel & 0xffffffffull);
        out_idx[tid] = cand0 + c;
        if (out_sc) out_sc[tid] = alpha[c];
      }
    }
    __syncthreads();
    return;
  }
  for (int i = tid; i < n2; i += blockDim.x)
    keys[i] = i < n ? score_key(alpha[i], (unsigned)i) : ~0ull;
  __syncthreads();
  bitonic_sort(keys, n2);
  // the first k_p keys are the selection; re-sort them by candidate index
  int k2 = 1;
  while (k2 < k_p) k2 <<= 1;
  for (int i = tid; i < k2; i += blockDim.x) keys[i] = i < k_p ? (keys[i] & 0xffffffffull) : ~0ull;
  __syncthreads();
  bitonic_sort(keys, k2);
  for (int i = tid; i < k_p; i += blockDim.x) {
    const int c = (int)(keys[i] & 0xffffffffull);
    out_idx[i] = cand0 + c;
    if (out_sc) out_sc[i] = alpha[c];
  }
  __syncthreads();
}

// Two CTAs per SM (at most 80 registers), so that every query tile of the
// one-layer WorldAttention chunk (12 x 26) and the prompt CTAs run in one wave.
template <typename T, int VPT>
__global__ void __launch_bounds__(kThreads, 2)
k_select_pages(const T* __restrict__ q, SelectArgs a) {
  extern __shared__ float smem[];
  __shared__ float s_red[33];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int n_tiles = a.n_cb * a.n_rb;
  const int b = blockIdx.x;
  if (b < n_tiles) {
    // ---- query tile: partial column sums of one row block over one column block
    const int cb = b / a.n_rb, rb = b % a.n_rb;
    const int r0 = rb * a.rows_per_block;
    const int r1 = min(a.n_q, r0 + a.rows_per_block);
    colsum_rows<T, VPT, true>(q + (size_t)cb * a.cw, (size_t)a.row_elems, a.cw, a.nvec, a.R, r0, r1,
                              smem);
    float* mine = a.partial + ((size_t)cb * a.n_rb + rb) * a.cw;
    for (int c = tid; c < a.cw; c += blockDim.x) mine[c] = smem[c];
    unsigned* counter = &a.ctrl->counters[kSelectCounter - 1 - cb];
    if (!last_ticket(counter, (unsigned)a.n_rb)) return;
    // the column block's mean query: thread group g adds row blocks g, g + G,
    // ... (one load each in flight), then the G group sums are added in order
    float* qbar = smem;
    const float* part = a.partial + (size_t)cb * a.n_rb * a.cw;
    const int n4 = a.cw / 4;
    const int G = n4 <= (int)blockDim.x ? min((int)blockDim.x / n4, a.n_rb) : 1;
    if (G > 1) {
      float4* red4 = reinterpret_cast<float4*>(smem + a.cw);   // [G][n4]
      const int col = tid % n4, grp = tid / n4;
      if (grp < G) {
        // row blocks grp, grp + G, ... in order, eight loads in flight
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r0 = grp; r0 < a.n_rb; r0 += 8 * G) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = r0 + u * G;
            v[u] = r < a.n_rb ? __ldcg(reinterpret_cast<const float4*>(part + (size_t)r * a.cw) + col)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (r0 + u * G < a.n_rb) {
              acc.x += v[u].x;
              acc.y += v[u].y;
              acc.z += v[u].z;
              acc.w += v[u].w;
            }
          }
        }
        red4[grp * n4 + col] = acc;
      }
      __syncthreads();
      const float inv = 1.0f / (float)a.n_q;
      for (int c = tid; c < n4; c += blockDim.x) {
        float4 t = red4[c];
        for (int g = 1; g < G; ++g) {
          const float4 v = red4[g * n4 + c];
          t.x += v.x;
          t.y += v.y;
          t.z += v.z;
          t.w += v.w;
        }
        reinterpret_cast<float4*>(qbar)[c] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
      }
    } else {
      sum_rows4(part, a.n_rb, a.cw, qbar, 1.0f / (float)a.n_q);
    }
    if (tid == 0) *counter = 0u;
    __syncthreads();
    // per-head partial scores of every page that can be a candidate, eight
    // (head, page) items per warp in flight
    const int h0 = cb * a.hpb;
    const int nh = min(a.hpb, a.n_heads - h0);
    const int n_items = nh * a.n_alpha;
    const bool vec = (a.head_dim & 3) == 0;
    for (int w0 = warp * 8; w0 < n_items; w0 += nwarps * 8) {
      float acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = 0.f;
      if (vec) {
        const int d4 = a.head_dim / 4;
        for (int c0 = 0; c0 < d4; c0 += 32) {
          const int c = c0 + lane;
          float4 y[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int w = w0 + u;
            y[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (w < n_items && c < d4) {
              const int hh = w / a.n_alpha, j = w % a.n_alpha;
              y[u] = __ldg(reinterpret_cast<const float4*>(a.kbar + (size_t)j * a.row_elems +
                                                           (size_t)(h0 + hh) * a.head_dim) + c);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int w = w0 + u;
            if (w < n_items && c < d4) {
              const float4 x = reinterpret_cast<const float4*>(qbar + (w / a.n_alpha) * a.head_dim)[c];
              acc[u] += x.x * y[u].x + x.y * y[u].y + x.z * y[u].z + x.w * y[u].w;
            }
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int w = w0 + u;
          if (w < n_items) {
            const int hh = w / a.n_alpha, j = w % a.n_alpha;
            const float* kb = a.kbar + (size_t)j * a.row_elems + (size_t)(h0 + hh) * a.head_dim;
            for (int e = lane; e < a.head_dim; e += 32) acc[u] += qbar[hh * a.head_dim + e] * kb[e];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float dot = warp_sum(acc[u]);
        const int w = w0 + u;
        if (lane == 0 && w < n_items) {
          const int hh = w / a.n_alpha, j = w % a.n_alpha;
          a.alpha_part[(size_t)(h0 + hh) * a.n_alpha + j] = dot;
        }
      }
    }
  } else {
    // ---- prompt CTA: cosine of the current prompt with chunk m's prompt
    const int m = b - n_tiles;
    const float* cm = a.prompt_chunks + (size_t)m * a.prompt_dim;
    float dot = 0.f, np = 0.f, nc = 0.f;
    if ((a.prompt_dim & 3) == 0 &&
        ((reinterpret_cast<uintptr_t>(a.prompt_cur) | reinterpret_cast<uintptr_t>(cm)) & 15) == 0) {
      const float4* x4 = reinterpret_cast<const float4*>(a.prompt_cur);
      const float4* y4 = reinterpret_cast<const float4*>(cm);
      const int n4 = a.prompt_dim / 4;
      for (int i0 = tid; i0 < n4; i0 += 4 * blockDim.x) {
        float4 x[4], y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * blockDim.x;
          x[u] = i < n4 ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          y[u] = i < n4 ? __ldg(y4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          dot += x[u].x * y[u].x + x[u].y * y[u].y + x[u].z * y[u].z + x[u].w * y[u].w;
          np += x[u].x * x[u].x + x[u].y * x[u].y + x[u].z * x[u].z + x[u].w * x[u].w;
          nc += y[u].x * y[u].x + y[u].y * y[u].y + y[u].z * y[u].z + y[u].w * y[u].w;
        }
      }
    } else {
      for (int i = tid; i < a.prompt_dim; i += blockDim.x) {
        const float x = a.prompt_cur[i], y = cm[i];
        dot += x * y;
        np += x * x;
        nc += y * y;
      }
    }
    dot = block_sum(dot, s_red);
    np = block_sum(np, s_red);
    nc = block_sum(nc, s_red);
    if (tid == 0) a.cosv[m] = (np > 0.f && nc > 0.f) ? dot / (sqrtf(np) * sqrtf(nc)) : 0.f;
  }
  if (!last_ticket(&a.ctrl->counters[kSelectCounter], (unsigned)(a.n_cb + a.n_chunks))) return;

  // ---- the last CTA: chunk pick, scores, top-k_p.  smem: alpha[n2] | keys[n2]
  __shared__ int s_chunk;
  float* cos_s = smem;   // [n_chunks], read before alpha reuses the space
  for (int m = tid; m < a.n_chunks; m += blockDim.x) cos_s[m] = __ldcg(a.cosv + m);
  __syncthreads();
  if (tid == 0) {
    int best_m = -1;
    float best = -INFINITY;
    for (int m = 0; m < a.n_chunks; ++m)   // ascending m: the first wins a tie
      if (best_m < 0 || cos_s[m] > best) {
        best = cos_s[m];
        best_m = m;
      }
    s_chunk = best_m;
  }
  __syncthreads();
  const int chunk = a.n_chunks > 0 ? s_chunk : -1;
  const int cand0 = a.n_chunks > 0 ? chunk * a.ppc : 0;
  const int n_cand = a.n_chunks > 0 ? a.ppc : a.n_pages;
  const float inv_sqrt_d = 1.0f / sqrtf((float)a.head_dim);
  float* alpha = smem;
  unsigned long long* keys =
      reinterpret_cast<unsigned long long*>(alpha + ((a.n_cand_max2 + 3) & ~3));
  if (a.per_head && n_cand <= 32 && a.k_p <= n_cand) {
    // a set per head with at most 32 candidates: a warp per head sorts its
    // candidates' keys in registers, then the chosen ones by candidate index
    for (int h = warp; h < a.n_heads; h += nwarps) {
      const float my_alpha =
          lane < n_cand ? __ldcg(a.alpha_part + (size_t)h * a.n_alpha + cand0 + lane) * inv_sqrt_d
                        : 0.f;
      unsigned long long key = lane < n_cand ? score_key(my_alpha, (unsigned)lane) : ~0ull;
      key = warp_sort32(key);
      unsigned long long sel = lane < a.k_p ? (key & 0xffffffffull) : ~0ull;
      sel = warp_sort32(sel);
      const int c = lane < a.k_p ? (int)(sel & 0xffffffffull) : 0;
      const float alpha_c = __shfl_sync(0xffffffffu, my_alpha, c);
      if (lane < a.k_p) {
        a.idx_out[h * a.k_p + lane] = cand0 + c;
        if (a.scores_out) a.scores_out[h * a.k_p + lane] = alpha_c;
      }
    }
  } else if (a.per_head) {
    for (int h = 0; h < a.n_heads; ++h) {
      for (int c = tid; c < n_cand; c += blockDim.x)
        alpha[c] = __ldcg(a.alpha_part + (size_t)h * a.n_alpha + cand0 + c) * inv_sqrt_d;
      __syncthreads();
      select_topk(alpha, n_cand, a.n_cand_max2, a.k_p, cand0, keys, a.idx_out + h * a.k_p,
                  a.scores_out ? a.scores_out + h * a.k_p : nullptr);
    }
  } else {
    // one page set: the heads' partial scores added in head order (staged in
    // shared memory first when they fit, so that all loads are in flight at once)
    float* stage = alpha + ((a.n_cand_max2 + 3) & ~3) + 2 * a.n_cand_max2;   // past the keys
    if ((size_t)n_cand * a.n_heads <= (size_t)a.stage_floats) {
      for (int i = tid; i < n_cand * a.n_heads; i += blockDim.x) {
        const int h = i / n_cand, c = i % n_cand;
        stage[i] = __ldcg(a.alpha_part + (size_t)h * a.n_alpha + cand0 + c);
      }
      __syncthreads();
      for (int c = tid; c < n_cand; c += blockDim.x) {
        float s = 0.f;
        for (int h = 0; h < a.n_heads; ++h) s += stage[h * n_cand + c];
        alpha[c] = s * inv_sqrt_d;
      }
    } else {
      for (int c = tid; c < n_cand; c += blockDim.x) {
        float s = 0.f;
        for (int h = 0; h < a.n_heads; ++h)
          s += __ldcg(a.alpha_part + (size_t)h * a.n_alpha + cand0 + c);
        alpha[c] = s * inv_sqrt_d;
      }
    }
    __syncthreads();
    select_topk(alpha, n_cand, a.n_cand_max2, a.k_p, cand0, keys, a.idx_out, a.scores_out);
  }
  if (tid == 0) {
    if (a.chunk_out) a.chunk_out[0] = chunk;
    a.ctrl->counters[kSelectCounter] = 0u;
  }
}

struct Plan {
  int nvec, R, vpt, threads;
};

template <typename T>
Plan plan_rows(int row_elems) {
  Plan p;
  p.nvec = row_elems / VecOf<T>::E;
  if (p.nvec <= kThreads) {
    p.R = kThreads / p.nvec;
    p.vpt = 1;
  } else {
    p.R = 1;
    p.vpt = (p.nvec + kThreads - 1) / kThreads;
    p.vpt = p.vpt <= 2 ? 2 : (p.vpt <= 4 ? 4 : 8);
  }
  p.threads = kThreads;
  return p;
}

// One segment of a summarize launch: rows x [n_rows][row_elems], means of
// consecutive groups of `block` rows (the last may be short) into out.
struct SegIn {
  const void* x;
  int n_rows, block;
  float* out;
};

template <typename T>
wa_status summarize_t(const SegIn* in, int n_seg, int row_elems, cudaStream_t st) {
  if (n_seg < 1 || n_seg > kMaxSegs) return WA_ERR_INVALID_ARG;
  // column blocks of 32 16-byte vectors (one warp per row) for long pages whose
  // rows divide into them, else whole rows (short blocks, such as the HSA
  // block means, already give one CTA per block without partials; cutting
  // them into column blocks only multiplies small CTAs: 0.046 -> 0.049 ms)
  const int E = VecOf<T>::E;
  int max_block = 0;
  for (int i = 0; i < n_seg; ++i) max_block = in[i].block > max_block ? in[i].block : max_block;
  const int cw = (row_elems / E) % 32 == 0 && max_block >= 1024 ? 32 * E : row_elems;
  const int n_cb = row_elems / cw;
  Plan p = plan_rows<T>(cw);
  SumSegs<T> segs{};
  segs.n = n_seg;
  size_t part_off[kMaxSegs], part_floats = 0;
  int ctas = 0, counters = 0;
  for (int i = 0; i < n_seg; ++i) {
    if (in[i].n_rows <= 0 || in[i].block <= 0) return WA_ERR_INVALID_ARG;
    const int page_tokens = in[i].block;
    const int n_pages = (in[i].n_rows + page_tokens - 1) / page_tokens;
    // About two waves of CTAs per segment: a single wave of long row ranges
    // ends with the slowest range, and more, shorter ranges add partial sums
    // (measured on the one-layer WorldAttention bank with whole-row CTAs:
    // 0.251 ms with one wave of 256-thread CTAs; with 384-thread CTAs, four
    // resident per SM, 0.2247 ms for two whole waves, 0.2278 for two and a
    // half, 0.2280 for three, 0.2315 for four).  Column blocks of one warp's
    // width (512 bytes of a bf16 row) keep the partials per output few: 40
    // pages take 5 row ranges each (0.2234 -> 0.2173 ms against whole rows in
    // 30 ranges), 8 pages 25 (0.0675 -> 0.0555 ms against 151 ranges, whose
    // last CTA added 151 partials one load batch after another).
    int splits = 2 * kTargetCtas / (n_pages * n_cb);
    if (splits < 1) splits = 1;
    // at least 16 rows of a whole row per CTA, 64 of a column block
    const int min_rows = n_cb > 1 ? 64 : 16;
    const int max_splits = (page_tokens + min_rows - 1) / min_rows;
    if (splits > max_splits) splits = max_splits;
    if (splits > 256) splits = 256;
    const int rps = (page_tokens + splits - 1) / splits;
    splits = (page_tokens + rps - 1) / rps;
    SumSeg<T>& g = segs.s[i];
    g.pages = static_cast<const T*>(in[i].x);
    g.kbar = in[i].out;
    g.page_tokens = page_tokens;
    g.n_rows = in[i].n_rows;
    g.splits = splits;
    g.rows_per_split = rps;
    g.cta0 = ctas;
    g.counter0 = counters;
    ctas += splits * n_pages * n_cb;
    if (splits > 1) counters += n_pages * n_cb;
    part_off[i] = part_floats;
    part_floats += (size_t)n_pages * splits * row_elems;
  }
  if (counters > (int)kSelectCounter) return WA_ERR_SHAPE;   // the select kernel's ticket
  Scratch sc;
  wa_status rc = get_scratch(part_floats * sizeof(float), &sc);
  if (rc != WA_OK) return rc;
  for (int i = 0; i < n_seg; ++i) segs.s[i].partial = static_cast<float*>(sc.data) + part_off[i];
  const size_t smem = (size_t)p.R * cw * sizeof(float);
  dim3 grid((unsigned)ctas);
  switch (p.vpt) {
#define WA_CASE(V)                                                                          \
  case V:                                                                                   \
    if (smem > 48 * 1024)                                                                   \
      cudaFuncSetAttribute(k_page_summarize<T, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                      \
    if (launch_pdl(k_page_summarize<T, V>, grid, dim3(p.threads), smem, st, segs, row_elems, \
                   cw, n_cb, p.nvec, p.R, sc.ctrl) != cudaSuccess)                          \
      return WA_ERR_CUDA;                                                                   \
    break;
    WA_CASE(1) WA_CASE(2) WA_CASE(4) WA_CASE(8)
#undef WA_CASE
    default: return WA_ERR_SHAPE;
  }
  return cuda_status(cudaPeekAtLastError());
}

// Launch shape and scratch layout of one selection (SelectArgs fields derived
// from the problem); returns the scratch floats it needs.
template <typename T>
size_t plan_select(SelectArgs& a, Plan* pl) {
  constexpr int E = VecOf<T>::E;
  const int d = a.head_dim;
  // heads per column block: enough for 32 vectors a row (at most 12 row phases
  // of 384 threads, so a row block of 8 * 12 rows is one batch of loads per
  // thread), a divisor of n_heads; a head row that is not whole 16-byte vectors
  // (or is under 32 values) puts all heads in one block
  if (d % E == 0 && d >= 32) {
    a.hpb = 1;
    while (a.hpb * (d / E) < 32 && a.n_heads % (2 * a.hpb) == 0) a.hpb *= 2;
  } else {
    a.hpb = a.n_heads;
  }
  a.cw = a.hpb * d;
  a.n_cb = (a.n_heads + a.hpb - 1) / a.hpb;
  // query tiles and prompt CTAs in about one wave of two CTAs per SM, at least
  // 16 rows a tile
  int n_rb = (2 * sm_count() - a.n_chunks) / a.n_cb;
  const int max_rb = (a.n_q + 15) / 16;
  if (n_rb > max_rb) n_rb = max_rb;
  if (n_rb < 1) n_rb = 1;
  a.rows_per_block = (a.n_q + n_rb - 1) / n_rb;
  a.n_rb = (a.n_q + a.rows_per_block - 1) / a.rows_per_block;
  *pl = plan_rows<T>(a.cw);
  a.nvec = pl->nvec;
  a.R = pl->R;
  a.n_alpha = a.n_chunks > 0 ? a.n_chunks * a.ppc : a.n_pages;
  const int n_cand = a.n_chunks > 0 ? a.ppc : a.n_pages;
  int n2 = 1;
  while (n2 < n_cand) n2 <<= 1;
  a.n_cand_max2 = n2;
  const size_t part = ((size_t)a.n_cb * a.n_rb * a.cw + 3) & ~(size_t)3;
  const size_t alpha = ((size_t)a.n_heads * a.n_alpha + 3) & ~(size_t)3;
  return part + alpha + (((size_t)a.n_chunks + 3) & ~(size_t)3);
}

// Launch the selection over `scratch` (plan_select's floats) and `ctrl`, whose
// counters kSelectCounter - n_cb .. kSelectCounter must be zero.
template <typename T>
wa_status launch_select(const T* q, SelectArgs a, const Plan& p, float* scratch, Ctrl* ctrl,
                        cudaStream_t st) {
  a.partial = scratch;
  a.alpha_part = scratch + (((size_t)a.n_cb * a.n_rb * a.cw + 3) & ~(size_t)3);
  a.cosv = a.alpha_part + (((size_t)a.n_heads * a.n_alpha + 3) & ~(size_t)3);
  a.ctrl = ctrl;
  // phase A: R rows of cw partial sums; then qbar + the group sums (<= blockDim
  // float4); final stage: alpha, keys and, when they fit in 16 KiB, the staged scores
  size_t smem_a = (size_t)p.R * a.cw * sizeof(float);
  const size_t smem_q = (size_t)a.cw * sizeof(float) + (size_t)p.threads * 16;
  if (smem_q > smem_a) smem_a = smem_q;
  const size_t stage = (size_t)a.n_heads * (a.n_chunks > 0 ? a.ppc : a.n_pages);
  a.stage_floats = stage <= 4096 ? (int)stage : 0;
  const size_t smem_b = (size_t)((a.n_cand_max2 + 3) & ~3) * 4 + (size_t)a.n_cand_max2 * 8 +
                        (size_t)a.stage_floats * 4;
  size_t smem = smem_a > smem_b ? smem_a : smem_b;
  if (smem < (size_t)a.n_chunks * sizeof(float)) smem = (size_t)a.n_chunks * sizeof(float);
  const unsigned grid = (unsigned)(a.n_cb * a.n_rb + a.n_chunks);
  switch (p.vpt) {
#define WA_CASE(V)                                                                          \
  case V:                                                                                   \
    if (smem > 48 * 1024)                                                                   \
      cudaFuncSetAttribute(k_select_pages<T, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                      \
    if (launch_pdl(k_select_pages<T, V>, dim3(grid), dim3(p.threads), smem, st, q, a) !=     \
        cudaSuccess)                                                                        \
      return WA_ERR_CUDA;                                                                   \
    break;
    WA_CASE(1) WA_CASE(2) WA_CASE(4) WA_CASE(8)
#undef WA_CASE
    default: return WA_ERR_SHAPE;
  }
  return cuda_status(cudaPeekAtLastError());
}

template <typename T>
wa_status select_t(const T* q, SelectArgs a, cudaStream_t st) {
  Plan p;
  const size_t floats = plan_select<T>(a, &p);
  Scratch sc;
  wa_status rc = get_scratch(floats * sizeof(float), &sc);
  if (rc != WA_OK) return rc;
  return launch_select<T>(q, a, p, static_cast<float*>(sc.data), sc.ctrl, st);
}

}  // namespace

wa_status launch_page_summarize(const void* k_pages, wa_dtype dt, int n_pages, int page_tokens,
                                int row_elems, float* kbar_out, cudaStream_t s) {
  const SegIn seg{k_pages, n_pages * page_tokens, page_tokens, kbar_out};
  if (dt == WA_BF16) return summarize_t<__nv_bfloat16>(&seg, 1, row_elems, s);
  return summarize_t<float>(&seg, 1, row_elems, s);
}

wa_status launch_block_means(int n_seg, const void* const* xs, const int* n_rows,
                             const int* blocks, wa_dtype dt, int row_elems,
                             float* const* means_out, cudaStream_t s) {
  if (n_seg < 1 || n_seg > kMaxSegs) return WA_ERR_INVALID_ARG;
  SegIn segs[kMaxSegs];
  for (int i = 0; i < n_seg; ++i) segs[i] = SegIn{xs[i], n_rows[i], blocks[i], means_out[i]};
  if (dt == WA_BF16) return summarize_t<__nv_bfloat16>(segs, n_seg, row_elems, s);
  return summarize_t<float>(segs, n_seg, row_elems, s);
}

wa_status launch_select_pages(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                              const float* kbar, int n_pages, const float* prompt_cur,
                              const float* prompt_chunks, int n_chunks, int prompt_dim,
                              int pages_per_chunk, int k_p, int32_t* idx_out, float* scores_out,
                              int32_t* chunk_out, cudaStream_t s, int per_head) {
  SelectArgs a{};
  a.per_head = per_head;
  a.n_q = n_q;
  a.row_elems = n_heads * head_dim;
  a.n_heads = n_heads;
  a.kbar = kbar;
  a.n_pages = n_pages;
  a.head_dim = head_dim;
  a.prompt_cur = prompt_cur;
  a.prompt_chunks = prompt_chunks;
  a.n_chunks = n_chunks;
  a.prompt_dim = prompt_dim;
  a.ppc = pages_per_chunk;
  a.k_p = k_p;
  a.idx_out = idx_out;
  a.scores_out = scores_out;
  a.chunk_out = chunk_out;
  if (dt == WA_BF16) return select_t((const __nv_bfloat16*)q, a, s);
  return select_t((const float*)q, a, s);
}

}  // namespace wa

// ---------------------------------------------------------------------------
// wa_select_pages_noalloc: the same retrieval with its scratch in a fixed
// array compiled into the library instead of the library's cudaMalloc'd
// arena.  For callers that must not allocate device memory once they are
// running: a serving process that has handed all free HBM to its own pool, or
// a latency-critical loop in which a cudaMalloc -- and the device-wide
// synchronize that growing the library's arena implies -- would stall other
// work on the GPU.  There is no counterpart on the pages.
// ---------------------------------------------------------------------------
namespace wa {
namespace {

constexpr size_t kNoAllocPartialBytes = size_t(2) << 20;      // 2 MiB of partial sums
constexpr size_t kNoAllocCtrlBytes = (sizeof(Ctrl) + 255) & ~size_t(255);

// Every device that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocCtrlBytes +
                                                                 kNoAllocPartialBytes];

std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[64] = {};   // device address of the array, per device

// Device address of g_select_scratch on the current device (host code must not
// use the symbol itself: on the host it is only a stand-in).
wa_status noalloc_scratch(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_select_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return WA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return WA_OK;
}

template <typename T>
wa_status select_noalloc_t(const T* q, SelectArgs a, cudaStream_t st) {
  Plan p;
  const size_t floats = plan_select<T>(a, &p);   // the layout of the allocating entry point
  if (floats * sizeof(float) > kNoAllocPartialBytes) return WA_ERR_SHAPE;
  unsigned char* base = nullptr;
  wa_status rc = noalloc_scratch(&base);
  if (rc != WA_OK) return rc;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base);
  // the ticket counters must start at zero; the array keeps the last call's contents
  if (cudaMemsetAsync(&ctrl->counters[kSelectCounter - a.n_cb], 0,
                      (a.n_cb + 1) * sizeof(unsigned), st) != cudaSuccess)
    return WA_ERR_CUDA;
  return launch_select<T>(q, a, p, reinterpret_cast<float*>(base + kNoAllocCtrlBytes), ctrl, st);
}

inline bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace wa

extern "C" wa_status wa_select_pages_noalloc(const void* q, wa_dtype dt, int n_q, int n_heads,
                                             int head_dim, const float* kbar, int n_pages,
                                             const float* prompt_cur, const float* prompt_chunks,
                                             int n_chunks, int prompt_dim, int pages_per_chunk,
                                             int k_p, int32_t* idx_out, float* scores_out,
                                             int32_t* chunk_out, wa_stream_t stream) {
  using namespace wa;
  if (dt != WA_BF16 && dt != WA_F32) return WA_ERR_DTYPE;
  if (!q || !kbar || !idx_out || n_q <= 0 || n_pages <= 0 || k_p <= 0 || n_chunks < 0)
    return WA_ERR_INVALID_ARG;
  if (n_heads <= 0 || head_dim <= 0) return WA_ERR_SHAPE;
  const long long row = (long long)n_heads * head_dim;
  if ((row * (dt == WA_BF16 ? 2 : 4)) % 16 != 0 || row > 8192) return WA_ERR_SHAPE;
  int n_cand = n_pages;
  if (n_chunks > 0) {
    if (!prompt_cur || !prompt_chunks || prompt_dim <= 0 || pages_per_chunk <= 0)
      return WA_ERR_INVALID_ARG;
    if ((long long)n_chunks * pages_per_chunk > n_pages) return WA_ERR_INVALID_ARG;
    n_cand = pages_per_chunk;
  }
  if (k_p > n_cand || k_p > 1024) return WA_ERR_INVALID_ARG;
  if (n_cand > 8192) return WA_ERR_SHAPE;
  if (!aligned16_ptr(q) || !aligned16_ptr(kbar)) return WA_ERR_ALIGN;
  SelectArgs a{};
  a.n_q = n_q;
  a.row_elems = (int)row;
  a.n_heads = n_heads;
  a.kbar = kbar;
  a.n_pages = n_pages;
  a.head_dim = head_dim;
  a.prompt_cur = prompt_cur;
  a.prompt_chunks = prompt_chunks;
  a.n_chunks = n_chunks;
  a.prompt_dim = prompt_dim;
  a.ppc = pages_per_chunk;
  a.k_p = k_p;
  a.idx_out = idx_out;
  a.scores_out = scores_out;
  a.chunk_out = chunk_out;
  cudaStream_t st = (cudaStream_t)stream;
  if (dt == WA_BF16) return select_noalloc_t((const __nv_bfloat16*)q, a, st);
  return select_noalloc_t((const float*)q, a, st);
}
