// Block selection of the HSA sparse branch (WorldAttention review page, HSA
// section and its appendix notes on the sparse branch): a pooled attention map
// between query-block means and key-block means, each head's block mass, the
// Gini coefficient of that mass, and the minimal set of blocks whose
// cumulative mass reaches the head's threshold.
//
// k_pooled_scores  S[h][qb][kb] = scale * Qbar_qb,h . Kbar_kb,h: one thread per
//                  (query block, key block) in 32 x 32 tiles, rows staged in
//                  shared memory.
// k_sparse_select  one CTA per head:
//   1. each query-block row's max and exp-sum (a warp per row, fixed order);
//   2. mass[kb] = mean over query blocks of the row-normalised exp (fixed order);
//   3. blocks ordered by (mass descending, index ascending): one bitonic sort
//      of (inverted mass bits, index) keys (mass >= 0, so the bit pattern
//      orders it);
//   4. Gini coefficient from that order (the ascending order reversed: equal
//      masses in another order leave the sum unchanged), tau = 1 - G unless
//      the caller gives tau[h];
//   5. cumulative mass by an inclusive scan in the sorted order; the first
//      position reaching tau ends the kept set (at least one block);
//   6. the kept blocks written in ascending block order (scan of flags).
// Every reduction and scan has a fixed order, so the result is deterministic.
#include <atomic>
#include <math.h>

#include "wa_internal.cuh"

namespace wa {
namespace {

constexpr int kScoreThreads = 1024;     // 32 query blocks x 32 key blocks per CTA
constexpr int kMaxQb = 4096;
constexpr int kSelThreads = 1024;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(kScoreThreads)
k_pooled_scores(const float* __restrict__ qbar, int n_qb, const float* __restrict__ kbar, int n_kb,
                int n_heads, int d, float scale, float* __restrict__ scores) {
  // CTA: 32 query blocks x 32 key blocks of one head; warp w = query block
  // qb0 + w, lane = key block kb0 + lane; rows staged in shared memory with
  // a 4-float pad (16-byte reads of 8 lanes hit distinct banks)
  extern __shared__ __align__(16) float sm[];
  const int h = blockIdx.z;
  const int kb0 = blockIdx.x * 32, qb0 = blockIdx.y * 32;
  const int dp = d + 4;
  float* q_s = sm;                // [32][d + 4]
  float* k_s = sm + 32 * dp;      // [32][d + 4]
  const int d4 = d / 4;
  for (int i = threadIdx.x; i < 32 * d4; i += blockDim.x) {
    const int r = i / d4, c = (i % d4) * 4;
    const int qb = qb0 + r, kb = kb0 + r;
    const float4 zq = qb < n_qb ? *reinterpret_cast<const float4*>(qbar + ((size_t)qb * n_heads + h) * d + c)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 zk = kb < n_kb ? *reinterpret_cast<const float4*>(kbar + ((size_t)kb * n_heads + h) * d + c)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(q_s + r * dp + c) = zq;
    *reinterpret_cast<float4*>(k_s + r * dp + c) = zk;
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = qb0 + w, kb = kb0 + lane;
  const float4* qr = reinterpret_cast<const float4*>(q_s + w * dp);
  const float4* kr = reinterpret_cast<const float4*>(k_s + lane * dp);
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
  for (int e = 0; e < d4; ++e) {
    const float4 a = qr[e], b = kr[e];
    acc0 = fmaf(a.x, b.x, acc0);
    acc1 = fmaf(a.y, b.y, acc1);
    acc0 = fmaf(a.z, b.z, acc0);
    acc1 = fmaf(a.w, b.w, acc1);
  }
  if (qb < n_qb && kb < n_kb) scores[((size_t)h * n_qb + qb) * n_kb + kb] = (acc0 + acc1) * scale;
}

// Ascending bitonic sort of n2 (power of two) keys in shared memory.
__device__ void bitonic_sort(unsigned long long* keys, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const unsigned long long a = keys[i], b = keys[ixj];
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// The same ascending sort for n2 <= blockDim.x keys, one per thread: stages
// whose partner is under 32 positions away exchange by warp shuffles, wider
// ones through shared memory (10 of the 45 stages for 512 keys need a barrier,
// against every stage above).  The keys are distinct, so the result is the
// same permutation.
__device__ void bitonic_sort_small(unsigned long long* keys, int n2) {
  const int i = threadIdx.x;
  const bool live = i < n2;
  const bool warp_live = (i & ~31) < n2;   // warp-uniform: warps wholly past n2 only meet barriers
  unsigned long long v = live ? keys[i] : ~0ull;
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        __syncthreads();   // the previous exchange has been read
        if (live) keys[i] = v;
        __syncthreads();
      }
      if (warp_live) {
        const unsigned long long w =
            j >= 32 ? (live ? keys[i ^ j] : ~0ull) : __shfl_xor_sync(0xffffffffu, v, j);
        // in an ascending run the lower position keeps the smaller key
        const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
        v = keep_min ? (v < w ? v : w) : (v < w ? w : v);
      }
    }
  }
  __syncthreads();
  if (live) keys[i] = v;
  __syncthreads();
}

__device__ void sort_keys(unsigned long long* keys, int n2) {
  if (n2 <= (int)blockDim.x)
    bitonic_sort_small(keys, n2);
  else
    bitonic_sort(keys, n2);
}

// Inclusive scan of x[0..n2) in place (Hillis-Steele, fixed order); tmp has n2 floats.
__device__ void scan_inclusive(float* x, float* tmp, int n2) {
  for (int off = 1; off < n2; off <<= 1) {
    for (int i = threadIdx.x; i < n2; i += blockDim.x) tmp[i] = x[i] + (i >= off ? x[i - off] : 0.f);
    __syncthreads();
    for (int i = threadIdx.x; i < n2; i += blockDim.x) x[i] = tmp[i];
    __syncthreads();
  }
}

// Sum of v over the CTA in a fixed order (warp butterflies, then across warps).
__device__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  return warp_sum(lane < nwarps ? red[lane] : 0.f);
}

template <bool kStage>
__global__ void __launch_bounds__(kSelThreads)
k_sparse_select(const float* __restrict__ scores, int n_qb, int n_kb, const float* __restrict__ tau,
                int32_t* __restrict__ sel, int32_t* __restrict__ count, float* __restrict__ gini_out,
                float* __restrict__ mass_out, int n2) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem_raw);   // [n2]
  float* mass = reinterpret_cast<float*>(keys + n2);                           // [n2]
  float* cum = mass + n2;                                                      // [n2]
  float* tmp = cum + n2;                                                       // [n2]
  float* red = tmp + n2;                                                       // [32]
  float* row_max = red + 32;                                                   // [n_qb]
  float* row_inv = row_max + n_qb;                                             // [n_qb]
  const float* sh = scores + (size_t)h * n_qb * n_kb;
  if (kStage) {
    // the head's score slab in shared memory (n_qb * n_kb floats, 16-byte chunks)
    const int off = 5 * n2 + 32 + 2 * n_qb;                 // floats before the slab
    float* stage = reinterpret_cast<float*>(smem_raw) + off + ((4 - (off & 3)) & 3);
    const int n = n_qb * n_kb;
    const float4* src4 = reinterpret_cast<const float4*>(sh);
    float4* dst4 = reinterpret_cast<float4*>(stage);
    for (int i = tid; i < n / 4; i += blockDim.x) dst4[i] = __ldg(src4 + i);
    for (int i = (n / 4) * 4 + tid; i < n; i += blockDim.x) stage[i] = __ldg(sh + i);
    __syncthreads();
    sh = stage;
  }
  // 1. per query-block row: max and 1 / sum of exp
  for (int qb = warp; qb < n_qb; qb += nwarps) {
    const float* row = sh + (size_t)qb * n_kb;
    float mx = -INFINITY;
    for (int kb = lane; kb < n_kb; kb += 32) mx = fmaxf(mx, row[kb]);
    mx = warp_max(mx);
    float s = 0.f;
    for (int kb = lane; kb < n_kb; kb += 32) s += expf(row[kb] - mx);
    s = warp_sum(s);
    if (lane == 0) {
      row_max[qb] = mx;
      row_inv[qb] = 1.0f / s;
    }
  }
  __syncthreads();
  // 2. block mass, summed over query blocks in order
  const float inv_q = 1.0f / (float)n_qb;
  for (int kb = tid; kb < n2; kb += blockDim.x) {
    float acc = 0.f;
    if (kb < n_kb) {
#pragma unroll 8
      for (int qb = 0; qb < n_qb; ++qb) acc += expf(sh[(size_t)qb * n_kb + kb] - row_max[qb]) * row_inv[qb];
    }
    mass[kb] = kb < n_kb ? acc * inv_q : 0.f;
    keys[kb] = kb < n_kb ? ((unsigned long long)(~__float_as_uint(acc * inv_q)) << 32) | (unsigned)kb
                         : ~0ull;
  }
  __syncthreads();
  // 3. mass descending, index ascending
  sort_keys(keys, n2);
  // 4. Gini coefficient G = sum_i (2i - n - 1) x_(i) / (n sum x) over the
  //    ascending order x_(1..n); position j of the descending order is i = n - j
  float num = 0.f, tot = 0.f;
  for (int j = tid; j < n_kb; j += blockDim.x) {
    const float x = mass[(unsigned)(keys[j] & 0xffffffffu)];
    num += (float)(n_kb - 1 - 2 * j) * x;
    tot += x;
  }
  num = block_sum(num, red);
  tot = block_sum(tot, red);
  const float g = tot > 0.f ? num / ((float)n_kb * tot) : 0.f;
  const float t = tau ? tau[h] : 1.0f - g;
  // 5. cumulative mass in the sorted order
  for (int i = tid; i < n2; i += blockDim.x)
    cum[i] = i < n_kb ? mass[(unsigned)(keys[i] & 0xffffffffu)] : 0.f;
  __syncthreads();
  scan_inclusive(cum, tmp, n2);
  // kept = 1 + the number of positions whose cumulative mass is still below tau
  float below = 0.f;
  for (int i = tid; i < n_kb; i += blockDim.x) below += (cum[i] < t) ? 1.f : 0.f;
  below = block_sum(below, red);
  int kept = (int)below + 1;
  if (kept > n_kb) kept = n_kb;
  // 6. kept blocks in ascending block order
  __syncthreads();
  for (int i = tid; i < n2; i += blockDim.x) cum[i] = 0.f;
  __syncthreads();
  for (int i = tid; i < kept; i += blockDim.x) cum[(unsigned)(keys[i] & 0xffffffffu)] = 1.f;
  __syncthreads();
  scan_inclusive(cum, tmp, n2);
  for (int kb = tid; kb < n_kb; kb += blockDim.x) {
    const float prev = kb == 0 ? 0.f : cum[kb - 1];
    if (cum[kb] - prev > 0.5f) sel[(size_t)h * n_kb + (int)(cum[kb] + 0.5f) - 1] = kb;
    if (mass_out) mass_out[(size_t)h * n_kb + kb] = mass[kb];
  }
  if (tid == 0) {
    count[h] = kept;
    if (gini_out) gini_out[h] = g;
  }
}

}  // namespace

wa_status launch_sparse_select(const float* qbar, int n_qb, const float* kbar, int n_kb,
                               int n_heads, int head_dim, float scale, const float* tau,
                               int32_t* sel_out, int32_t* count_out, float* gini_out,
                               float* mass_out, cudaStream_t s) {
  Scratch sc;
  const size_t score_bytes = (size_t)n_heads * n_qb * n_kb * sizeof(float);
  wa_status rc = get_scratch(score_bytes, &sc);
  if (rc != WA_OK) return rc;
  float* scores = static_cast<float*>(sc.data);
  const size_t smem1 = (size_t)64 * (head_dim + 4) * sizeof(float);
  static std::atomic<bool> attr_done[64];   // per device; setting it twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  int n2 = 1;
  while (n2 < n_kb) n2 <<= 1;
  const size_t smem2 = (size_t)n2 * 8 + (size_t)3 * n2 * 4 + 32 * 4 + (size_t)2 * n_qb * 4;
  // the score slab goes to shared memory when it fits (scores are in the scratch arena, so
  // the slab offset of every head keeps 16-byte alignment when n_qb * n_kb % 4 == 0)
  const size_t slab = (size_t)n_qb * n_kb * sizeof(float) + 16;
  const bool stage = smem2 + slab <= 220 * 1024 && ((size_t)n_qb * n_kb) % 4 == 0;
  if (dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k_pooled_scores, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024) != cudaSuccess ||
        cudaFuncSetAttribute(k_sparse_select<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024) != cudaSuccess ||
        cudaFuncSetAttribute(k_sparse_select<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024) != cudaSuccess)
      return WA_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  dim3 g1((n_kb + 31) / 32, (n_qb + 31) / 32, n_heads);
  k_pooled_scores<<<g1, kScoreThreads, smem1, s>>>(qbar, n_qb, kbar, n_kb, n_heads, head_dim, scale,
                                                    scores);
  if (stage)
    k_sparse_select<true><<<n_heads, kSelThreads, smem2 + slab, s>>>(
        scores, n_qb, n_kb, tau, sel_out, count_out, gini_out, mass_out, n2);
  else
    k_sparse_select<false><<<n_heads, kSelThreads, smem2, s>>>(
        scores, n_qb, n_kb, tau, sel_out, count_out, gini_out, mass_out, n2);
  return cuda_status(cudaPeekAtLastError());
}

// Limits the host checks before launch_sparse_select.
int sparse_select_max_qb() { return kMaxQb; }
size_t sparse_select_smem(int n_qb, int n_kb, int head_dim) {
  int n2 = 1;
  while (n2 < n_kb) n2 <<= 1;
  const size_t s1 = (size_t)64 * (head_dim + 4) * sizeof(float);
  const size_t s2 = (size_t)n2 * 8 + (size_t)3 * n2 * 4 + 32 * 4 + (size_t)2 * n_qb * 4;
  return s1 > s2 ? s1 : s2;
}

}  // namespace wa
