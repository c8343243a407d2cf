// Compressed DRAM tier, NVFP4 form: E2M1 codes with E4M3 scales per 16-element
// block and one fp32 scale per (token, head) row.
//
// WorldAttention (review page), HKV tiers: pages not in use live in CPU DRAM
// and return over the CPU-GPU link.  FP4 storage with per-block scales moves
// 76 bytes per 128-value row instead of 256 (bf16) or 132 (the FP8 form).
// Per row of d values:
//   g  = amax(|row|) / 2688                       (2688 = 6 * 448)
//   sb = E4M3 RNE( amax(|block|) / (6 g) )        per block of 16
//   c  = E2M1 RNE, saturating at 6, of x / (sb g)
// every quotient and product one IEEE fp32 operation, in that order; codes
// pack two elements per byte (the even element in the low nibble).  Decoding
// gives bf16 RNE( fp32(value(c) * fp32(value(sb) * g)) ).
//
// One warp per row, E = d / 32 values per lane, a block spans 16 / E lanes,
// four rows in flight per warp.  The gather-decode reads codes and scales
// where they live (device memory or pinned host memory through its device
// mapping) and writes the bf16 attention buffer.
#include <cuda_fp16.h>

#include "wa_internal.cuh"

namespace wa {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;      // rows per warp per step

// two fp32 -> one byte of E2M1 codes: `lo` in bits 0-3, `hi` in bits 4-7
__device__ __forceinline__ uint32_t enc_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}
// one byte of E2M1 codes -> the two values (x: low nibble, y: high nibble)
__device__ __forceinline__ float2 dec_e2m1x2(uint32_t c) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(c));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}
// fp32 -> E4M3 code (round to nearest even, saturating) and back
__device__ __forceinline__ uint32_t enc_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}
__device__ __forceinline__ float dec_e4m3(uint32_t c) {
  uint32_t h2;
  const uint16_t c16 = (uint16_t)c;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
  return __low2float(*reinterpret_cast<const __half2*>(&h2));
}

template <int E> struct V;
template <> struct V<2> { using In = uint32_t; using Code = uint8_t; };
template <> struct V<4> { using In = uint2; using Code = uint16_t; };
template <> struct V<8> { using In = uint4; using Code = uint32_t; };

template <int E>
__device__ __forceinline__ void unpack(const typename V<E>::In& in, float (&x)[E]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&in);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int E>
__global__ void __launch_bounds__(kThreads)
k_nvfp4_encode(const __nv_bfloat16* __restrict__ src, size_t n_rows, uint8_t* __restrict__ codes,
               uint8_t* __restrict__ bscales, float* __restrict__ rscales) {
  using In = typename V<E>::In;
  constexpr int L = 16 / E;               // lanes per block
  constexpr int NB = 2 * E;               // blocks per row (d / 16)
  const int lane = threadIdx.x & 31;
  const size_t step = (size_t)gridDim.x * (kThreads / 32) * kRows;
  for (size_t r0 = ((size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kRows; r0 < n_rows;
       r0 += step) {
    In in[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j)
      if (r0 + j < n_rows) in[j] = __ldcs(reinterpret_cast<const In*>(src + (r0 + j) * 32 * E) + lane);
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      if (r0 + j >= n_rows) break;
      const size_t r = r0 + j;
      float x[E];
      unpack<E>(in[j], x);
      float lmax = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) lmax = fmaxf(lmax, fabsf(x[i]));
      float amax = lmax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      float bmax = lmax;                   // this lane's block
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
      const float g = __fdiv_rn(amax, 2688.0f);
      const float den = __fmul_rn(g, 6.0f);
      const uint32_t sb = den > 0.f ? enc_e4m3(__fdiv_rn(bmax, den)) : 0u;
      const float es = __fmul_rn(dec_e4m3(sb), g);
      typename V<E>::Code out = 0;
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        const uint32_t byte = es > 0.f ? enc_e2m1x2(__fdiv_rn(x[2 * i], es), __fdiv_rn(x[2 * i + 1], es))
                                       : 0u;
        out |= (typename V<E>::Code)(byte << (8 * i));
      }
      reinterpret_cast<typename V<E>::Code*>(codes + r * 16 * E)[lane] = out;
      if (lane % L == 0) bscales[r * NB + lane / L] = (uint8_t)sb;
      if (lane == 0) rscales[r] = g;
    }
  }
}

// out[s*P + t][h] = decode(pages[idx[s]][t][h]); idx NULL: out row r = row r.
template <int E>
__global__ void __launch_bounds__(kThreads)
k_nvfp4_decode(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ bscales,
               const float* __restrict__ rscales, const int32_t* __restrict__ idx, int n_pages,
               size_t page_rows, size_t n_rows, __nv_bfloat16* __restrict__ out, Ctrl* ctrl) {
  using Code = typename V<E>::Code;
  constexpr int L = 16 / E;
  constexpr int NB = 2 * E;
  const int lane = threadIdx.x & 31;
  const size_t step = (size_t)gridDim.x * (kThreads / 32) * kRows;
  for (size_t r0 = ((size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kRows; r0 < n_rows;
       r0 += step) {
    Code c[kRows];
    uint32_t sb[kRows];
    float g[kRows];
    bool bad[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const size_t r = r0 + j;
      bad[j] = false;
      if (r >= n_rows) continue;
      size_t src_row = r;
      if (idx) {
        const int page = __ldg(idx + r / page_rows);
        bad[j] = page < 0 || page >= n_pages;
        src_row = (size_t)(bad[j] ? 0 : page) * page_rows + r % page_rows;
      }
      if (!bad[j]) {
        c[j] = reinterpret_cast<const Code*>(codes + src_row * 16 * E)[lane];
        sb[j] = bscales[src_row * NB + lane / L];
        g[j] = rscales[src_row];
      }
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const size_t r = r0 + j;
      if (r >= n_rows) break;
      typename V<E>::In o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
      if (bad[j]) {
#pragma unroll
        for (int i = 0; i < E / 2; ++i) ow[i] = 0u;
        if (lane == 0 && r % page_rows == 0) atomicOr(&ctrl->status, kStatusIndex);
      } else {
        const float es = __fmul_rn(dec_e4m3(sb[j]), g[j]);
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
          const float2 v = dec_e2m1x2((uint32_t)(c[j] >> (8 * i)) & 0xFFu);
          const __nv_bfloat16 lo = __float2bfloat16_rn(__fmul_rn(v.x, es));
          const __nv_bfloat16 hi = __float2bfloat16_rn(__fmul_rn(v.y, es));
          ow[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
        }
      }
      reinterpret_cast<typename V<E>::In*>(out + r * 32 * E)[lane] = o;
    }
  }
}

unsigned grid_for(size_t rows) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t per_block = (size_t)(kThreads / 32) * kRows;
  const size_t need = (rows + per_block - 1) / per_block;
  const size_t cap = (size_t)sms * 8;
  return (unsigned)(need < cap ? need : cap);
}

}  // namespace

wa_status launch_nvfp4_encode(const void* src, size_t n_rows, int head_dim, void* codes,
                              void* bscales, float* rscales, cudaStream_t s) {
  const unsigned g = grid_for(n_rows);
  const auto* x = static_cast<const __nv_bfloat16*>(src);
  auto* c = static_cast<uint8_t*>(codes);
  auto* b = static_cast<uint8_t*>(bscales);
  switch (head_dim / 32) {
    case 2: k_nvfp4_encode<2><<<g, kThreads, 0, s>>>(x, n_rows, c, b, rscales); break;
    case 4: k_nvfp4_encode<4><<<g, kThreads, 0, s>>>(x, n_rows, c, b, rscales); break;
    case 8: k_nvfp4_encode<8><<<g, kThreads, 0, s>>>(x, n_rows, c, b, rscales); break;
    default: return WA_ERR_SHAPE;
  }
  return cuda_status(cudaPeekAtLastError());
}

wa_status launch_nvfp4_decode(const void* codes, const void* bscales, const float* rscales,
                              const int32_t* idx, int n_pages, size_t page_rows, size_t n_rows,
                              int head_dim, void* out, cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const unsigned g = grid_for(n_rows);
  const auto* c = static_cast<const uint8_t*>(codes);
  const auto* b = static_cast<const uint8_t*>(bscales);
  auto* o = static_cast<__nv_bfloat16*>(out);
  switch (head_dim / 32) {
    case 2: k_nvfp4_decode<2><<<g, kThreads, 0, s>>>(c, b, rscales, idx, n_pages, page_rows, n_rows, o, ctrl); break;
    case 4: k_nvfp4_decode<4><<<g, kThreads, 0, s>>>(c, b, rscales, idx, n_pages, page_rows, n_rows, o, ctrl); break;
    case 8: k_nvfp4_decode<8><<<g, kThreads, 0, s>>>(c, b, rscales, idx, n_pages, page_rows, n_rows, o, ctrl); break;
    default: return WA_ERR_SHAPE;
  }
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa
