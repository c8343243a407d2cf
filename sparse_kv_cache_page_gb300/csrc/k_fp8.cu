// Compressed DRAM tier: FP8 E4M3 page codec.
//
// WorldAttention (review page), HKV tiers: pages not in use live in CPU DRAM
// and return over the CPU-GPU link, which bounds the long-video (stress)
// workload.  Storing those pages as FP8 halves the bytes that cross the link.
// Each (token, head) row of d values keeps one fp32 scale:
//   s = amax(|row|) / 448,  code = E4M3 round-to-nearest-even(x / s)
// (IEEE fp32 divisions, `cvt.rn.satfinite.e4m3x2.f32`), and decoding gives
//   bf16 RNE( fp32(value(code) * s) ).
// A zero row has s = 0 and codes 0.
//
// One warp per row (d = 32 e, e in {2, 4, 8} values per lane), four rows in
// flight per warp.  The
// gather-decode kernel reads the selected pages' codes and scales where they
// live -- device memory or pinned host memory through its device mapping, so
// a fetch from the DRAM tier moves the FP8 bytes only -- and writes the bf16
// attention buffer.
#include <cuda_fp16.h>

#include "wa_internal.cuh"

namespace wa {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;      // rows per warp per step

__device__ __forceinline__ uint16_t enc2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 dec2(uint16_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);   // .x = lower byte's value, .y = upper byte's
}

template <int E>
struct Vec;
template <> struct Vec<2> { using In = uint32_t; using Code = uint16_t; };
template <> struct Vec<4> { using In = uint2; using Code = uint32_t; };
template <> struct Vec<8> { using In = uint4; using Code = uint2; };

template <int E>
__device__ __forceinline__ void unpack_bf16(const typename Vec<E>::In& in, float (&x)[E]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&in);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Each warp takes kRows consecutive rows per step: their loads are issued
// together, so enough bytes are in flight to stream at HBM (or link) speed.
template <int E>
__global__ void __launch_bounds__(kThreads)
k_fp8_encode(const __nv_bfloat16* __restrict__ src, size_t n_rows, uint8_t* __restrict__ codes,
             float* __restrict__ scales) {
  using In = typename Vec<E>::In;
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
      unpack_bf16<E>(in[j], x);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = __fdiv_rn(amax, 448.0f);
      typename Vec<E>::Code out;
      uint16_t* o16 = reinterpret_cast<uint16_t*>(&out);
#pragma unroll
      for (int i = 0; i < E / 2; ++i)
        o16[i] = s > 0.f ? enc2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s)) : (uint16_t)0;
      reinterpret_cast<typename Vec<E>::Code*>(codes + r * 32 * E)[lane] = out;
      if (lane == 0) scales[r] = s;
    }
  }
}

// out[s*P + t][h] = decode(pages[idx[s]][t][h]); idx NULL: out row r = row r.
template <int E>
__global__ void __launch_bounds__(kThreads)
k_fp8_decode(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
             const int32_t* __restrict__ idx, int n_pages, size_t page_rows, size_t n_rows,
             __nv_bfloat16* __restrict__ out, Ctrl* ctrl) {
  using Code = typename Vec<E>::Code;
  const int lane = threadIdx.x & 31;
  const size_t step = (size_t)gridDim.x * (kThreads / 32) * kRows;
  for (size_t r0 = ((size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kRows; r0 < n_rows;
       r0 += step) {
    Code c[kRows];
    float sc[kRows];
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
        c[j] = reinterpret_cast<const Code*>(codes + src_row * 32 * E)[lane];
        sc[j] = scales[src_row];
      }
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const size_t r = r0 + j;
      if (r >= n_rows) break;
      typename Vec<E>::In o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
      if (bad[j]) {
#pragma unroll
        for (int i = 0; i < E / 2; ++i) ow[i] = 0u;
        if (lane == 0 && r % page_rows == 0) atomicOr(&ctrl->status, kStatusIndex);
      } else {
        const uint16_t* c16 = reinterpret_cast<const uint16_t*>(&c[j]);
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
          const float2 v = dec2(c16[i]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(__fmul_rn(v.x, sc[j]));
          const __nv_bfloat16 hi = __float2bfloat16_rn(__fmul_rn(v.y, sc[j]));
          ow[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
        }
      }
      reinterpret_cast<typename Vec<E>::In*>(out + r * 32 * E)[lane] = o;
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

wa_status launch_fp8_encode(const void* src, size_t n_rows, int head_dim, void* codes,
                            float* scales, cudaStream_t s) {
  const unsigned g = grid_for(n_rows);
  const auto* x = static_cast<const __nv_bfloat16*>(src);
  auto* c = static_cast<uint8_t*>(codes);
  switch (head_dim / 32) {
    case 2: k_fp8_encode<2><<<g, kThreads, 0, s>>>(x, n_rows, c, scales); break;
    case 4: k_fp8_encode<4><<<g, kThreads, 0, s>>>(x, n_rows, c, scales); break;
    case 8: k_fp8_encode<8><<<g, kThreads, 0, s>>>(x, n_rows, c, scales); break;
    default: return WA_ERR_SHAPE;
  }
  return cuda_status(cudaPeekAtLastError());
}

wa_status launch_fp8_decode(const void* codes, const float* scales, const int32_t* idx, int n_pages,
                            size_t page_rows, size_t n_rows, int head_dim, void* out,
                            cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const unsigned g = grid_for(n_rows);
  const auto* c = static_cast<const uint8_t*>(codes);
  auto* o = static_cast<__nv_bfloat16*>(out);
  switch (head_dim / 32) {
    case 2: k_fp8_decode<2><<<g, kThreads, 0, s>>>(c, scales, idx, n_pages, page_rows, n_rows, o, ctrl); break;
    case 4: k_fp8_decode<4><<<g, kThreads, 0, s>>>(c, scales, idx, n_pages, page_rows, n_rows, o, ctrl); break;
    case 8: k_fp8_decode<8><<<g, kThreads, 0, s>>>(c, scales, idx, n_pages, page_rows, n_rows, o, ctrl); break;
    default: return WA_ERR_SHAPE;
  }
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa
