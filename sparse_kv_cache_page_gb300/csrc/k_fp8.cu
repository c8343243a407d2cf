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
// A lane per 16-value chunk of a row (d / 16 lanes per row), two row groups in
// flight per warp.  The
// gather-decode kernel reads the selected pages' codes and scales where they
// live -- device memory or pinned host memory through its device mapping, so
// a fetch from the DRAM tier moves the FP8 bytes only -- and writes the bf16
// attention buffer.
#include <cuda_fp16.h>

#include "codec_math.cuh"
#include "wa_internal.cuh"

namespace wa {
namespace {

using namespace codec;

constexpr int kThreads = 256;

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

// Each lane owns a 16-value chunk of a row (LPR = d / 16 lanes per row, 32 / LPR
// rows per warp step): a 32-byte load, the row maximum over the row's lanes,
// 16 codes (one 16-byte store), the quotients two at a time in packed fp32.
// kSteps row groups are in flight per warp.
constexpr int kSteps = 2;
constexpr int kDecSteps = 4;   // decoding: more row groups in flight (reads are small)

template <int LPR>
__global__ void __launch_bounds__(kThreads)
k_fp8_encode(const __nv_bfloat16* __restrict__ src, size_t n_rows, uint8_t* __restrict__ codes,
             float* __restrict__ scales) {
  constexpr int RPW = 32 / LPR;                 // rows per warp step
  constexpr int D = 16 * LPR;
  const int lane = threadIdx.x & 31, sub = lane / LPR, b = lane % LPR;
  const size_t warps = (size_t)gridDim.x * (kThreads / 32);
  const float r448 = __frcp_rn(448.0f);
  for (size_t g0 = ((size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * RPW * kSteps;
       g0 < n_rows; g0 += warps * RPW * kSteps) {
    uint4 in[kSteps][2];
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
      const size_t r = g0 + (size_t)k * RPW + sub;
      in[k][0] = in[k][1] = make_uint4(0, 0, 0, 0);
      if (r < n_rows) {
        const uint4* p = reinterpret_cast<const uint4*>(src + r * D + 16 * b);
        in[k][0] = __ldcs(p);
        in[k][1] = __ldcs(p + 1);
      }
    }
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
      const size_t r = g0 + (size_t)k * RPW + sub;
      const bool live = r < n_rows;             // uniform within a row's lanes
      const uint32_t w[8] = {in[k][0].x, in[k][0].y, in[k][0].z, in[k][0].w,
                             in[k][1].x, in[k][1].y, in[k][1].z, in[k][1].w};
      float amax = absmax16_bf16(w);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (!live) continue;
      const float s = dividend_ok(amax) ? div_rn(amax, 448.0f, r448) : __fdiv_rn(amax, 448.0f);
      uint32_t out[4];
      uint16_t* o16 = reinterpret_cast<uint16_t*>(out);
      if (div_fast_ok(s)) {
        const uint64_t nb2 = dup2(-s), r2 = dup2(__frcp_rn(s));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float q0, q1;
          div2_rn(q0, q1, bf16_lo(w[i]), bf16_hi(w[i]), nb2, r2);
          o16[i] = enc2(q0, q1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o16[i] = s > 0.f ? enc2(__fdiv_rn(bf16_lo(w[i]), s), __fdiv_rn(bf16_hi(w[i]), s))
                           : (uint16_t)0;
      }
      *reinterpret_cast<uint4*>(codes + r * D + 16 * b) = make_uint4(out[0], out[1], out[2], out[3]);
      if (b == 0) scales[r] = s;
    }
  }
}

// out[s*P + t][h] = decode(pages[idx[s]][t][h]); idx NULL: out row r = row r.
template <int LPR>
__global__ void __launch_bounds__(kThreads)
k_fp8_decode(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
             const int32_t* __restrict__ idx, int n_pages, size_t page_rows, size_t n_rows,
             __nv_bfloat16* __restrict__ out, Ctrl* ctrl) {
  constexpr int RPW = 32 / LPR;
  constexpr int D = 16 * LPR;
  const int lane = threadIdx.x & 31, sub = lane / LPR, b = lane % LPR;
  const size_t warps = (size_t)gridDim.x * (kThreads / 32);
  for (size_t g0 = ((size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * RPW * kDecSteps;
       g0 < n_rows; g0 += warps * RPW * kDecSteps) {
    uint4 c[kDecSteps];
    float sc[kDecSteps];
    bool bad[kDecSteps];
#pragma unroll
    for (int k = 0; k < kDecSteps; ++k) {
      const size_t r = g0 + (size_t)k * RPW + sub;
      bad[k] = false;
      if (r >= n_rows) continue;
      size_t src_row = r;
      if (idx) {
        const int page = __ldg(idx + r / page_rows);
        bad[k] = page < 0 || page >= n_pages;
        src_row = (size_t)(bad[k] ? 0 : page) * page_rows + r % page_rows;
      }
      if (!bad[k]) {
        c[k] = *reinterpret_cast<const uint4*>(codes + src_row * D + 16 * b);
        sc[k] = scales[src_row];
      }
    }
#pragma unroll
    for (int k = 0; k < kDecSteps; ++k) {
      const size_t r = g0 + (size_t)k * RPW + sub;
      if (r >= n_rows) continue;
      uint32_t o[8];
      if (bad[k]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = 0u;
        if (b == 0 && r % page_rows == 0) atomicOr(&ctrl->status, kStatusIndex);
      } else {
        const uint16_t* c16 = reinterpret_cast<const uint16_t*>(&c[k]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 v = dec2(c16[i]);
          float lo, hi;
          fmul2(lo, hi, v.x, v.y, sc[k], sc[k]);
          o[i] = bf16x2(lo, hi);
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(out + r * D + 16 * b);
      __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
      __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
    }
  }
}

// Blocks for n_rows rows: one per row group, at most `cap`.  The encoder takes
// the resident block count (every block starts at once: 0.075 against 0.079 ms
// with 8 blocks per SM, 8 pages); the decoder, whose traffic is mostly writes,
// 8 blocks per SM, more than fit at once, so that blocks that start late fill
// the SMs that finish early (0.084 against 0.087 ms with the resident count).
inline unsigned grid_for(size_t rows, int head_dim, int steps, size_t cap) {
  const size_t per_block = (size_t)(kThreads / 32) * (512 / head_dim) * steps;
  const size_t need = (rows + per_block - 1) / per_block;
  return (unsigned)(need < cap ? need : cap);
}

}  // namespace

wa_status launch_fp8_encode(const void* src, size_t n_rows, int head_dim, void* codes,
                            float* scales, cudaStream_t s) {
  const auto* x = static_cast<const __nv_bfloat16*>(src);
  auto* c = static_cast<uint8_t*>(codes);
  auto run = [&](auto kernel) {
    if (n_rows == 0) return WA_OK;
    kernel<<<grid_for(n_rows, head_dim, kSteps, resident_blocks(kernel, kThreads)), kThreads, 0,
             s>>>(x, n_rows, c, scales);
    return cuda_status(cudaPeekAtLastError());
  };
  switch (head_dim / 16) {
    case 4: return run(k_fp8_encode<4>);
    case 8: return run(k_fp8_encode<8>);
    case 16: return run(k_fp8_encode<16>);
    default: return WA_ERR_SHAPE;
  }
}

wa_status launch_fp8_decode(const void* codes, const float* scales, const int32_t* idx, int n_pages,
                            size_t page_rows, size_t n_rows, int head_dim, void* out,
                            cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const auto* c = static_cast<const uint8_t*>(codes);
  auto* o = static_cast<__nv_bfloat16*>(out);
  auto run = [&](auto kernel) {
    if (n_rows == 0) return WA_OK;
    kernel<<<grid_for(n_rows, head_dim, kDecSteps, (size_t)sm_count() * 8), kThreads, 0, s>>>(
        c, scales, idx, n_pages, page_rows, n_rows, o, ctrl);
    return cuda_status(cudaPeekAtLastError());
  };
  switch (head_dim / 16) {
    case 4: return run(k_fp8_decode<4>);
    case 8: return run(k_fp8_decode<8>);
    case 16: return run(k_fp8_decode<16>);
    default: return WA_ERR_SHAPE;
  }
}

}  // namespace wa
