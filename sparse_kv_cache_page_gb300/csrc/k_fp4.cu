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
// A lane per 16-value block (d / 16 lanes per row), two row groups in flight
// per warp.  The gather-decode reads codes and scales
// where they live (device memory or pinned host memory through its device
// mapping) and writes the bf16 attention buffer.
#include <cuda_fp16.h>

#include "codec_math.cuh"
#include "wa_internal.cuh"

namespace wa {
namespace {

using namespace codec;

constexpr int kThreads = 256;

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

// Each lane owns one 16-value block of a row (LPR = d / 16 lanes per row, 32 /
// LPR rows per warp step): a 32-byte load, its block maximum in registers, the
// row maximum over the row's lanes, 8 bytes of codes and its block scale.
// kSteps row groups are in flight per warp.
constexpr int kSteps = 2;
constexpr int kDecSteps = 4;   // decoding: more row groups in flight (reads are small)

template <int LPR>
__global__ void __launch_bounds__(kThreads)
k_nvfp4_encode(const __nv_bfloat16* __restrict__ src, size_t n_rows, uint8_t* __restrict__ codes,
               uint8_t* __restrict__ bscales, float* __restrict__ rscales) {
  constexpr int RPW = 32 / LPR;
  constexpr int D = 16 * LPR;
  const int lane = threadIdx.x & 31, sub = lane / LPR, b = lane % LPR;
  const size_t warps = (size_t)gridDim.x * (kThreads / 32);
  const float r2688 = __frcp_rn(2688.0f);
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
      const float bmax = absmax16_bf16(w);
      float amax = bmax;
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (!live) continue;
      const float g = dividend_ok(amax) ? div_rn(amax, 2688.0f, r2688) : __fdiv_rn(amax, 2688.0f);
      const float den = __fmul_rn(g, 6.0f);
      const uint32_t sb = den > 0.f ? enc_e4m3(__fdiv_rn(bmax, den)) : 0u;
      const float es = __fmul_rn(dec_e4m3(sb), g);
      uint32_t c[8];
      if (div_fast_ok(es)) {
        const uint64_t nb2 = dup2(-es), r2 = dup2(__frcp_rn(es));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float q0, q1;
          div2_rn(q0, q1, bf16_lo(w[i]), bf16_hi(w[i]), nb2, r2);
          c[i] = enc_e2m1x2(q0, q1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          c[i] = es > 0.f ? enc_e2m1x2(__fdiv_rn(bf16_lo(w[i]), es), __fdiv_rn(bf16_hi(w[i]), es))
                          : 0u;
      }
      // code bytes 0-3 and 4-7 into two words (byte i = pair i)
      uint32_t out[2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
        out[h] = __byte_perm(__byte_perm(c[4 * h], c[4 * h + 1], 0x0040),
                             __byte_perm(c[4 * h + 2], c[4 * h + 3], 0x0040), 0x5410);
      *reinterpret_cast<uint2*>(codes + r * (D / 2) + 8 * b) = make_uint2(out[0], out[1]);
      bscales[r * LPR + b] = (uint8_t)sb;
      if (b == 0) rscales[r] = g;
    }
  }
}

// out[s*P + t][h] = decode(pages[idx[s]][t][h]); idx NULL: out row r = row r.
template <int LPR>
__global__ void __launch_bounds__(kThreads)
k_nvfp4_decode(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ bscales,
               const float* __restrict__ rscales, const int32_t* __restrict__ idx, int n_pages,
               size_t page_rows, size_t n_rows, __nv_bfloat16* __restrict__ out, Ctrl* ctrl) {
  constexpr int RPW = 32 / LPR;
  constexpr int D = 16 * LPR;
  const int lane = threadIdx.x & 31, sub = lane / LPR, b = lane % LPR;
  const size_t warps = (size_t)gridDim.x * (kThreads / 32);
  for (size_t g0 = ((size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * RPW * kDecSteps;
       g0 < n_rows; g0 += warps * RPW * kDecSteps) {
    uint2 c[kDecSteps];
    uint32_t sb[kDecSteps];
    float g[kDecSteps];
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
        c[k] = *reinterpret_cast<const uint2*>(codes + src_row * (D / 2) + 8 * b);
        sb[k] = bscales[src_row * LPR + b];
        g[k] = rscales[src_row];
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
        const float es = __fmul_rn(dec_e4m3(sb[k]), g[k]);
        const uint32_t cw[2] = {c[k].x, c[k].y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 v = dec_e2m1x2((cw[i >> 2] >> (8 * (i & 3))) & 0xFFu);
          float lo, hi;
          fmul2(lo, hi, v.x, v.y, es, es);
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
// the resident block count (as the FP8 encoder, where it measured faster); the
// decoder, whose traffic is mostly writes, 8 blocks per SM, more than fit at
// once, so that blocks that start late fill the SMs that finish early (0.079
// against 0.084 ms with the resident count, 8 pages).
inline unsigned grid_for(size_t rows, int head_dim, int steps, size_t cap) {
  const size_t per_block = (size_t)(kThreads / 32) * (512 / head_dim) * steps;
  const size_t need = (rows + per_block - 1) / per_block;
  return (unsigned)(need < cap ? need : cap);
}

}  // namespace

wa_status launch_nvfp4_encode(const void* src, size_t n_rows, int head_dim, void* codes,
                              void* bscales, float* rscales, cudaStream_t s) {
  const auto* x = static_cast<const __nv_bfloat16*>(src);
  auto* c = static_cast<uint8_t*>(codes);
  auto* b = static_cast<uint8_t*>(bscales);
  auto run = [&](auto kernel) {
    if (n_rows == 0) return WA_OK;
    kernel<<<grid_for(n_rows, head_dim, kSteps, resident_blocks(kernel, kThreads)), kThreads, 0,
             s>>>(x, n_rows, c, b,
                                                                           rscales);
    return cuda_status(cudaPeekAtLastError());
  };
  switch (head_dim / 16) {
    case 4: return run(k_nvfp4_encode<4>);
    case 8: return run(k_nvfp4_encode<8>);
    case 16: return run(k_nvfp4_encode<16>);
    default: return WA_ERR_SHAPE;
  }
}

wa_status launch_nvfp4_decode(const void* codes, const void* bscales, const float* rscales,
                              const int32_t* idx, int n_pages, size_t page_rows, size_t n_rows,
                              int head_dim, void* out, cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const auto* c = static_cast<const uint8_t*>(codes);
  const auto* b = static_cast<const uint8_t*>(bscales);
  auto* o = static_cast<__nv_bfloat16*>(out);
  auto run = [&](auto kernel) {
    if (n_rows == 0) return WA_OK;
    kernel<<<grid_for(n_rows, head_dim, kDecSteps, (size_t)sm_count() * 8), kThreads, 0, s>>>(
        c, b, rscales, idx, n_pages, page_rows, n_rows, o, ctrl);
    return cuda_status(cudaPeekAtLastError());
  };
  switch (head_dim / 16) {
    case 4: return run(k_nvfp4_decode<4>);
    case 8: return run(k_nvfp4_decode<8>);
    case 16: return run(k_nvfp4_decode<16>);
    default: return WA_ERR_SHAPE;
  }
}

}  // namespace wa
