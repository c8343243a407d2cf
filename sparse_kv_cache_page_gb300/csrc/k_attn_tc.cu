// Block attention on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Inferix (summary page), §3 Technical Approach, Step 3:
//   O = Attention(Q, [K_cache (+) K_t], [V_cache (+) V_t]) -- the chunk's queries
//   attend, with no mask, to the cached KV (here the contiguous buffer of the
//   retrieved pages) followed by the chunk's own local KV.
// WorldAttention (review page), HKV section: the attention runs over the
// 4 x 8 x 1,560 = 49,920 retrieved tokens held in HBM (tier L1), staged
// through on-chip SRAM (tier L0) FlashAttention-style.
//
// Design (one CTA = one head x two 128-row query tiles, 10 warps):
//   warp 8      TMA producer: Q0/Q1 once, then K_j, V_j alternately into a
//               4-stage ring of 32 KiB slots (two 64-column boxes each,
//               128-byte swizzle, rows past a segment end read as zero).
//   warp 9      TMEM owner (alloc 512 columns) and MMA issuer (one thread):
//               S_i = Q_i K_j^T into TMEM (M=128, N=128, K=128, both operands
//               K-major from shared memory), then O_i += P_i V_j with P_i read
//               from TMEM (bf16, aliasing S_i) and V_j MN-major from shared
//               memory.  S_i(j+1) is issued only after O_i += P_i(j) V_j has
//               completed, because P_i lives in S_i's columns.
//   warps 0-3   softmax of query tile 0 (one thread per row = TMEM lane);
//   warps 4-7   softmax of query tile 1.  Each row keeps a running max m and
//               sum l; exponentials are taken against m, and O_i and l are
//               rescaled only when a tile raises the max by more than 2^8
//               (in exp2 units), so most tiles skip the O round trip.
//   TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
//   Epilogue: O / l rounded to bf16 (optionally fused with an existing
//   output: o = w_old[h] * o + w_new[h] * O) and LSE = scale*m + ln l.
#include <math.h>
#include <string.h>

#include "tc_ptx.cuh"
#include "wa_internal.cuh"

namespace wa {
namespace {

using namespace ptx;

constexpr int BM = 128;                  // query rows per tile
constexpr int BN = 128;                  // keys per tile
constexpr int HD = 128;                  // head dim
constexpr int NS = 4;                    // ring slots
constexpr int kHalfBytes = BN * 64 * 2;  // one 64-column box: 16 KiB
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

__device__ __forceinline__ uint32_t col_s(int i) { return 128u * i; }          // S_i / P_i
__device__ __forceinline__ uint32_t col_o(int i) { return 256u + 128u * i; }   // O_i

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);   // A, B K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);   // A (TMEM) K-major, B MN-major

struct SmemLayout {
  // all offsets from a 1024-byte aligned base
  static constexpr int q = 0;                          // 2 tiles x 32 KiB
  static constexpr int ring = 2 * kTileBytes;          // NS x 32 KiB
  static constexpr int bars = ring + NS * kTileBytes;  // mbarriers
  static constexpr int total = bars + 256;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[NS];
  uint64_t kv_empty[NS];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_ready[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block too large");

struct Params {
  int n_q, n_heads, n_main, n_loc, nt_main, nt_loc;
  float scale, scale_log2;
  void* o;
  float* lse;
  int accumulate;
  const float* w_old;
  const float* w_new;
  int* status;
};

__device__ __forceinline__ int tile_valid(const Params& p, int j) {
  if (j < p.nt_main) return min(BN, p.n_main - j * BN);
  return min(BN, p.n_loc - (j - p.nt_main) * BN);
}

// Output row store: 128 values of one (query, head), optionally fused with the
// values already there (o = w_old * o + w_new * x).
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&x)[32], bool acc,
                                            float wo) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = x[8 * v + e];
    if (acc) {
      const uint4 old = d[v];
      const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        y[2 * e] += wo * __uint_as_float(ow[e] << 16);
        y[2 * e + 1] += wo * __uint_as_float(ow[e] & 0xffff0000u);
      }
    }
    d[v] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
  }
}
__device__ __forceinline__ void store_row32(float* dst, const float (&x)[32], bool acc, float wo) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    float4 y = make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
    if (acc) {
      const float4 old = d[v];
      y.x += wo * old.x;
      y.y += wo * old.y;
      y.z += wo * old.z;
      y.w += wo * old.w;
    }
    d[v] = y;
  }
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
k_block_attn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_km,
                const __grid_constant__ CUtensorMap tm_vm, const __grid_constant__ CUtensorMap tm_kl,
                const __grid_constant__ CUtensorMap tm_vl, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + SmemLayout::bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y;
  const int q0 = blockIdx.x * (2 * BM);
  const int nkv = p.nt_main + p.nt_loc;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_ready[i], 128);
      mbar_init(&bars->o_ready[i], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      const int xq = head * HD;
      mbar_arrive_expect_tx(&bars->q_full, 2 * kTileBytes);
      for (int i = 0; i < 2; ++i)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(&tm_q, &bars->q_full, smem + SmemLayout::q + i * kTileBytes + hf * kHalfBytes,
                      xq + hf * 64, q0 + i * BM);
      int issued = 0;
      for (int t = 0; t < 2 * nkv; ++t) {
        const int slot = t % NS;
        if (t >= NS && !mbar_wait(&bars->kv_empty[slot], ((t / NS) - 1) & 1, abort_flag, p.status))
          break;
        const int j = t >> 1;
        const bool is_v = t & 1;
        const CUtensorMap* map;
        int row;
        if (j < p.nt_main) {
          map = is_v ? &tm_vm : &tm_km;
          row = j * BN;
        } else {
          map = is_v ? &tm_vl : &tm_kl;
          row = (j - p.nt_main) * BN;
        }
        uint8_t* dst = smem + SmemLayout::ring + slot * kTileBytes;
        mbar_arrive_expect_tx(&bars->kv_full[slot], kTileBytes);
        tma_load_2d(map, &bars->kv_full[slot], dst, xq, row);
        tma_load_2d(map, &bars->kv_full[slot], dst + kHalfBytes, xq + 64, row);
        issued = t + 1;
      }
      if (*abort_flag) {
        // drain: wait (bounded) for the copies still in flight
        for (int t = issued - NS < 0 ? 0 : issued - NS; t < issued; ++t)
          mbar_wait_drain(&bars->kv_full[t % NS], (t / NS) & 1, 100000000ull);
        mbar_wait_drain(&bars->q_full, 0, 100000000ull);
      }
    }
    __syncwarp();   // lanes 1-31 wait here for lane 0: the warp reaches the CTA barrier converged
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t q_base = smem_u32(smem + SmemLayout::q);
      const uint32_t ring_base = smem_u32(smem + SmemLayout::ring);
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.status);
      tc_fence_after();
      for (int j = 0; ok && j < nkv; ++j) {
        const int tk = 2 * j, tv = 2 * j + 1;
        const int sk = tk % NS, sv = tv % NS;
        if (!(ok = mbar_wait(&bars->kv_full[sk], (tk / NS) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        const uint32_t kb = ring_base + sk * kTileBytes;
        for (int i = 0; i < 2; ++i) {
          if (j > 0) {
            if (!(ok = mbar_wait(&bars->o_ready[i], (j - 1) & 1, abort_flag, p.status))) break;
            tc_fence_after();
          }
          const uint32_t qb = q_base + i * kTileBytes;
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks) {
            const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
            mma_ss(tmem + col_s(i), sdesc(qb + off, 16, 1024, kSwizzle128B),
                   sdesc(kb + off, 16, 1024, kSwizzle128B), kIdescQK, ks > 0);
          }
          mma_commit(&bars->s_full[i]);
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[sk]);
        if (!(ok = mbar_wait(&bars->kv_full[sv], (tv / NS) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        const uint32_t vb = ring_base + sv * kTileBytes;
        for (int i = 0; i < 2; ++i) {
          if (!(ok = mbar_wait(&bars->p_ready[i], j & 1, abort_flag, p.status))) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            // B = V_j rows [16ks, 16ks+16): MN-major, 64-column boxes 16 KiB apart
            // (leading byte offset), 8-row groups 1 KiB apart (stride byte offset)
            mma_ts(tmem + col_o(i), tmem + col_s(i) + ks * 8,
                   sdesc(vb + ks * 16 * 128, kHalfBytes, 1024, kSwizzle128B), kIdescPV,
                   (j > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(&bars->o_ready[i]);
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[sv]);
      }
      // all issued MMAs complete before teardown
      mma_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else {
    // softmax warpgroups
    const int qt = warp >> 2;                       // query tile 0 or 1
    const int row = 32 * (warp & 3) + lane;         // TMEM lane = row of the tile
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t s_addr = lane_addr + col_s(qt);
    const uint32_t o_addr = lane_addr + col_o(qt);
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // Every tcgen05.ld/st below is .sync.aligned: all 32 lanes of the warp must
    // execute it together, so branch conditions around them are warp-uniform.
    for (int j = 0; j < nkv; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[qt], j & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + 32 * c, sr[c]);
      tmem_ld_wait();
      const int valid = tile_valid(p, j);   // warp-uniform
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= valid) sr[c][e] = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mx[c] = __uint_as_float(sr[c][0]);
#pragma unroll
        for (int e = 1; e < 31; e += 2)
          mx[c] = fmax3(mx[c], __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
        mx[c] = fmaxf(mx[c], __uint_as_float(sr[c][31]));
      }
      const float tmax = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
      // rows whose max rose by more than 2^8 (exp2 units) rescale O and l
      const bool need = j > 0 && (tmax - m) * sl2 > 8.0f;
      if (j == 0) m = tmax;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? ex2((m - tmax) * sl2) : 1.0f;
        if (need) {
          m = tmax;
          l *= f;
        }
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t orow[32];
          tmem_ld32(o_addr + 32 * c, orow);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * f);
          tmem_st32(o_addr + 32 * c, orow);
        }
      }
      // p = 2^(s*sl2 - m*sl2) rounded to bf16 for the P V product; the row sum
      // adds the same rounded values, so numerator and denominator agree.
      const float nmsl2 = -m * sl2;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[32];   // bf16 pairs for keys 64*hf .. 64*hf+63
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int c = 2 * hf + c2;
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]), sl2, sl2,
                  nmsl2, nmsl2);
            const uint32_t w = pack_bf16x2(ex2(x0), ex2(x1));
            pk[16 * c2 + (e >> 1)] = w;
            fadd2_acc(rs0, rs1, __uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
          }
        tmem_st32(s_addr + 32 * hf, pk);
      }
      l += rs0 + rs1;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[qt]);
    }
    if (ok)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&bars->o_ready[qt], (nkv - 1) & 1, abort_flag, p.status));
    tc_fence_after();
    const int grow = q0 + qt * BM + row;
    const bool store = grow < p.n_q;
    if (ok) {
      const float inv_l = 1.0f / l;
      OutT* orow_g = static_cast<OutT*>(p.o) + ((size_t)(store ? grow : 0) * p.n_heads + head) * HD;
      const float wo = p.accumulate ? (p.w_old ? p.w_old[head] : 1.0f) : 0.0f;
      const float wn = (p.accumulate ? (p.w_new ? p.w_new[head] : 1.0f) : 1.0f) * inv_l;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t orow[32];
        tmem_ld32(o_addr + 32 * c, orow);   // whole warp
        tmem_ld_wait();
        if (store) {
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(orow[e]) * wn;
          store_row32(orow_g + 32 * c, x, p.accumulate != 0, wo);
        }
      }
      if (store && p.lse) p.lse[(size_t)head * p.n_q + grow] = m * p.scale + logf(l);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

wa_status launch_attn_tc(const void* q, int n_q, const void* k_main, const void* v_main,
                         int n_main, const void* k_loc, const void* v_loc, int n_loc, int n_heads,
                         float scale, void* o, int o_f32, float* lse, int accumulate,
                         const float* w_old, const float* w_new, cudaStream_t s) {
  Ctrl* ctrl = nullptr;
  wa_status rc = get_ctrl(&ctrl);
  if (rc != WA_OK) return rc;
  const uint64_t cols = (uint64_t)n_heads * HD;
  CUtensorMap tq, tkm, tvm, tkl, tvl;
  memset(&tkm, 0, sizeof(tkm));
  memset(&tvm, 0, sizeof(tvm));
  memset(&tkl, 0, sizeof(tkl));
  memset(&tvl, 0, sizeof(tvl));
  if ((rc = make_tmap_2d_bf16(&tq, q, cols, n_q, cols, 64, BM)) != WA_OK) return rc;
  if (n_main > 0) {
    if ((rc = make_tmap_2d_bf16(&tkm, k_main, cols, n_main, cols, 64, BN)) != WA_OK) return rc;
    if ((rc = make_tmap_2d_bf16(&tvm, v_main, cols, n_main, cols, 64, BN)) != WA_OK) return rc;
  }
  if (n_loc > 0) {
    if ((rc = make_tmap_2d_bf16(&tkl, k_loc, cols, n_loc, cols, 64, BN)) != WA_OK) return rc;
    if ((rc = make_tmap_2d_bf16(&tvl, v_loc, cols, n_loc, cols, 64, BN)) != WA_OK) return rc;
  }
  Params p;
  p.n_q = n_q;
  p.n_heads = n_heads;
  p.n_main = n_main;
  p.n_loc = n_loc;
  p.nt_main = (n_main + BN - 1) / BN;
  p.nt_loc = (n_loc + BN - 1) / BN;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.accumulate = accumulate;
  p.w_old = w_old;
  p.w_new = w_new;
  p.status = &ctrl->status;
  const int smem = SmemLayout::total + 1024;
  static bool attr_done[64][2] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = o_f32 ? k_block_attn_tc<float> : k_block_attn_tc<__nv_bfloat16>;
  if (dev < 64 && !attr_done[dev][o_f32 ? 1 : 0]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return WA_ERR_CUDA;
    attr_done[dev][o_f32 ? 1 : 0] = true;
  }
  dim3 grid((n_q + 2 * BM - 1) / (2 * BM), n_heads);
  kern<<<grid, kThreads, smem, s>>>(tq, tkm, tvm, tkl, tvl, p);
  return cuda_status(cudaPeekAtLastError());
}

}  // namespace wa
