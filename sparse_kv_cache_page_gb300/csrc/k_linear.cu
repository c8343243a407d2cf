// Linformer-style low-rank branch.
//
// WorldAttention (review page), HSA section (paper §3.2 HSA, Appx. Linear
// Branch): for each head h, learned E_K^(h), E_V^(h) in R^{L x r} compress the
// L retrieved + local keys and values to r rows, cutting the cost from
// O(L^2 d_k) to O(L r d_k); the two branches are then fused by a per-head
// gate.  The page leaves the projection equation out; it is read as Linformer:
//   K'_h = E_K^(h)T [K_buf ; K_loc]_h,  V'_h = E_V^(h)T [V_buf ; V_loc]_h   (r x d)
//   O_lin = softmax(Q_h K'_h^T / sqrt(d)) V'_h,   o = w_attn[h] o + w_lin[h] O_lin.
//
// K7 (k_linformer_proj): one CTA per (head, K or V, key-range split).  A TMA
// ring streams E tiles (64 keys x rank, MN-major A operand) and the matching
// K or V tiles (64 keys x 128, MN-major B operand); one thread issues
// tcgen05 MMAs (M = 128 per rank block, N = 128, K = 16) accumulating rank/128
// fp32 tiles in TMEM; the epilogue writes the CTA's partial sums.  The step
// reads E (L x r per head and tensor) and K, V once: it is HBM-bound.
// K7b (k_linformer_reduce): sums the split partials in a fixed order and rounds
// K', V' to bf16, token-major [r][H][128], the layout the attention reads.
// K8: the tensor-core attention kernel over the r projected keys, with its
// fused epilogue o = w_attn o + w_lin O_lin.
#include <atomic>
#include <math.h>
#include <string.h>

#include "tc_ptx.cuh"
#include "wa_internal.cuh"

namespace wa {
namespace {

using namespace ptx;

constexpr int LT = 64;                     // keys per tile
constexpr int HD = 128;
constexpr int kThreads = 128;              // 4 warps: producer, MMA, all four in the epilogue
constexpr int kEBox = LT * 64 * 2;         // one E box: 64 keys x 64 rank columns = 8 KiB
constexpr int kXBox = LT * 64 * 2;         // one K/V box: 64 keys x 64 features = 8 KiB

template <int RB>   // rank blocks of 128
struct LinCfg {
  static constexpr int rank = 128 * RB;
  static constexpr int e_bytes = (rank / 64) * kEBox;     // E tile
  static constexpr int x_bytes = 2 * kXBox;               // K or V tile
  static constexpr int stage = e_bytes + x_bytes;
  static constexpr int ns = (200 * 1024) / stage > 4 ? 4 : (200 * 1024) / stage;
  static constexpr int bars = ns * stage;
  static constexpr int total = bars + 128;
  static constexpr uint32_t tmem_cols = rank <= 128 ? 128 : (rank <= 256 ? 256 : 512);  // power of 2
};

struct LinParams {
  int n_main, n_loc, nt_main, nt_loc, n_split, n_heads, L;
  float* partial;   // [split][tensor][head][rank][128]
  int* status;
  unsigned long long wait_ns;   // limit of each bounded wait (host-set)
};

template <int RB>
__global__ void __launch_bounds__(kThreads, 1)
k_linformer_proj(const __grid_constant__ CUtensorMap tm_ek, const __grid_constant__ CUtensorMap tm_ev,
                 const __grid_constant__ CUtensorMap tm_km, const __grid_constant__ CUtensorMap tm_vm,
                 const __grid_constant__ CUtensorMap tm_kl, const __grid_constant__ CUtensorMap tm_vl,
                 const LinParams p) {
  using C = LinCfg<RB>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  struct Bars {
    uint64_t full[C::ns];
    uint64_t empty[C::ns];
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
  };
  static_assert(sizeof(Bars) <= 128, "barrier block");
  Bars* bars = reinterpret_cast<Bars*>(smem + C::bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int tensor = blockIdx.y / p.n_heads;      // 0 = keys, 1 = values
  const int head = blockIdx.y % p.n_heads;
  const int nt = p.nt_main + p.nt_loc;
  const int t0 = (int)(((long long)nt * split) / p.n_split);
  const int t1 = (int)(((long long)nt * (split + 1)) / p.n_split);
  const int ntl = t1 - t0;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::ns; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const CUtensorMap* tm_e = tensor ? &tm_ev : &tm_ek;

  if (warp == 0) {
    if (lane == 0 && ntl > 0) {
      int issued = 0;
      for (int t = 0; t < ntl; ++t) {
        const int slot = t % C::ns;
        if (t >= C::ns &&
            !mbar_wait(&bars->empty[slot], ((t / C::ns) - 1) & 1, abort_flag, p.status, p.wait_ns))
          break;
        const int g = t0 + t;
        const CUtensorMap* tm_x;
        int xrow, erow;
        if (g < p.nt_main) {
          tm_x = tensor ? &tm_vm : &tm_km;
          xrow = g * LT;
          erow = xrow;
        } else {
          tm_x = tensor ? &tm_vl : &tm_kl;
          xrow = (g - p.nt_main) * LT;
          erow = p.n_main + xrow;
        }
        uint8_t* st = smem + slot * C::stage;
        mbar_arrive_expect_tx(&bars->full[slot], C::stage);
        // E rows past the end of a segment are multiplied by zero K/V rows (the
        // K/V map reads rows past its segment as 0), so they need no masking.
        for (int b = 0; b < C::rank / 64; ++b)
          tma_load_3d(tm_e, &bars->full[slot], st + b * kEBox, b * 64, erow, head);
        for (int b = 0; b < 2; ++b)
          tma_load_2d(tm_x, &bars->full[slot], st + C::e_bytes + b * kXBox, head * HD + b * 64,
                      xrow);
        issued = t + 1;
      }
      if (*abort_flag) {
        for (int t = issued - C::ns < 0 ? 0 : issued - C::ns; t < issued; ++t)
          mbar_wait_drain(&bars->full[t % C::ns], (t / C::ns) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 1, 1);   // A and B MN-major
      const uint32_t base = smem_u32(smem);
      bool ok = true;
      for (int t = 0; ok && t < ntl; ++t) {
        const int slot = t % C::ns;
        if (!(ok = mbar_wait(&bars->full[slot], (t / C::ns) & 1, abort_flag, p.status, p.wait_ns))) break;
        tc_fence_after();
        const uint32_t st = base + slot * C::stage;
#pragma unroll
        for (int m = 0; m < RB; ++m)
#pragma unroll
          for (int ks = 0; ks < LT / 16; ++ks) {
            // A: rank rows 128m..128m+127 = E boxes 2m, 2m+1 (8 KiB apart);
            // B: the K/V tile's two 64-feature boxes; both advance 16 keys = 2 KiB
            const uint64_t da = sdesc(st + 2 * m * kEBox + ks * 2048, kEBox, 1024, kSwizzle128B);
            const uint64_t db = sdesc(st + C::e_bytes + ks * 2048, kXBox, 1024, kSwizzle128B);
            mma_ss(tmem + 128 * m, da, db, idesc, (t > 0 || ks > 0) ? 1u : 0u);
          }
        mma_commit(&bars->empty[slot]);
      }
      mma_commit(&bars->done);
      mbar_wait_drain(&bars->done, 0, 1000000000ull);
    }
    __syncwarp();
  }
  // epilogue (all four warps): TMEM lane = rank row within a block
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->done, 0, abort_flag, p.status, p.wait_ns));
  tc_fence_after();
  if (ok) {
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    for (int m = 0; m < RB; ++m) {
      const int r = 128 * m + 32 * warp + lane;
      float* dst = p.partial +
                   ((((size_t)split * 2 + tensor) * p.n_heads + head) * C::rank + r) * HD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_addr + 128 * m + 32 * c, v);
        tmem_ld_wait();
        float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float4 x;
          if (ntl > 0)
            x = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                            __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
          else
            x = make_float4(0.f, 0.f, 0.f, 0.f);
          __stcg(d4 + e, x);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, C::tmem_cols);
  }
}

// out[tensor][r][h][e] = bf16( sum_s partial[s][tensor][h][r][e] ), fixed order
__global__ void __launch_bounds__(256)
k_linformer_reduce(const float* __restrict__ partial, int n_split, int n_heads, int rank,
                   __nv_bfloat16* __restrict__ kv_out) {
  const size_t per_split = (size_t)2 * n_heads * rank * HD;
  const size_t n4 = per_split / 4;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 acc = __ldcg(reinterpret_cast<const float4*>(partial) + i);
    for (int s = 1; s < n_split; ++s) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(partial + s * per_split) + i);
      acc.x += t.x;
      acc.y += t.y;
      acc.z += t.z;
      acc.w += t.w;
    }
    const size_t flat = i * 4;                    // [tensor][h][r][e]
    const int e = (int)(flat % HD);
    const size_t rest = flat / HD;
    const int r = (int)(rest % rank);
    const int h = (int)((rest / rank) % n_heads);
    const int tensor = (int)(rest / ((size_t)rank * n_heads));
    __nv_bfloat16* d = kv_out + (((size_t)tensor * rank + r) * n_heads + h) * HD + e;
    const uint32_t lo = pack_bf16x2(acc.x, acc.y), hi = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(d) = make_uint2(lo, hi);
  }
}

template <int RB>
wa_status proj_t(const CUtensorMap* maps, const LinParams& p, int grid_y, cudaStream_t s) {
  using C = LinCfg<RB>;
  const int smem = C::total + 1024;
  static std::atomic<bool> attr_done[64];   // per device; setting it twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k_linformer_proj<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return WA_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  dim3 grid(p.n_split, grid_y);
  k_linformer_proj<RB><<<grid, kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                    maps[5], p);
  return cuda_status(cudaPeekAtLastError());
}

wa_status make_tmap_e(CUtensorMap* map, const void* e, int rank, int L, int n_heads) {
  // E as a 3-D tensor (rank, L, head); box = 64 rank columns x 64 keys x 1 head
  return make_tmap_3d_bf16(map, e, (uint64_t)rank, (uint64_t)L, (uint64_t)n_heads,
                           (uint64_t)rank, (uint64_t)rank * L, 64, LT);
}

}  // namespace

wa_status launch_linear_branch(const void* q, int n_q, const void* k_main, const void* v_main,
                               int n_main, const void* k_loc, const void* v_loc, int n_loc,
                               const void* e_k, const void* e_v, int rank, int n_heads,
                               float scale, const float* w_attn, const float* w_lin,
                               int accumulate, void* o, int o_f32, cudaStream_t s) {
  const int L = n_main + n_loc;
  const uint64_t cols = (uint64_t)n_heads * HD;
  CUtensorMap maps[6];
  memset(maps, 0, sizeof(maps));
  wa_status rc;
  if ((rc = make_tmap_e(&maps[0], e_k, rank, L, n_heads)) != WA_OK) return rc;
  if ((rc = make_tmap_e(&maps[1], e_v, rank, L, n_heads)) != WA_OK) return rc;
  if (n_main > 0) {
    if ((rc = make_tmap_2d_bf16(&maps[2], k_main, cols, n_main, cols, 64, LT)) != WA_OK) return rc;
    if ((rc = make_tmap_2d_bf16(&maps[3], v_main, cols, n_main, cols, 64, LT)) != WA_OK) return rc;
  }
  if (n_loc > 0) {
    if ((rc = make_tmap_2d_bf16(&maps[4], k_loc, cols, n_loc, cols, 64, LT)) != WA_OK) return rc;
    if ((rc = make_tmap_2d_bf16(&maps[5], v_loc, cols, n_loc, cols, 64, LT)) != WA_OK) return rc;
  }
  LinParams p;
  p.n_main = n_main;
  p.n_loc = n_loc;
  p.nt_main = (n_main + LT - 1) / LT;
  p.nt_loc = (n_loc + LT - 1) / LT;
  p.n_heads = n_heads;
  p.L = L;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one wave: (2 tensors x heads x splits) CTAs on at most the SM count
  int n_split = sms / (2 * n_heads);
  if (n_split < 1) n_split = 1;
  const int nt = p.nt_main + p.nt_loc;
  if (n_split > nt) n_split = nt;
  p.n_split = n_split;
  // scratch: partials, then K'|V' in bf16 (token-major [r][H][128] each)
  const size_t part_bytes = (size_t)n_split * 2 * n_heads * rank * HD * sizeof(float);
  const size_t kv_bytes = (size_t)2 * rank * n_heads * HD * sizeof(__nv_bfloat16);
  Scratch sc;
  if ((rc = get_scratch(part_bytes + kv_bytes, &sc)) != WA_OK) return rc;
  p.partial = static_cast<float*>(sc.data);
  p.status = &sc.ctrl->status;
  p.wait_ns = wait_limit_ns();
  __nv_bfloat16* kv = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(sc.data) + part_bytes);
  const int gy = 2 * n_heads;
  switch (rank / 128) {
    case 1: rc = proj_t<1>(maps, p, gy, s); break;
    case 2: rc = proj_t<2>(maps, p, gy, s); break;
    case 3: rc = proj_t<3>(maps, p, gy, s); break;
    case 4: rc = proj_t<4>(maps, p, gy, s); break;
    default: return WA_ERR_SHAPE;
  }
  if (rc != WA_OK) return rc;
  const size_t n4 = (size_t)2 * n_heads * rank * HD / 4;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > sms * 8) blocks = sms * 8;
  k_linformer_reduce<<<blocks, 256, 0, s>>>(p.partial, n_split, n_heads, rank, kv);
  if ((rc = cuda_status(cudaPeekAtLastError())) != WA_OK) return rc;
  const __nv_bfloat16* kp = kv;
  const __nv_bfloat16* vp = kv + (size_t)rank * n_heads * HD;
  // K8: low-rank attention over the rank projected keys, fused into o
  return launch_attn_tc(q, n_q, kp, vp, rank, nullptr, nullptr, 0, n_heads, scale, o, o_f32,
                        nullptr, accumulate, w_attn, w_lin, /*max_split=*/1, s);
}

}  // namespace wa
