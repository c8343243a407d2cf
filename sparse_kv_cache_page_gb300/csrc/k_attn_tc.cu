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
// Design (one CTA = one head x two 128-row query tiles x one range of 128-key
// tiles; 12 warps in three warpgroups):
//   warp 8      TMA producer: Q0/Q1 once, then K_j, V_j alternately into a
//               5-slot ring of 32 KiB (two 64-column boxes of 128 rows each,
//               128-byte swizzle, rows past a segment end read as zero).
//   warp 9      S issuer (one thread; also owns the 512 TMEM columns):
//               S_0(j) = Q_0 K_j^T, then S_1(j) = Q_1 K_j^T, into the same
//               128 TMEM columns (M=128, N=128, K=128, both operands K-major
//               from shared memory), each as soon as the other tile's softmax
//               has read the previous S out of those columns.
//   warp 10     P V issuer (one thread, both tiles): O_i += P_i(j) V_j with
//               P_i read from TMEM (bf16) and V_j MN-major from shared memory
//               (M=128, N=128, K=128), as soon as P_i(j) is published.
//   warps 0-3   softmax of query tile 0 (one thread per row = TMEM lane);
//   warps 4-7   softmax of query tile 1.  Each row keeps a running max m and
//               a sum l of the bf16-rounded p (the values the P V product
//               uses); exponentials are taken against m, and O_i and l are
//               rescaled only when a tile raises the max by more than 2^8
//               (in exp2 units), so most tiles skip the O round trip.
//   TMEM columns: S [0,128) (shared by the two tiles in turn), P_0 [128,192),
//   P_1 [192,256), O_0 [256,384), O_1 [384,512).  N=128 key tiles halve the
//   shared-memory reads of Q per key against 64-key tiles: an N=64 S MMA
//   (4 KiB of Q + 2 KiB of K per 32 tensor cycles) outruns the 128 bytes per
//   cycle that shared memory delivers, an N=128 one (8 KiB per 64) does not.
//   Key tiles are split into n_split contiguous ranges so that the grid fills
//   whole waves of the 152 SMs; each CTA of a split stores its unnormalised
//   O, m and l to scratch, and the CTA that finishes last for its (head,
//   query pair) combines them (no spin-wait: a ticket counter).
//   Epilogue: O / l (fp32 or rounded to bf16; optionally fused with an
//   existing output: o = w_old[h] * o + w_new[h] * O) and LSE = scale*m + ln l.
//
// Paged form (the gather fused into the producer): the buffer segment is not
// read from a contiguous buffer but from the page bank, buffer row r being row
// r % P of page idx[r / P] (P = page_tokens, a multiple of 8).  A tile inside
// one page comes as 128-row boxes, a tile across a page boundary (or past the
// buffer's end) as 64-row boxes when P is a multiple of 64, else 8-row boxes,
// each box inside one page (64-row boxes throughout measured 13% slower).  The ring
// receives the same bytes as from the gathered buffer, so the results are
// bit-identical to gather then attention.  With a buffer given, the CTA of
// query pair j % n_qpairs also writes buffer tile j (K and V) from its ring
// slot by TMA store -- the gather's output, without the gather's second read
// of the pages: warp 11 issues each store as soon as the tile lands, and a
// slot is reused once its MMA and any store have read it.
#include <atomic>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "tc_ptx.cuh"
#include "wa_internal.cuh"

namespace wa {
namespace {

using namespace ptx;

constexpr int BM = 128;                  // query rows per tile
constexpr int BN = 128;                  // keys per tile
constexpr int HD = 128;                  // head dim
constexpr int NS = 5;                    // ring slots (K and V tiles alternate)
constexpr int kQHalf = BM * 64 * 2;      // Q box: 128 rows x 64 columns = 16 KiB
constexpr int kQTile = 2 * kQHalf;
constexpr int kKvHalf = BN * 64 * 2;     // K/V box: 128 rows x 64 columns = 16 KiB
constexpr int kKvTile = 2 * kKvHalf;
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;              // S issuer of both query tiles, TMEM owner
constexpr int kPvWarp = 10;              // P V issuer of both query tiles
constexpr int kStoreWarp = 11;           // paged form: buffer stores
constexpr int kMaxUnits = 8192;          // split attention: one ticket per (head, query pair)

constexpr uint32_t kColS = 0;            // S, shared by the two query tiles in turn
__device__ __forceinline__ uint32_t col_p(int i) { return 128u + 64u * i; }   // P_i (bf16 pairs)
__device__ __forceinline__ uint32_t col_o(int i) { return 256u + 128u * i; }  // O_i

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, BN, 0, 0);    // A, B K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);   // A (TMEM) K-major, B MN-major

struct SmemLayout {
  // all offsets from a 1024-byte aligned base
  static constexpr int q = 0;                          // 2 tiles x 32 KiB
  static constexpr int ring = 2 * kQTile;              // NS x 16 KiB
  static constexpr int bars = ring + NS * kKvTile;     // mbarriers
  static constexpr int total = bars + 512;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[NS];
  uint64_t kv_empty[NS];
  uint64_t s_full[2];       // S_i(j) computed (in the shared S columns)
  uint64_t s_free[2];       // softmax i has read S_i(j)
  uint64_t p_ready[2];      // P_i(j) written
  uint64_t o_ready[2];      // O_i += P_i(j) V_j done
  uint64_t drain;
  uint64_t comb;            // bulk copy of another split's rows (split combine)
  uint64_t st_done;         // paged form: every buffer store has read the ring
  uint32_t tmem_base;
  int abort_flag;
  unsigned ticket;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");
static_assert(SmemLayout::total + 1024 <= 232448, "shared memory per CTA");

struct Params {
  int n_q, n_heads, n_main, n_loc, nt_main, nt_loc;
  int n_split, n_qpairs;
  float scale, scale_log2;
  void* o;
  float* lse;
  int accumulate;
  const float* w_old;
  const float* w_new;
  int* status;
  float* part_o;             // [unit][split][256][128] unnormalised O (split > 1)
  float4* part_ml;           // [unit][split][256] (m, l, l_exact, -)
  unsigned* counters;        // [unit] tickets, zero between launches
  // block-sparse form: head h attends to key tiles tiles[h][0 .. tile_count[h]),
  // each {segment << 30 | first row, rows (<= 128)}; dense form: 128-key tiles
  // over [main ; local]
  const int2* tiles;
  const int32_t* tile_count;
  int tile_stride;
  unsigned long long wait_ns;   // limit of each bounded wait (host-set)
  int withhold_q;               // fault injection: the query tiles are never copied
  // paged form: buffer row r = row r % page_tokens of page idx[idx_stride * head + r / page_tokens]
  // of the bank's bank_rows = n_pages * page_tokens rows
  const int32_t* idx;
  int idx_stride, page_tokens, n_pages, bank_rows;
  int box_rows;                 // rows of the boxes that split a tile across pages: 64 or 8
  int store_buf;                // write each buffer tile to the buffer (one CTA per tile)
};

// Key tile j of head h: segment (0 = buffer, 1 = local), first row, valid rows.
struct TileRef {
  int seg, row, valid;
};
template <bool kSparse>
__device__ __forceinline__ TileRef tile_ref(const Params& p, int head, int j) {
  if (kSparse) {
    const int2 t = __ldg(p.tiles + (size_t)head * p.tile_stride + j);
    return {t.x >> 30, t.x & ((1 << 30) - 1), t.y};
  }
  if (j < p.nt_main) return {0, j * BN, min(BN, p.n_main - j * BN)};
  const int r = (j - p.nt_main) * BN;
  return {1, r, min(BN, p.n_loc - r)};
}

// Paged form: bank row of buffer row r (the first of a 64-row box) for head
// `head`; rows past the buffer and bad page indices give a row past the bank,
// which the copy fills with zeros (a bad index is recorded, as by the gather).
__device__ __forceinline__ int bank_row(const Params& p, int head, int r) {
  if (r >= p.n_main) return p.bank_rows;
  const int slot = r / p.page_tokens;
  const int pg = __ldg(p.idx + (size_t)head * p.idx_stride + slot);
  if (pg < 0 || pg >= p.n_pages) {
    atomicOr(p.status, kStatusIndex);
    return p.bank_rows;
  }
  return pg * p.page_tokens + (r - slot * p.page_tokens);
}

// Paged form: ring tile u of a CTA (K for even u, V for odd) is key tile
// jb + u/2; the CTA writes it to the buffer when it is buffer tile j with
// j % n_qpairs equal to the CTA's query pair (one writer per tile).
__device__ __forceinline__ bool owns_tile(const Params& p, int jb, int qpair, int u) {
  const int j = jb + (u >> 1);
  return p.store_buf && j < p.nt_main && j % p.n_qpairs == qpair;
}

// Key tiles [j0, j1) of split `sp`: contiguous, sizes differ by at most one.
__device__ __forceinline__ void split_range(int nkv, int n_split, int sp, int& j0, int& j1) {
  j0 = (int)(((long long)nkv * sp) / n_split);
  j1 = (int)(((long long)nkv * (sp + 1)) / n_split);
}

__device__ __forceinline__ void softmax_bar() {   // the 256 softmax threads only
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// AND of v over the 256 softmax threads (their barrier, with a reduction).
__device__ __forceinline__ bool softmax_all(bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, 1, 256, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((int)v)
      : "memory");
  return r != 0;
}

// Four consecutive output values of one row as fp32 (exact for bf16).
__device__ __forceinline__ float4 load4(const float* src) {
  return *reinterpret_cast<const float4*>(src);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* src) {
  const uint2 w = *reinterpret_cast<const uint2*>(src);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
// Store four consecutive output values, optionally fused with the old ones
// (o = w_old * o + x); the sum in fp32, then one rounding to the output type.
__device__ __forceinline__ void put4(float* dst, float4 x, bool acc, float4 old, float wo) {
  if (acc) {
    x.x += wo * old.x;
    x.y += wo * old.y;
    x.z += wo * old.z;
    x.w += wo * old.w;
  }
  *reinterpret_cast<float4*>(dst) = x;
}
__device__ __forceinline__ void put4(__nv_bfloat16* dst, float4 x, bool acc, float4 old, float wo) {
  if (acc) {
    x.x += wo * old.x;
    x.y += wo * old.y;
    x.z += wo * old.z;
    x.w += wo * old.w;
  }
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
}

// Split partials are staged row-major in shared memory with this row pitch
// (floats): 528-byte rows put the 32 rows a warp writes at once on distinct
// bank groups.
constexpr int kStagePitch = HD + 4;
constexpr int kMaxSplit = 16;     // ticket and done counts share one 32-bit counter
static_assert(256 * kStagePitch * 4 + 128 * HD * 4 + kMaxSplit * 256 * 4 <= SmemLayout::bars,
              "staging, the combine buffer and the split weights overlay Q and the ring only");

template <typename OutT, bool kLse, bool kSparse, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
k_block_attn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_km,
                const __grid_constant__ CUtensorMap tm_vm, const __grid_constant__ CUtensorMap tm_kl,
                const __grid_constant__ CUtensorMap tm_vl, const __grid_constant__ CUtensorMap tm_kp,
                const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kq,
                const __grid_constant__ CUtensorMap tm_vq, const Params p) {
  static_assert(!(kSparse && kPaged), "one form at a time");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + SmemLayout::bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.y;
  const int qpair = blockIdx.x / p.n_split;
  const int split = blockIdx.x % p.n_split;
  const int q0 = qpair * (2 * BM);
  int jb, je;
  const int nkv = kSparse ? __ldg(p.tile_count + head) : p.nt_main + p.nt_loc;
  split_range(nkv, p.n_split, split, jb, je);
  const int nloc = je - jb;                 // key tiles of this CTA (0 only in the block-sparse form)
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      // (paged form: the MMA's commit and the store warp's arrival)
      mbar_init(&bars->kv_empty[s], kPaged ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 128);
      mbar_init(&bars->p_ready[i], 128);
      mbar_init(&bars->o_ready[i], 1);
    }
    mbar_init(&bars->drain, 2);
    mbar_init(&bars->comb, 1);
    mbar_init(&bars->st_done, 1);
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
  // set-up done (barriers, tensor memory): wait for the previous kernel on the
  // stream before the first global access
  pdl_wait();

  if (warp >= 8) {
    // ---------------- warpgroup 2: producer, S issuer, P V issuer (and, in
    // the paged form, the buffer store warp)
    if (warp == kProducerWarp) {
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        const int xq = head * HD;
        // (with withhold_q the query copy is never issued: every wait on it
        // runs out at the wait limit -- the host-side test of the timeout path)
        if (!p.withhold_q) {
          mbar_arrive_expect_tx(&bars->q_full, 2 * kQTile);
          for (int i = 0; i < 2; ++i)
            for (int hf = 0; hf < 2; ++hf)
              tma_load_2d(&tm_q, &bars->q_full, smem + SmemLayout::q + i * kQTile + hf * kQHalf,
                          xq + hf * 64, q0 + i * BM);
        }
        int issued = 0;
        for (int t = 0; t < 2 * nloc; ++t) {
          const int slot = t % NS;
          const TileRef tr = tile_ref<kSparse>(p, head, jb + (t >> 1));
          const bool is_v = t & 1;
          // paged form: the tile's first bank row, looked up before its slot is
          // free; a tile inside one page is one 128-row box per column half,
          // else boxes of box_rows (64, or 8 when the pages are not whole
          // 64-row boxes), each from its own page (a page boundary, or the
          // buffer's end, between)
          bool whole = true;
          int y0 = 0;
          if (kPaged && tr.seg == 0) {
            const int r0 = tr.row;
            whole = r0 + BN - 1 < p.n_main && r0 / p.page_tokens == (r0 + BN - 1) / p.page_tokens;
            y0 = bank_row(p, head, r0);
          }
          if (t >= NS) {
            if (!mbar_wait_sleep(&bars->kv_empty[slot], ((t / NS) - 1) & 1, abort_flag, p.status, p.wait_ns))
              break;
          }
          uint8_t* dst = smem + SmemLayout::ring + slot * kKvTile;
          mbar_arrive_expect_tx(&bars->kv_full[slot], kKvTile);
          if (kPaged && tr.seg == 0) {
            if (whole) {
              const CUtensorMap* map = is_v ? &tm_vq : &tm_kq;
              tma_load_2d(map, &bars->kv_full[slot], dst, xq, y0);
              tma_load_2d(map, &bars->kv_full[slot], dst + kKvHalf, xq + 64, y0);
            } else {
              const CUtensorMap* map = is_v ? &tm_vp : &tm_kp;
              const int br = p.box_rows;
              for (int b = 0; b < BN / br; ++b) {
                const int y = b == 0 ? y0 : bank_row(p, head, tr.row + b * br);
                tma_load_2d(map, &bars->kv_full[slot], dst + b * br * 128, xq, y);
                tma_load_2d(map, &bars->kv_full[slot], dst + kKvHalf + b * br * 128, xq + 64, y);
              }
            }
          } else {
            const CUtensorMap* map = tr.seg == 0 ? (is_v ? &tm_vm : &tm_km) : (is_v ? &tm_vl : &tm_kl);
            const int row = tr.row;
            tma_load_2d(map, &bars->kv_full[slot], dst, xq, row);
            tma_load_2d(map, &bars->kv_full[slot], dst + kKvHalf, xq + 64, row);
          }
          issued = t + 1;
        }
        if (*abort_flag) {
          // drain: wait (bounded) for the copies still in flight
          for (int t = issued - NS < 0 ? 0 : issued - NS; t < issued; ++t)
            mbar_wait_drain(&bars->kv_full[t % NS], (t / NS) & 1, 100000000ull);
          if (!p.withhold_q) mbar_wait_drain(&bars->q_full, 0, 100000000ull);
        }
      }
      __syncwarp();   // lanes 1-31 wait here for lane 0: the warp reaches the CTA barrier converged
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        // S issuer of both query tiles: S_0(j), then S_1(j), into the same
        // TMEM columns, each once the other tile's softmax has read the last S
        const uint32_t q_base = smem_u32(smem + SmemLayout::q);
        const uint32_t ring_base = smem_u32(smem + SmemLayout::ring);
        bool ok = mbar_wait_sleep(&bars->q_full, 0, abort_flag, p.status, p.wait_ns);
        tc_fence_after();
        for (int jj = 0; ok && jj < nloc; ++jj) {
          const int tk = 2 * jj, sk = tk % NS;
          if (!(ok = mbar_wait_sleep(&bars->kv_full[sk], (tk / NS) & 1, abort_flag, p.status, p.wait_ns))) break;
          const uint32_t kb = ring_base + sk * kKvTile;
          for (int i = 0; i < 2; ++i) {
            // the S columns were last read by softmax 1 (tile jj-1) or softmax 0 (tile jj)
            if (i == 0 && jj > 0 &&
                !(ok = mbar_wait_sleep(&bars->s_free[1], (jj - 1) & 1, abort_flag, p.status, p.wait_ns)))
              break;
            if (i == 1 && !(ok = mbar_wait_sleep(&bars->s_free[0], jj & 1, abort_flag, p.status, p.wait_ns)))
              break;
            tc_fence_after();
            const uint32_t qb = q_base + i * kQTile;
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
              const uint32_t qoff = (ks >> 2) * kQHalf + (ks & 3) * 32;
              const uint32_t koff = (ks >> 2) * kKvHalf + (ks & 3) * 32;
              mma_ss(tmem + kColS, sdesc(qb + qoff, 16, 1024, kSwizzle128B),
                     sdesc(kb + koff, 16, 1024, kSwizzle128B), kIdescQK, ks > 0);
            }
            mma_commit(&bars->s_full[i]);
          }
          if (!ok) break;
          mma_commit(&bars->kv_empty[sk]);
        }
        // all issued MMAs complete before teardown
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, 1000000000ull);
      }
      __syncwarp();
    } else if (warp == kPvWarp) {
      if (lane == 0) {
        // P V issuer of both query tiles
        const uint32_t ring_base = smem_u32(smem + SmemLayout::ring);
        bool ok = true;
        for (int jj = 0; ok && jj < nloc; ++jj) {
          const int tv = 2 * jj + 1, sv = tv % NS;
          if (!(ok = mbar_wait_sleep(&bars->kv_full[sv], (tv / NS) & 1, abort_flag, p.status, p.wait_ns))) break;
          const uint32_t vb = ring_base + sv * kKvTile;
          for (int i = 0; i < 2; ++i) {
            if (!(ok = mbar_wait_sleep(&bars->p_ready[i], jj & 1, abort_flag, p.status, p.wait_ns)))
              break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks) {
              // B = V_j rows [16ks, 16ks+16): MN-major, 64-column boxes 8 KiB apart
              // (leading byte offset), 8-row groups 1 KiB apart (stride byte offset)
              mma_ts(tmem + col_o(i), tmem + col_p(i) + ks * 8,
                     sdesc(vb + ks * 16 * 128, kKvHalf, 1024, kSwizzle128B), kIdescPV,
                     (jj > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(&bars->o_ready[i]);
          }
          if (!ok) break;
          mma_commit(&bars->kv_empty[sv]);
        }
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, 1000000000ull);
      }
      __syncwarp();
    } else if (kPaged && warp == kStoreWarp) {
      if (lane == 0) {
        // every ring tile in order: the ones this CTA writes to the buffer are
        // stored as soon as they land; each slot is released (the second of the
        // two arrivals its reuse waits for) once any store has read it.  Seeing
        // every tile keeps each parity wait within one phase of its barrier.
        const int xq = head * HD;
        for (int u = 0; u < 2 * nloc; ++u) {
          const int slot = u % NS;
          if (!mbar_wait_sleep(&bars->kv_full[slot], (u / NS) & 1, abort_flag, p.status, p.wait_ns))
            break;
          if (owns_tile(p, jb, qpair, u)) {
            const uint8_t* src = smem + SmemLayout::ring + slot * kKvTile;
            const CUtensorMap* map = (u & 1) ? &tm_vm : &tm_km;
            const int row = (jb + (u >> 1)) * BN;
            tma_store_2d(map, src, xq, row);
            tma_store_2d(map, src + kKvHalf, xq + 64, row);
            bulk_commit();
            bulk_wait_read_all();
          }
          mbar_arrive(&bars->kv_empty[slot]);
        }
        bulk_wait_read_all();
        mbar_arrive(&bars->st_done);   // the epilogue may now overlay the ring
        bulk_wait_all();               // the stores' writes, before the CTA exits
      }
      __syncwarp();
    }
  } else {
    // ---------------- warpgroups 0-1: softmax and epilogue
    const int qt = warp >> 2;                       // query tile 0 or 1
    const int row = 32 * (warp & 3) + lane;         // TMEM lane = row of the tile
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t s_addr = lane_addr + kColS;
    const uint32_t o_addr = lane_addr + col_o(qt);
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f, lx = 0.f;   // lx: exact (unrounded) sum, for the LSE
    bool ok = true;
    // Every tcgen05.ld/st below is .sync.aligned: all 32 lanes of the warp must
    // execute it together, so branch conditions around them are warp-uniform.
    for (int jj = 0; jj < nloc; ++jj) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[qt], jj & 1, abort_flag, p.status, p.wait_ns));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + 32 * c, sr[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars->s_free[qt]);            // the other tile's S may now be computed
      const int valid = tile_ref<kSparse>(p, head, jb + jj).valid;   // warp-uniform
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
      // rows whose max rose by more than 2^8 (exp2 units) move to the new max
      const bool need = jj > 0 && (tmax - m) * sl2 > 8.0f;
      const float f = need ? ex2((m - tmax) * sl2) : 1.0f;
      if (jj == 0 || need) m = tmax;
      l *= f;
      if (kLse) lx *= f;
      // p = 2^(s*sl2 - m*sl2) rounded to bf16 for the P V product; the row sum
      // adds the same rounded values, so numerator and denominator agree.
      const float nmsl2 = -m * sl2;
      float rs0 = 0.f, rs1 = 0.f, xs0 = 0.f, xs1 = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]), sl2, sl2,
                nmsl2, nmsl2);
          const float p0 = ex2(x0), p1 = ex2(x1);
          const uint32_t w = pack_bf16x2(p0, p1);
          pk[c >> 1][16 * (c & 1) + (e >> 1)] = w;
          acc_bf16x2(rs0, rs1, w);
          if (kLse) fadd2_acc(xs0, xs1, p0, p1);
        }
      // P_i was last read by O += P(jj-1) V, which must also be done before O
      // is rescaled.  (The wait is at most one phase behind.)
      if (jj >= 1)
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[qt], (jj - 1) & 1, abort_flag,
                                               p.status, p.wait_ns));
      if (!ok) break;
      tc_fence_after();
      tmem_st32(lane_addr + col_p(qt), pk[0]);
      tmem_st32(lane_addr + col_p(qt) + 32, pk[1]);
      if (__any_sync(0xffffffffu, need)) {
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
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[qt]);
      l += rs0 + rs1;
      if (kLse) lx += xs0 + xs1;
    }
    if (ok && nloc > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[qt], (nloc - 1) & 1, abort_flag,
                                             p.status, p.wait_ns));
    tc_fence_after();
    // The staging area below overlays the Q tiles: their copy must have landed
    // (a CTA with no key tiles, block-sparse form, reaches here without having
    // waited for anything).  Every K/V copy was consumed by an MMA the loop
    // waited for.
    // (paged form: and the store warp's buffer stores have read the ring)
    bool staging_ok =
        ok && __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, abort_flag, p.status, p.wait_ns));
    if (kPaged)
      staging_ok = staging_ok &&
                   __all_sync(0xffffffffu, mbar_wait(&bars->st_done, 0, abort_flag, p.status, p.wait_ns));
    const int grow = q0 + qt * BM + row;
    const bool store = grow < p.n_q;
    const float wo = p.accumulate ? (p.w_old ? p.w_old[head] : 1.0f) : 0.0f;
    const float wn0 = p.accumulate ? (p.w_new ? p.w_new[head] : 1.0f) : 1.0f;
    if (p.n_split == 1) {
      // normalised rows staged in shared memory (over the idle Q tiles and K/V
      // ring), then stored a 512-byte row per warp instruction; with output
      // fusion, four rows' old values are loaded before any is written
      const int prow = qt * BM + row;                     // 0..255
      const int sw = threadIdx.x >> 5;                    // softmax warp 0..7: rows 32 sw ..
      float* stage = reinterpret_cast<float*>(smem);      // [256][kStagePitch]
      const bool all_ok = softmax_all(staging_ok);
      if (all_ok) {
        // a head with no key blocks (block-sparse form) has O = 0, LSE = -inf
        const float wn = nloc > 0 ? wn0 / l : 0.0f;
        float* mine = stage + (size_t)prow * kStagePitch;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t orow[32];
          if (nloc > 0) {
            tmem_ld32(o_addr + 32 * c, orow);   // whole warp
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = 0u;
          }
          float4* d4 = reinterpret_cast<float4*>(mine + 32 * c);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            d4[v] = make_float4(__uint_as_float(orow[4 * v]) * wn, __uint_as_float(orow[4 * v + 1]) * wn,
                                __uint_as_float(orow[4 * v + 2]) * wn,
                                __uint_as_float(orow[4 * v + 3]) * wn);
        }
        if (kLse && store && p.lse)
          p.lse[(size_t)head * p.n_q + grow] = nloc > 0 ? m * p.scale + logf(lx) : -INFINITY;
        softmax_bar();
        const bool acc = p.accumulate != 0;
        for (int r0 = 0; r0 < 32; r0 += 4) {
          if (q0 + 32 * sw + r0 >= p.n_q) break;          // rows ascend (warp-uniform)
          float4 y[4], old[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = 32 * sw + r0 + u;
            y[u] = reinterpret_cast<const float4*>(stage + (size_t)r * kStagePitch)[lane];
            if (acc && q0 + r < p.n_q)
              old[u] = load4(static_cast<OutT*>(p.o) + ((size_t)(q0 + r) * p.n_heads + head) * HD +
                             4 * lane);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = 32 * sw + r0 + u;
            if (q0 + r >= p.n_q) break;
            put4(static_cast<OutT*>(p.o) + ((size_t)(q0 + r) * p.n_heads + head) * HD + 4 * lane, y[u],
                 acc, old[u], wo);
          }
        }
      }
    } else {
      // split: the unit's (head, query pair) key ranges meet through one
      // counter.  Each CTA takes an arrival ticket (low 16 bits); the last to
      // arrive combines, the others store their unnormalised rows and (m, l, lx)
      // to scratch and then count themselves done (high 16 bits).  The last CTA
      // waits (bounded) for the done count -- every CTA it waits for holds an
      // earlier ticket, so it is running and the wait is short -- and never
      // stores its own partial: its row statistics stay in registers and its
      // rows in the staging area.  It brings each other split's rows into shared
      // memory with bulk copies (64 KiB, half of the rows, at a time) and adds
      // the splits in split order, the same arithmetic as adding stored partials.
      const int unit = head * p.n_qpairs + qpair;
      const int prow = qt * BM + row;                     // 0..255 (= threadIdx.x)
      const int sw = threadIdx.x >> 5;                    // softmax warp 0..7
      float* stage = reinterpret_cast<float*>(smem);      // [256][kStagePitch]
      float* cbuf = stage + 256 * kStagePitch;            // [128][HD]: one split's half
      float* wts = cbuf + 128 * HD;                       // [n_split][256] row weights
      const bool all_ok = softmax_all(staging_ok);
      if (all_ok) {
        float* mine = stage + (size_t)prow * kStagePitch;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t orow[32];
          if (nloc > 0) {   // an empty key range (block-sparse form) leaves O = 0, m = -inf, l = 0
            tmem_ld32(o_addr + 32 * c, orow);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = 0u;
          }
          float4* d4 = reinterpret_cast<float4*>(mine + 32 * c);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            d4[v] = make_float4(__uint_as_float(orow[4 * v]), __uint_as_float(orow[4 * v + 1]),
                                __uint_as_float(orow[4 * v + 2]), __uint_as_float(orow[4 * v + 3]));
        }
      }
      softmax_bar();
      if (threadIdx.x == 0) bars->ticket = atomicAdd(&p.counters[unit], 1u);
      softmax_bar();
      const bool last = (bars->ticket & 0xffffu) == (unsigned)(p.n_split - 1);
      if (!last) {
        if (all_ok) {
          __stcg(p.part_ml + ((size_t)unit * p.n_split + split) * 256 + prow,
                 make_float4(m, l, lx, 0.f));
          float* dst = p.part_o + ((size_t)unit * p.n_split + split) * 256 * HD;
#pragma unroll 4
          for (int rr = 0; rr < 32; ++rr) {
            const int r = 32 * sw + rr;
            __stcg(reinterpret_cast<float4*>(dst + (size_t)r * HD) + lane,
                   reinterpret_cast<const float4*>(stage + (size_t)r * kStagePitch)[lane]);
          }
        }
        // one fence, by the thread that counts: the barrier orders the other
        // threads' stores before it (a fence is cumulative)
        softmax_bar();
        if (threadIdx.x == 0) {
          __threadfence();
          atomicAdd(&p.counters[unit], 1u << 16);
        }
      } else {
        if (threadIdx.x == 0) {
          volatile unsigned* cnt = &p.counters[unit];
          const unsigned need = (unsigned)(p.n_split - 1);
          bool done = (*cnt >> 16) >= need;
          const unsigned long long t0 = globaltimer();
          for (uint32_t it = 1; !done; ++it) {
            __nanosleep(64);
            done = (*cnt >> 16) >= need;
            if (!done && (it & 63u) == 0 && globaltimer() - t0 > p.wait_ns) break;
          }
          if (done) {
            __threadfence();
            // the bulk copies below read, through the async proxy, what the other
            // splits stored through the generic one
            asm volatile("fence.proxy.async.global;" ::: "memory");
            *cnt = 0u;
          } else {
            atomicOr(p.status, kStatusTimeout);
          }
          bars->ticket = done ? 1u : 0u;
        }
        softmax_bar();   // thread 0 fenced after seeing the done count: the others read after it
        bool go = all_ok && bars->ticket == 1u;
        if (go) {
          // this thread's row: statistics of every split (its own from registers),
          // the common maximum, the denominators, the LSE and the split weights
          const float4* mlp = p.part_ml + (size_t)unit * p.n_split * 256 + prow;
          float mm = -INFINITY;
          for (int s = 0; s < p.n_split; ++s)
            mm = fmaxf(mm, s == split ? m : __ldcg(mlp + (size_t)s * 256).x);
          const bool none = !(mm > -INFINITY);   // no keys in any split: O = 0, LSE = -inf
          float den = 0.f, denx = 0.f;
          for (int s = 0; s < p.n_split; ++s) {
            const float4 t = s == split ? make_float4(m, l, lx, 0.f) : __ldcg(mlp + (size_t)s * 256);
            const float w = none ? 0.f : ex2((t.x - mm) * sl2);
            den += w * t.y;
            denx += w * t.z;
          }
          const float wn = none ? 0.f : wn0 / den;
          for (int s = 0; s < p.n_split; ++s) {
            const float ms = s == split ? m : __ldcg(mlp + (size_t)s * 256).x;
            wts[s * 256 + prow] = none ? 0.f : ex2((ms - mm) * sl2) * wn;
          }
          if (kLse && p.lse && q0 + prow < p.n_q)
            p.lse[(size_t)head * p.n_q + q0 + prow] = none ? -INFINITY : mm * p.scale + logf(denx);
        }
        softmax_bar();
        // rows in two halves of 128; warp sw adds rows 128 h + 16 sw .. + 15,
        // lane = four output columns
        uint32_t cphase = 0;
        for (int h = 0; go && h < 2; ++h) {
          float4 x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s = 0; go && s < p.n_split; ++s) {
            const float* src;
            int pitch;
            if (s == split) {
              src = stage + (size_t)(128 * h) * kStagePitch;
              pitch = kStagePitch;
            } else {
              if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(&bars->comb, 128 * HD * 4);
                bulk_g2s(cbuf, p.part_o + (((size_t)unit * p.n_split + s) * 256 + 128 * h) * HD,
                         128 * HD * 4, &bars->comb);
              }
              go = softmax_all(mbar_wait(&bars->comb, cphase & 1, abort_flag, p.status, p.wait_ns));
              // a wait that gave up: the copy still lands before the CTA leaves
              if (!go) mbar_wait_drain(&bars->comb, cphase & 1, 100000000ull);
              ++cphase;
              src = cbuf;
              pitch = HD;
            }
            if (go) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int r = 16 * sw + i;
                const float w = wts[s * 256 + 128 * h + r];
                const float4 y = reinterpret_cast<const float4*>(src + (size_t)r * pitch)[lane];
                x[i].x += w * y.x;
                x[i].y += w * y.y;
                x[i].z += w * y.z;
                x[i].w += w * y.w;
              }
            }
            if (s != split) {
              // the buffer's readers finish before the next copy overwrites it
              fence_proxy_async_smem();
              softmax_bar();
            }
          }
          if (go) {
            // four rows at a time: with output fusion their old values are all
            // loaded before any is written
            const bool acc = p.accumulate != 0;
#pragma unroll
            for (int i0 = 0; i0 < 16; i0 += 4) {
              float4 old[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int grow_r = q0 + 128 * h + 16 * sw + i0 + u;
                old[u] = (acc && grow_r < p.n_q)
                             ? load4(static_cast<OutT*>(p.o) +
                                     ((size_t)grow_r * p.n_heads + head) * HD + 4 * lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int grow_r = q0 + 128 * h + 16 * sw + i0 + u;
                if (grow_r < p.n_q)
                  put4(static_cast<OutT*>(p.o) + ((size_t)grow_r * p.n_heads + head) * HD + 4 * lane,
                       x[i0 + u], acc, old[u], wo);
              }
            }
          }
        }
      }
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

// Key tiles of the block-sparse form, one CTA per head.  A segment's blocks
// of b rows are grouped m = floor(128 / b) to a tile by block number (blocks
// m t .. m t + m - 1 of the segment); kept blocks of one group that follow
// each other share a tile, others get tiles of their own.  Entry i of the
// head's kept list starts a tile unless it continues the previous entry:
// same group, block number one higher.  Tile k starts at the k-th starting
// entry (an exclusive scan of the start flags, fixed order).
__global__ void __launch_bounds__(128)
k_sparse_tiles(const int32_t* __restrict__ sel, const int32_t* __restrict__ count, int stride,
               int nb_main, int b_main, int b_loc, int n_main, int n_loc, int2* __restrict__ tiles,
               int32_t* __restrict__ tile_count) {
  extern __shared__ int32_t blk[];             // [stride] kept blocks, then [128] partial counts
  int32_t* part = blk + stride;
  const int h = blockIdx.x;
  const int n = min(max(__ldg(count + h), 0), stride);
  for (int i = threadIdx.x; i < n; i += blockDim.x) blk[i] = __ldg(sel + (size_t)h * stride + i);
  __syncthreads();
  const int m_main = max(1, BN / b_main), m_loc = max(1, BN / b_loc);
  auto group_of = [&](int b) {
    return b < nb_main ? b / m_main : (1 << 29) + (b - nb_main) / m_loc;
  };
  auto starts = [&](int i) {
    if (i == 0) return true;
    const int b = blk[i], pb = blk[i - 1];
    return !(pb == b - 1 && group_of(pb) == group_of(b));
  };
  // each thread takes a contiguous chunk of the list
  const int chunk = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = min(n, (int)threadIdx.x * chunk), i1 = min(n, i0 + chunk);
  int mine = 0;
  for (int i = i0; i < i1; ++i) mine += starts(i) ? 1 : 0;
  part[threadIdx.x] = mine;
  __syncthreads();
  int t = 0;   // exclusive prefix over the threads before this one, in order
  for (int k = 0; k < (int)threadIdx.x; ++k) t += part[k];
  int2* out = tiles + (size_t)h * stride;
  for (int i = i0; i < i1; ++i) {
    if (!starts(i)) continue;
    const int b = blk[i];
    int e = i;
    while (e + 1 < n && !starts(e + 1)) ++e;       // the tile's last kept block
    const int sg = b < nb_main ? 0 : 1;
    const int r0 = sg == 0 ? b * b_main : (b - nb_main) * b_loc;
    const int be = blk[e];
    const int r_end = sg == 0 ? min(n_main, (be + 1) * b_main) : min(n_loc, (be - nb_main + 1) * b_loc);
    out[t++] = make_int2((sg << 30) | r0, r_end - r0);
  }
  if (threadIdx.x == blockDim.x - 1) tile_count[h] = t;
}

// Split count: fewest whole waves of the SMs per unit of work; a split adds a
// small combine cost, so ties keep the smaller count.
int choose_split(int units, int nkv, int sms) {
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 4; ++s) {
    if (nkv < 2 * s && s > 1) break;
    if (s > 1 && units > kMaxUnits) break;
    const long long ctas = (long long)units * s;
    const double waves = (double)((ctas + sms - 1) / sms);
    const double cost = waves / s * (s > 1 ? 1.03 : 1.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

struct Maps {
  CUtensorMap q, km, vm, kl, vl, kp, vp, kq, vq;
};

template <typename OutT, bool kLse, bool kSparse, bool kPaged>
wa_status launch_t(const Maps& m, const Params& p, int n_heads, cudaStream_t s) {
  const int smem = SmemLayout::total + 1024;
  static std::atomic<bool> attr_done[64];   // per device; setting it twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = k_block_attn_tc<OutT, kLse, kSparse, kPaged>;
  if (dev < 64 && !attr_done[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return WA_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_relaxed);
  }
  dim3 grid(p.n_qpairs * p.n_split, n_heads);
  return cuda_status(launch_pdl(kern, grid, dim3(kThreads), (size_t)smem, s, m.q, m.km, m.vm, m.kl,
                                m.vl, m.kp, m.vp, m.kq, m.vq, p));
}

template <bool kSparse, bool kPaged>
wa_status launch_form(const Maps& m, const Params& p, int n_heads, bool o_f32, bool want_lse,
                      cudaStream_t s) {
  if (o_f32)
    return want_lse ? launch_t<float, true, kSparse, kPaged>(m, p, n_heads, s)
                    : launch_t<float, false, kSparse, kPaged>(m, p, n_heads, s);
  return want_lse ? launch_t<__nv_bfloat16, true, kSparse, kPaged>(m, p, n_heads, s)
                  : launch_t<__nv_bfloat16, false, kSparse, kPaged>(m, p, n_heads, s);
}

}  // namespace

wa_status launch_attn_tc(const void* q, int n_q, const void* k_main, const void* v_main,
                         int n_main, const void* k_loc, const void* v_loc, int n_loc, int n_heads,
                         float scale, void* o, int o_f32, float* lse, int accumulate,
                         const float* w_old, const float* w_new, int max_split, cudaStream_t s,
                         const SparseBlocks* sparse, const PagedKV* paged) {
  if (sparse && paged) return WA_ERR_INVALID_ARG;
  const uint64_t cols = (uint64_t)n_heads * HD;
  Maps m;
  memset(&m, 0, sizeof(m));
  wa_status rc;
  if ((rc = make_tmap_2d_bf16(&m.q, q, cols, n_q, cols, 64, BM)) != WA_OK) return rc;
  // the buffer segment (paged form: the buffer as the stores' destination, if given)
  if (n_main > 0 && k_main) {
    if ((rc = make_tmap_2d_bf16(&m.km, k_main, cols, n_main, cols, 64, BN)) != WA_OK) return rc;
    if ((rc = make_tmap_2d_bf16(&m.vm, v_main, cols, n_main, cols, 64, BN)) != WA_OK) return rc;
  }
  if (n_loc > 0) {
    if ((rc = make_tmap_2d_bf16(&m.kl, k_loc, cols, n_loc, cols, 64, BN)) != WA_OK) return rc;
    if ((rc = make_tmap_2d_bf16(&m.vl, v_loc, cols, n_loc, cols, 64, BN)) != WA_OK) return rc;
  }
  if (paged) {
    // the page bank, read in 128-row boxes and in boxes of box_rows
    const uint64_t bank_rows = (uint64_t)paged->n_pages * paged->page_tokens;
    const uint32_t br = paged->page_tokens % 64 == 0 ? 64 : 8;
    if ((rc = make_tmap_2d_bf16(&m.kp, paged->k_pages, cols, bank_rows, cols, 64, br)) != WA_OK)
      return rc;
    if ((rc = make_tmap_2d_bf16(&m.vp, paged->v_pages, cols, bank_rows, cols, 64, br)) != WA_OK)
      return rc;
    if ((rc = make_tmap_2d_bf16(&m.kq, paged->k_pages, cols, bank_rows, cols, 64, 128)) != WA_OK)
      return rc;
    if ((rc = make_tmap_2d_bf16(&m.vq, paged->v_pages, cols, bank_rows, cols, 64, 128)) != WA_OK)
      return rc;
  }
  Params p;
  p.n_q = n_q;
  p.n_heads = n_heads;
  p.n_main = n_main;
  p.n_loc = n_loc;
  p.nt_main = (n_main + BN - 1) / BN;
  p.nt_loc = (n_loc + BN - 1) / BN;
  p.n_qpairs = (n_q + 2 * BM - 1) / (2 * BM);
  p.tiles = nullptr;
  p.tile_count = nullptr;
  p.tile_stride = sparse ? sparse->stride : 0;
  // the block-sparse form sizes its splits for every block kept (the counts
  // live on the device); CTAs whose share is empty finish at once
  const int nkv_max = sparse ? sparse->stride : p.nt_main + p.nt_loc;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  p.n_split = choose_split(p.n_qpairs * n_heads, nkv_max, sms);
  // WA_ATTN_SPLIT=n forces the split count (clamped to what the tiles allow)
  if (const char* env = getenv("WA_ATTN_SPLIT")) {
    int f = atoi(env);
    const int nkv = nkv_max;
    if (f >= 1) p.n_split = f > nkv ? nkv : f;
    if (p.n_split > kMaxSplit) p.n_split = kMaxSplit;
    if ((size_t)p.n_qpairs * n_heads > (size_t)kMaxUnits) p.n_split = 1;
  }
  if (max_split > 0 && p.n_split > max_split) p.n_split = max_split;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.accumulate = accumulate;
  p.w_old = w_old;
  p.w_new = w_new;
  p.part_o = nullptr;
  p.part_ml = nullptr;
  p.counters = nullptr;
  p.wait_ns = wait_limit_ns();
  p.withhold_q = fault_mode() == WA_FAULT_WAIT;
  p.idx = paged ? paged->idx : nullptr;
  p.idx_stride = paged ? paged->idx_stride : 0;
  p.page_tokens = paged ? paged->page_tokens : 0;
  p.n_pages = paged ? paged->n_pages : 0;
  p.bank_rows = paged ? paged->n_pages * paged->page_tokens : 0;
  p.box_rows = paged && paged->page_tokens % 64 != 0 ? 8 : 64;
  p.store_buf = paged && k_main ? 1 : 0;
  Scratch sc;
  const size_t units = (size_t)p.n_qpairs * n_heads;
  // scratch: [tiles (block-sparse form)][split partials]
  const size_t tile_bytes =
      sparse ? (((size_t)n_heads * p.tile_stride * sizeof(int2) + n_heads * sizeof(int32_t)) + 255) &
                   ~(size_t)255
             : 0;
  const size_t part_o_bytes = p.n_split > 1 ? units * p.n_split * 256 * HD * sizeof(float) : 0;
  const size_t part_ml_bytes = p.n_split > 1 ? units * p.n_split * 256 * sizeof(float4) : 0;
  if ((rc = get_scratch(tile_bytes + part_o_bytes + part_ml_bytes, &sc)) != WA_OK) return rc;
  p.status = &sc.ctrl->status;
  char* base = static_cast<char*>(sc.data);
  if (sparse) {
    int2* tiles = reinterpret_cast<int2*>(base);
    int32_t* tcount = reinterpret_cast<int32_t*>(tiles + (size_t)n_heads * p.tile_stride);
    const int nb_main = (n_main + sparse->b_main - 1) / sparse->b_main;
    k_sparse_tiles<<<n_heads, 128, (p.tile_stride + 128) * sizeof(int32_t), s>>>(
        sparse->sel, sparse->count, p.tile_stride, nb_main, sparse->b_main, sparse->b_loc, n_main,
        n_loc, tiles, tcount);
    if ((rc = cuda_status(cudaPeekAtLastError())) != WA_OK) return rc;
    p.tiles = tiles;
    p.tile_count = tcount;
  }
  if (p.n_split > 1) {
    p.part_o = reinterpret_cast<float*>(base + tile_bytes);
    p.part_ml = reinterpret_cast<float4*>(base + tile_bytes + part_o_bytes);
    p.counters = sc.ctrl->attn_counters;
  }
  const bool want_lse = lse != nullptr;
  if (sparse) return launch_form<true, false>(m, p, n_heads, o_f32, want_lse, s);
  if (paged) return launch_form<false, true>(m, p, n_heads, o_f32, want_lse, s);
  return launch_form<false, false>(m, p, n_heads, o_f32, want_lse, s);
}

}  // namespace wa
