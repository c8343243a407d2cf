// Internal declarations shared by the libwa translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/wa.h"

namespace wa {

// Device status word bits (OR-ed by kernels, read and cleared by wa_check).
enum : int {
  kStatusIndex = 1,     // a gather index was outside [0, n_pages)
  kStatusTimeout = 2,   // a bounded wait gave up
};

// Process-wide settings read by the launchers (wa_set_wait_limit_ns, wa_set_fault).
unsigned long long wait_limit_ns();
int fault_mode();

// Per-device control block at the start of the scratch arena.
struct Ctrl {
  int status;           // kStatus* bits
  int pad[31];
  unsigned int counters[4096];        // zero between launches; "last CTA" tickets
  unsigned int attn_counters[8192];   // per (head, query-tile pair) of a split attention
};

// Scratch arena of the current device: Ctrl block + `bytes` of data.
// Grows (after cudaDeviceSynchronize) when a call needs more.
struct Scratch {
  Ctrl* ctrl;
  void* data;
  size_t bytes;
};
wa_status get_scratch(size_t bytes, Scratch* out);

// Status word of the current device (allocates the arena if needed).
wa_status get_ctrl(Ctrl** out);

inline wa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? WA_OK : WA_ERR_CUDA; }

// Programmatic dependent launch.  The kernels of one chunk (summaries,
// selection, gather, attention) are launched with the programmatic-stream-
// serialization attribute, so that the launch of a kernel overlaps the drain of
// the previous kernel on the stream; each such kernel calls pdl_wait() before
// its first access to global memory, which returns once every earlier kernel
// on the stream has finished and its writes are visible (it is a no-op for a
// kernel launched without the attribute).  None of them triggers its
// dependents early: measured on the one-layer WorldAttention step, CTAs of the
// next kernel placed while a kernel still ran made the step 36 us slower,
// while launching at grid completion made it 10 us faster than no attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int sm_count() {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// Blocks of `kernel` that are resident on the whole GPU at once (SM count x
// blocks per SM at this block size).
template <typename Kernel>
size_t resident_blocks(Kernel kernel, int threads, size_t dyn_smem = 0) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  return (size_t)sm_count() * (size_t)per_sm;
}

// 2-D bf16 TMA descriptor over a row-major [rows][cols] matrix with a row
// stride of `row_stride` elements; box = box_rows x box_cols (box_cols * 2
// bytes <= 128), 128-byte swizzle, out-of-range rows and columns read as 0.
wa_status make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                            uint64_t row_stride, uint32_t box_cols, uint32_t box_rows);

// 3-D bf16 TMA descriptor over [d2][d1][d0] (d0 contiguous) with strides s1, s2
// (elements) for dims 1 and 2; box = 1 x box1 x box0, 128-byte swizzle, zero fill.
wa_status make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t d2, uint64_t s1, uint64_t s2, uint32_t box0, uint32_t box1);

// ---------------------------------------------------------------------------
// kernel launchers (one per translation unit / kernel family)
// ---------------------------------------------------------------------------
wa_status launch_page_summarize(const void* k_pages, wa_dtype dt, int n_pages, int page_tokens,
                                int row_elems, float* kbar_out, cudaStream_t s);

wa_status launch_select_pages(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                              const float* kbar, int n_pages, const float* prompt_cur,
                              const float* prompt_chunks, int n_chunks, int prompt_dim,
                              int pages_per_chunk, int k_p, int32_t* idx_out, float* scores_out,
                              int32_t* chunk_out, cudaStream_t s, int per_head = 0);

// Per-head gather: k_buf[s*P + t][h] = k_pages[idx[h*k_p + s]][t][h] (and V); 16-byte
// vectors of each head row, indices read on the device.
wa_status launch_gather_per_head(const void* k_pages, const void* v_pages, int n_pages,
                                 int page_tokens, int n_heads, size_t head_row_bytes,
                                 const int32_t* idx_dev, int k_p, void* k_buf, void* v_buf,
                                 cudaStream_t s);

wa_status launch_gather_device(const void* k_pages, const void* v_pages, size_t page_bytes,
                               int n_pages, const int32_t* idx_dev, int k_p, void* k_buf,
                               void* v_buf, cudaStream_t s);

struct PagedKV;
// fp32 attention on the CUDA cores; with `paged`, the buffer segment comes from
// the page bank (k_main/v_main then name the buffer to write, or are NULL).
wa_status launch_attn_f32(const float* q, int n_q, const float* k_main, const float* v_main,
                          int n_main, const float* k_loc, const float* v_loc, int n_loc,
                          int n_heads, int head_dim, float scale, float* o, float* lse,
                          cudaStream_t s, const PagedKV* paged = nullptr);

// bf16 tensor-core attention.  w_old/w_new: per-head fusion weights for the
// epilogue o = w_old[h]*o + w_new[h]*O (accumulate != 0), may be NULL.
// max_split: 0 = choose the key-range split automatically, else an upper
// bound (1 = no split, which also means no scratch is touched).
// Block-sparse form of the attention: head h attends to the key blocks
// sel[h * stride + t], t < count[h] (device arrays), each block b_main buffer
// rows (index < ceil(n_main / b_main)) or b_loc local rows; b_main, b_loc <= 128.
struct SparseBlocks {
  const int32_t* sel;
  const int32_t* count;
  int stride, b_main, b_loc;
};
// Paged form: the buffer segment's n_main = k_p * page_tokens rows are read from
// the page bank [n_pages][page_tokens][n_heads][128] through device indices
// idx[idx_stride * h + s] (page_tokens a multiple of 64); k_main/v_main, if
// given, receive the gathered buffer.
struct PagedKV {
  const void* k_pages;
  const void* v_pages;
  int n_pages, page_tokens;
  const int32_t* idx;
  int idx_stride;
};
wa_status launch_attn_tc(const void* q, int n_q, const void* k_main, const void* v_main,
                         int n_main, const void* k_loc, const void* v_loc, int n_loc,
                         int n_heads, float scale, void* o, int o_f32, float* lse, int accumulate,
                         const float* w_old, const float* w_new, int max_split, cudaStream_t s,
                         const SparseBlocks* sparse = nullptr, const PagedKV* paged = nullptr);

// FP8 E4M3 page codec (k_fp8.cu).  Rows are (token, head) rows of head_dim
// values; codes and scales may live in pinned host memory (device-mapped pointers).
wa_status launch_fp8_encode(const void* src, size_t n_rows, int head_dim, void* codes,
                            float* scales, cudaStream_t s);
wa_status launch_fp8_decode(const void* codes, const float* scales, const int32_t* idx, int n_pages,
                            size_t page_rows, size_t n_rows, int head_dim, void* out,
                            cudaStream_t s);

// NVFP4 page codec (k_fp4.cu): E2M1 codes [rows][d/2], E4M3 block scales
// [rows][d/16], fp32 row scales [rows]; host-mapped pointers allowed.
wa_status launch_nvfp4_encode(const void* src, size_t n_rows, int head_dim, void* codes,
                              void* bscales, float* rscales, cudaStream_t s);
wa_status launch_nvfp4_decode(const void* codes, const void* bscales, const float* rscales,
                              const int32_t* idx, int n_pages, size_t page_rows, size_t n_rows,
                              int head_dim, void* out, cudaStream_t s);

// Block means of n_seg (1..3) row sets xs[i] [n_rows[i]][row_elems] in blocks of
// blocks[i] rows (ragged last block) into means_out[i], in one launch.
wa_status launch_block_means(int n_seg, const void* const* xs, const int* n_rows,
                             const int* blocks, wa_dtype dt, int row_elems,
                             float* const* means_out, cudaStream_t s);

// HSA block selection (k_sparse.cu) and the limits its host checks use.
wa_status launch_sparse_select(const float* qbar, int n_qb, const float* kbar, int n_kb,
                               int n_heads, int head_dim, float scale, const float* tau,
                               int32_t* sel_out, int32_t* count_out, float* gini_out,
                               float* mass_out, cudaStream_t s);
int sparse_select_max_qb();
size_t sparse_select_smem(int n_qb, int n_kb, int head_dim);

wa_status launch_linear_branch(const void* q, int n_q, const void* k_main, const void* v_main,
                               int n_main, const void* k_loc, const void* v_loc, int n_loc,
                               const void* e_k, const void* e_v, int rank, int n_heads,
                               float scale, const float* w_attn, const float* w_lin,
                               int accumulate, void* o, int o_f32, cudaStream_t s);

}  // namespace wa
