/*
 * wa.h -- C ABI of libwa: page-retrieval sparse attention for one generated
 * chunk of a block-diffusion world model, on one GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   [WA] "WorldAttention: An Efficient Attention Architecture for Interactive
 *        Video World Models" (review page): HKV section (paper §3.1 HKV) --
 *        8-frame pages, page mean keys, prompt-stage top-1 chunk by cosine,
 *        page-stage score alpha = Qbar^T Kbar / sqrt(d_k), top-K_p (K_p = 4);
 *        Fig. 1 custom-kernels prong -- retrieved pages reorganised into one
 *        contiguous buffer; HSA section (paper §3.2 HSA) -- Linformer-style
 *        low-rank branch with per-head E_K, E_V in R^{L x r} and a per-head
 *        gate fusing the branches.
 *   [IX] "Inferix: A Block-Diffusion based Next-Generation Inference Engine
 *        for World Simulation" (summary page): §3 Technical Approach, Step 3
 *        -- Attention(Q, [K_cache (+) K_t], [V_cache (+) V_t]), no mask; KV
 *        Cache Manager -- range access, index-based selective fetch, offload
 *        to main memory.
 *
 * Conventions shared by every call
 *   - Layout is token-major: a KV or Q tensor is [tokens][n_heads][head_dim],
 *     dense, row stride n_heads*head_dim elements.  A page bank is
 *     [n_pages][page_tokens][n_heads][head_dim], so page j is one contiguous
 *     slab of page_tokens*n_heads*head_dim elements.
 *   - Element types: WA_BF16 (2-byte bfloat16) or WA_F32 (4-byte float).
 *     Page summaries, scores, prompt embeddings and LSE are always float32.
 *   - Pointers are device pointers unless stated, 16-byte aligned.  The
 *     caller owns every buffer.  Every call is asynchronous on `stream`
 *     (NULL = the legacy default stream) and returns after enqueueing.
 *   - The library keeps one internal scratch arena per device, allocated
 *     with cudaMalloc on first need and grown (after a device-wide
 *     synchronize) when a call needs more; wa_shutdown() frees it.  Calls
 *     that use scratch or its ticket counters (wa_page_summarize,
 *     wa_block_means, wa_block_means_segments, wa_select_pages and its
 *     per-head form, wa_sparse_select, and the attention calls
 *     wa_block_attn, wa_gather_attn, wa_sparse_attn, wa_linear_branch,
 *     whose key-range splits meet in scratch) must not run concurrently on
 *     one device: issue them on one stream, or order the streams.
 *   - Errors: arguments are validated on the host before any launch; a bad
 *     argument returns a status and enqueues nothing.  A launch failure
 *     returns WA_ERR_CUDA.  Kernels never trap: a device-side problem (a
 *     page index out of range, a wait that timed out) is recorded in a
 *     device status word that wa_check() reads.  No C++ exception crosses
 *     this ABI.  Non-finite inputs give unspecified (but memory-safe)
 *     results.
 */
#ifndef WA_H_
#define WA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* == cudaStream_t */
typedef struct CUstream_st* wa_stream_t;

typedef enum {
  WA_OK = 0,
  WA_ERR_INVALID_ARG = 1,   /* NULL pointer, non-positive size, k_p too large  */
  WA_ERR_SHAPE = 2,         /* a size the kernels do not support              */
  WA_ERR_DTYPE = 3,         /* unknown or unsupported element type            */
  WA_ERR_ALIGN = 4,         /* pointer not 16-byte aligned                    */
  WA_ERR_INDEX = 5,         /* page index out of range                        */
  WA_ERR_OOM = 6,           /* scratch allocation failed                      */
  WA_ERR_CUDA = 7,          /* CUDA runtime/launch error                      */
  WA_ERR_TIMEOUT = 8,       /* a device wait exceeded its limit (wa_check)    */
  WA_ERR_UNIMPLEMENTED = 9
} wa_status;

typedef enum { WA_F32 = 0, WA_BF16 = 1 } wa_dtype;

/* Human-readable name of a status.  Never NULL. */
const char* wa_strerror(wa_status s);

/* Library version, e.g. "wa 0.1.0 sm_103a". */
const char* wa_version(void);

/*
 * Page summaries ([WA] HKV: each page is scored through its mean key).
 *
 *   kbar_out[j][h][e] = (1/page_tokens) * sum_t k_pages[j][t][h][e]
 *
 * k_pages  : device, [n_pages][page_tokens][n_heads][head_dim] of `dt`.
 * kbar_out : device float32 [n_pages][n_heads][head_dim] (written).
 * Sums are fp32 in a fixed order (deterministic run to run).
 * Needs n_heads*head_dim <= 8192 and a multiple of 8 (bf16) / 4 (f32).
 */
wa_status wa_page_summarize(const void* k_pages, wa_dtype dt, int n_pages, int page_tokens,
                            int n_heads, int head_dim, float* kbar_out, wa_stream_t stream);

/*
 * Two-stage page retrieval for one chunk ([WA] HKV, stages 1 and 2).
 *
 *   Qbar[h]  = (1/n_q) sum_i q[i][h]                       (mean query)
 *   stage 1  : c* = argmax_m cos(prompt_cur, prompt_chunks[m]); a zero-norm
 *              vector has cosine 0; exact ties go to the lowest m.  Chunk m
 *              owns pages [m*pages_per_chunk, (m+1)*pages_per_chunk).
 *              With n_chunks == 0 the stage is skipped: every page is a
 *              candidate and *chunk_out = -1.
 *   stage 2  : alpha_j = sum_h Qbar[h] . kbar[j][h] / sqrt(head_dim) for each
 *              candidate j (one page set shared by all heads); keep the k_p
 *              largest, ties to the lowest page index.
 *
 * q            : device [n_q][n_heads][head_dim] of `dt`.
 * kbar         : device float32 [n_pages][n_heads][head_dim].
 * prompt_cur   : device float32 [prompt_dim]; prompt_chunks: device float32
 *                [n_chunks][prompt_dim] (both ignored when n_chunks == 0).
 * idx_out      : device int32 [k_p], written in ascending page order.
 * scores_out   : device float32 [k_p], alpha of idx_out (may be NULL).
 * chunk_out    : device int32 [1], the chunk picked (may be NULL).
 * k_p must not exceed the candidate count (pages_per_chunk, or n_pages
 * without the prompt stage) nor 1024: else WA_ERR_INVALID_ARG.  With the
 * prompt stage, n_chunks*pages_per_chunk must not exceed n_pages.
 * Indices never return to the host; the call does not synchronize.
 */
wa_status wa_select_pages(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                          const float* kbar, int n_pages,
                          const float* prompt_cur, const float* prompt_chunks, int n_chunks,
                          int prompt_dim, int pages_per_chunk, int k_p,
                          int32_t* idx_out, float* scores_out, int32_t* chunk_out,
                          wa_stream_t stream);

/*
 * wa_select_pages without any device allocation (there is no counterpart on
 * the pages; this is a deployment variant).  Same arguments, results and
 * errors as wa_select_pages, for callers that must not allocate device
 * memory once they are running -- a serving process that has handed all free
 * HBM to its own pool, or a latency-critical loop where a cudaMalloc (and the
 * device-wide synchronize that growing the library's scratch arena implies)
 * would stall other work.  This call performs no cudaMalloc or cudaFree.
 *
 * Its scratch is a fixed 2 MiB array (plus a 48 KiB control block) compiled
 * into the library; every GPU that loads the library holds it until the
 * process exits.  Limit: 4 * (B * n_heads * head_dim + n_heads * n_alpha +
 * n_chunks) bytes (each term rounded up to a multiple of 4 floats) must fit
 * in 2 MiB, where n_alpha = n_chunks * pages_per_chunk with the prompt stage
 * and n_pages without it, and B is the number of query row blocks:
 * B0 = min(floor((2 * SMs - n_chunks) / C), ceil(n_q / 16)), at least 1, then
 * B = ceil(n_q / ceil(n_q / B0)).  C, the column blocks, is n_heads / g with g
 * the smallest power of two that divides n_heads and makes g * head_dim at
 * least 32 16-byte vectors (doubling stops at the first g that no longer
 * divides n_heads) when head_dim is a whole number of 16-byte vectors of at
 * least 32 values, else C = 1.  The one-layer WorldAttention shape on 152 SMs
 * has g = 2, C = 6, B = 49: 49 * 1536 + 12 * 40 + 5 floats, about 296 KiB.
 * Larger requests return WA_ERR_SHAPE and enqueue nothing.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress; make that first call before any stream capture.
 * Every call shares the one array, which keeps the previous call's contents:
 * the call clears its ticket counters itself (cudaMemsetAsync on `stream`),
 * and calls that overlap on the GPU (other streams, other host threads)
 * race on the array and give wrong results; serialize them.
 */
wa_status wa_select_pages_noalloc(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                                  const float* kbar, int n_pages,
                                  const float* prompt_cur, const float* prompt_chunks,
                                  int n_chunks, int prompt_dim, int pages_per_chunk, int k_p,
                                  int32_t* idx_out, float* scores_out, int32_t* chunk_out,
                                  wa_stream_t stream);

/*
 * Gather of the retrieved pages into one contiguous buffer ([WA] Fig. 1,
 * custom kernels; [IX] KV Cache Manager, index-based selective fetch):
 *
 *   k_buf[s*page_tokens + t] = k_pages[idx[s]][t],  likewise v   (s < k_p)
 *
 * Source in device memory: a copy kernel reads the indices from idx_dev
 * (device int32 [k_p]); an index outside [0, n_pages) makes that slot's rows
 * zero and is recorded in the status word (WA_ERR_INDEX from wa_check).
 * Source in pinned host memory (cudaHostAlloc / cudaHostRegister; the DRAM
 * tier of [WA] HKV and [IX] offload), two ways:
 *   - idx_host given (host int32 [k_p]): one cudaMemcpyAsync per page and
 *     tensor on `stream` (copy engine); indices are checked on the host
 *     (WA_ERR_INDEX, nothing enqueued);
 *   - idx_host NULL, idx_dev given: the copy kernel reads the pages through
 *     their device mapping (the GPU's own loads over the CPU-GPU link), so
 *     the indices never return to the host; bad indices as for a device
 *     source.  The host memory must be mapped for the device (pinned memory
 *     under unified addressing is); else WA_ERR_INVALID_ARG.
 * k_buf, v_buf : device [k_p*page_tokens][n_heads][head_dim] of `dt`.
 * v_pages/v_buf may be NULL together (keys only).
 */
wa_status wa_gather_pages(const void* k_pages, const void* v_pages, wa_dtype dt, int n_pages,
                          int page_tokens, int n_heads, int head_dim,
                          const int32_t* idx_dev, const int32_t* idx_host, int k_p,
                          void* k_buf, void* v_buf, wa_stream_t stream);

/*
 * Per-head page selection (the per-head variant of the page stage, [WA] HKV
 * stage 2 scored one head at a time): the prompt stage as in
 * wa_select_pages, then for every head h
 *
 *   alpha[h][j] = qbar[h] . kbar[j][h] / sqrt(head_dim)
 *
 * and head h's top-k_p candidates (ties to the lower page index), ascending.
 * idx_out    : device int32 [n_heads][k_p]; scores_out: device float32
 *              [n_heads][k_p] or NULL; chunk_out: device int32 [1] or NULL.
 * Other arguments and errors as for wa_select_pages.
 */
wa_status wa_select_pages_per_head(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                                   const float* kbar, int n_pages, const float* prompt_cur,
                                   const float* prompt_chunks, int n_chunks, int prompt_dim,
                                   int pages_per_chunk, int k_p, int32_t* idx_out,
                                   float* scores_out, int32_t* chunk_out, wa_stream_t stream);

/*
 * Per-head gather: each head's slice of the contiguous buffer comes from that
 * head's pages,
 *
 *   k_buf[s*page_tokens + t][h][:] = k_pages[idx[h][s]][t][h][:]   (likewise V),
 *
 * so the buffer keeps the token-major [k_p*page_tokens][n_heads][head_dim]
 * layout that wa_block_attn reads.  idx_dev: device int32 [n_heads][k_p].
 * Device sources only (pages in pinned host memory: WA_ERR_INVALID_ARG); a
 * head row must be whole 16-byte vectors, n_heads <= 1024 and k_p <= 32767
 * (WA_ERR_SHAPE).  Bad indices zero
 * the head's slice of that slot and record WA_ERR_INDEX for wa_check.
 */
wa_status wa_gather_pages_per_head(const void* k_pages, const void* v_pages, wa_dtype dt,
                                   int n_pages, int page_tokens, int n_heads, int head_dim,
                                   const int32_t* idx_dev, int k_p, void* k_buf, void* v_buf,
                                   wa_stream_t stream);

/*
 * Block attention of the chunk's queries over the retrieved buffer plus the
 * chunk's own KV ([IX] §3 Step 3; no mask, bidirectional):
 *
 *   O[i][h]  = sum_k softmax_k(scale * q[i][h] . K[k][h]) V[k][h]
 *   lse[h][i] = ln sum_k exp(scale * q[i][h] . K[k][h])
 *   with K = [k_main ; k_loc] and V = [v_main ; v_loc] along tokens.
 *
 * q        : device [n_q][n_heads][head_dim] of `dt`.
 * o        : device [n_q][n_heads][head_dim] of `o_dt`, written: WA_F32 keeps
 *            the fp32 result; WA_BF16 rounds it to nearest even (adds up to
 *            half a bf16 ulp, 2^-8 relative).  With dt == WA_F32, o_dt must be
 *            WA_F32.
 * k_main, v_main : device [n_main][n_heads][head_dim]; k_loc, v_loc :
 *            [n_loc][n_heads][head_dim].  Either segment may be empty
 *            (size 0, pointers may be NULL) but not both.
 * lse      : device float32 [n_heads][n_q] or NULL.
 * scale <= 0 means 1/sqrt(head_dim).
 * WA_BF16 runs on the tensor cores (tcgen05, fp32 accumulation in TMEM) and
 * needs head_dim == 128.  WA_F32 runs fp32 FMA on the CUDA cores and needs
 * head_dim <= 256 and a multiple of 4.
 */
wa_status wa_block_attn(const void* q, int n_q, const void* k_main, const void* v_main, int n_main,
                        const void* k_loc, const void* v_loc, int n_loc, wa_dtype dt,
                        int n_heads, int head_dim, float scale, void* o, wa_dtype o_dt,
                        float* lse, wa_stream_t stream);

/*
 * Gather and block attention in one launch: the page gather ([WA] Fig. 1,
 * custom kernels) done by the attention's own tile copies.  The result is
 * that of wa_gather_pages (or wa_gather_pages_per_head) into k_buf, v_buf
 * followed by wa_block_attn over [k_buf ; k_loc], [v_buf ; v_loc], bit for bit:
 *
 *   k_buf[s*page_tokens + t][h] = k_pages[idx[s]][t][h]          (per_head == 0)
 *                               = k_pages[idx[h][s]][t][h]       (per_head != 0)
 *   O, lse as wa_block_attn with n_main = k_p * page_tokens      (likewise v)
 *
 * The attention reads its key and value tiles straight from the pages; each
 * buffer tile is also written to k_buf/v_buf once, from on-chip memory, so the
 * pages are read once instead of twice (gather, then attention).
 * k_pages, v_pages : device [n_pages][page_tokens][n_heads][head_dim] of `dt`.
 * idx_dev  : device int32 [k_p] (per_head == 0) or [n_heads][k_p]; an index
 *            outside [0, n_pages) reads as a page of zeros (its buffer rows
 *            are written as zeros) and is recorded (WA_ERR_INDEX from wa_check).
 * k_buf, v_buf : device [k_p*page_tokens][n_heads][head_dim] of `dt`, written;
 *            or both NULL (attention only, no buffer written).
 * k_loc, v_loc, n_loc, q, o, o_dt, lse, scale : as for wa_block_attn.
 * WA_BF16 runs the tensor-core kernel and needs head_dim == 128 and
 * page_tokens a multiple of 8 (a multiple of 64 keeps the tiles that cross a
 * page boundary at 4 copies instead of 32); WA_F32 runs the CUDA-core kernel (o_dt
 * WA_F32, head_dim <= 256 and a multiple of 4, any page_tokens), where each
 * head's first CTA writes that head's buffer rows as it reads them
 * (WA_ERR_SHAPE / WA_ERR_DTYPE otherwise).  Pages in device memory
 * (WA_ERR_INVALID_ARG); 16-byte aligned pointers (WA_ERR_ALIGN).  Pages in
 * pinned host memory: wa_gather_pages, then wa_block_attn.
 */
wa_status wa_gather_attn(const void* q, int n_q, const void* k_pages, const void* v_pages,
                         int n_pages, int page_tokens, const int32_t* idx_dev, int k_p,
                         int per_head, void* k_buf, void* v_buf, const void* k_loc,
                         const void* v_loc, int n_loc, wa_dtype dt, int n_heads, int head_dim,
                         float scale, void* o, wa_dtype o_dt, float* lse, wa_stream_t stream);

/*
 * Linformer-style low-rank branch and gate fusion ([WA] HSA, linear branch;
 * the projection and gate equations are missing on the page and read as
 * Linformer and a per-head weighted sum):
 *
 *   K'[h] = E_K[h]^T [k_main ; k_loc][h],  V'[h] = E_V[h]^T [v_main ; v_loc][h]
 *   O_lin[i][h] = sum_r softmax_r(scale * q[i][h] . K'[h][r]) V'[h][r]
 *   accumulate != 0 :  o = w_attn[h] * o + w_lin[h] * O_lin
 *   accumulate == 0 :  o = O_lin
 *
 * e_k, e_v : device [n_heads][n_main+n_loc][rank] of `dt` (rows aligned to
 *            [main ; local]).  K', V' are accumulated in fp32 and rounded to
 *            `dt` before the second contraction.
 * o        : device [n_q][n_heads][head_dim] of `o_dt` (WA_BF16 or WA_F32).
 * w_attn, w_lin : device float32 [n_heads] or NULL (= all ones).
 * WA_BF16 only; needs head_dim == 128 and rank a multiple of 128, <= 512.
 */
wa_status wa_linear_branch(const void* q, int n_q, const void* k_main, const void* v_main,
                           int n_main, const void* k_loc, const void* v_loc, int n_loc,
                           const void* e_k, const void* e_v, int rank, wa_dtype dt,
                           int n_heads, int head_dim, float scale,
                           const float* w_attn, const float* w_lin, int accumulate,
                           void* o, wa_dtype o_dt, wa_stream_t stream);

/*
 * Block means ([WA] HSA, sparse branch: pooled tokens of a block):
 *
 *   means[b][h][:] = mean of x[r][h][:] over rows r in [b*block, min((b+1)*block, n_rows))
 *
 * a ragged last block divided by its own row count.
 * x         : device [n_rows][n_heads][head_dim] of `dt` (16-byte aligned).
 * means_out : device float32 [ceil(n_rows/block)][n_heads][head_dim].
 * Errors: WA_ERR_SHAPE when n_heads*head_dim is not whole 16-byte vectors or
 * exceeds 8192, or there are more than 4000 blocks.
 */
wa_status wa_block_means(const void* x, wa_dtype dt, int n_rows, int block, int n_heads,
                         int head_dim, float* means_out, wa_stream_t stream);

/*
 * Block means of up to three row sets in one launch (the HSA step pools the
 * queries, the retrieved buffer and the local KV at once; a launch per set
 * leaves most SMs idle on the two small ones):
 *
 *   means_out[i][b][h][:] = mean of xs[i][r][h][:] over rows r in
 *                           [b*blocks[i], min((b+1)*blocks[i], n_rows[i]))
 *
 * n_seg      : 1..3.
 * xs, n_rows, blocks, means_out : host arrays of n_seg entries; xs[i] and
 *              means_out[i] are device pointers laid out as in wa_block_means.
 * Every set's means equal those of wa_block_means on that set alone, bit for
 * bit (a set's row ranges and reduction order do not depend on the others).
 * Errors: as wa_block_means, per set; WA_ERR_INVALID_ARG for n_seg outside 1..3.
 */
wa_status wa_block_means_segments(int n_seg, const void* const* xs, const int* n_rows,
                                  const int* blocks, wa_dtype dt, int n_heads, int head_dim,
                                  float* const* means_out, wa_stream_t stream);

/*
 * Block selection of the HSA sparse branch ([WA] HSA: pooled attention map,
 * head-adaptive cumulative-mass selection; the Gini-to-threshold formula is
 * missing on the page and read as tau_h = 1 - G_h):
 *
 *   A_h[qb][kb] = softmax_kb(scale * qbar[qb][h] . kbar[kb][h])
 *   mass_h[kb]  = mean over qb of A_h[qb][kb]
 *   G_h         = Gini coefficient of mass_h
 *   tau_h       = tau[h] if tau != NULL, else 1 - G_h
 *   kept_h      = the fewest blocks in order of mass (descending; ties to the
 *                 lower index) whose cumulative mass reaches tau_h (>= 1 block)
 *
 * qbar      : device float32 [n_qb][n_heads][head_dim] (query-block means).
 * kbar      : device float32 [n_kb][n_heads][head_dim] (key-block means, the
 *             buffer's blocks first, then the local blocks).
 * tau       : device float32 [n_heads] or NULL.
 * sel_out   : device int32 [n_heads][n_kb]: row h starts with the count_out[h]
 *             kept block indices in ascending order; the rest is unspecified.
 * count_out : device int32 [n_heads].
 * gini_out  : device float32 [n_heads] or NULL; mass_out : device float32
 *             [n_heads][n_kb] or NULL.
 * scale <= 0 means 1/sqrt(head_dim).  Deterministic (fixed-order sums).
 * Needs n_qb <= 4096 and head_dim <= 256, a multiple of 4 (else WA_ERR_SHAPE),
 * and 16-byte aligned qbar, kbar (else WA_ERR_ALIGN).
 */
wa_status wa_sparse_select(const float* qbar, int n_qb, const float* kbar, int n_kb, int n_heads,
                           int head_dim, float scale, const float* tau, int32_t* sel_out,
                           int32_t* count_out, float* gini_out, float* mass_out,
                           wa_stream_t stream);

/*
 * Block-sparse attention of the HSA sparse branch: wa_block_attn restricted,
 * per head, to the tokens of the kept key blocks:
 *
 *   O[i][h] = sum_{k in kept blocks of h} softmax_k(scale * q[i][h] . K[k][h]) V[k][h]
 *
 * Key block b < nb = ceil(n_main/block_main) covers buffer rows
 * [b*block_main, min((b+1)*block_main, n_main)); block b >= nb covers local
 * rows [(b-nb)*block_loc, ...) of k_loc/v_loc.
 * sel, count : device int32 [n_heads][nb + ceil(n_loc/block_loc)] and
 *             [n_heads] as written by wa_sparse_select.  A head with count 0
 *             gets O = 0 and LSE = -inf; indices must be valid block numbers
 *             (the kernel does not check them).
 * block_main, block_loc : 1 .. 128; at most 12,000 blocks in all.
 * Adjacent kept blocks of one segment are processed as one key tile of up to
 * 128 rows (two 64-token local blocks share a tile).
 * Other arguments as for wa_block_attn; WA_BF16 only, head_dim == 128.
 */
wa_status wa_sparse_attn(const void* q, int n_q, const void* k_main, const void* v_main, int n_main,
                         const void* k_loc, const void* v_loc, int n_loc, int block_main,
                         int block_loc, const int32_t* sel, const int32_t* count, wa_dtype dt,
                         int n_heads, int head_dim, float scale, void* o, wa_dtype o_dt,
                         float* lse, wa_stream_t stream);

/*
 * Compressed DRAM tier: FP8 E4M3 codec for pages ([WA] HKV tier L2; pages
 * crossing the CPU-GPU link as FP8 halve the bytes).  Per (token, head) row
 * of head_dim values: s = amax(|row|) / 448 and code = E4M3 round-to-nearest-
 * even of x / s (IEEE fp32 divisions); decoding writes bf16 RNE(value(code) * s).
 * A zero row has s = 0 and codes 0.  head_dim must be 64, 128 or 256
 * (WA_ERR_SHAPE); all pointers 16-byte aligned (WA_ERR_ALIGN).  Codes and
 * scales may be device memory or pinned host memory (read or written through
 * the device mapping, i.e. across the link); x and out are device memory.
 *
 * wa_fp8_encode       : x bf16 [n_tokens][n_heads][head_dim] -> codes uint8
 *                       [n_tokens][n_heads][head_dim], scales float32 [n_tokens][n_heads].
 * wa_fp8_decode       : the inverse, into out bf16 [n_tokens][n_heads][head_dim].
 * wa_gather_pages_fp8 : out[s*page_tokens + t] = decode(page idx_dev[s], token t) for
 *                       code pages [n_pages][page_tokens][n_heads][head_dim] and scale
 *                       pages [n_pages][page_tokens][n_heads]; idx_dev device int32 [k_p];
 *                       a bad index zeroes the slot and records WA_ERR_INDEX.
 */
wa_status wa_fp8_encode(const void* x, int n_tokens, int n_heads, int head_dim, uint8_t* codes_out,
                        float* scales_out, wa_stream_t stream);
wa_status wa_fp8_decode(const uint8_t* codes, const float* scales, int n_tokens, int n_heads,
                        int head_dim, void* out, wa_stream_t stream);
wa_status wa_gather_pages_fp8(const uint8_t* code_pages, const float* scale_pages, int n_pages,
                              int page_tokens, int n_heads, int head_dim, const int32_t* idx_dev,
                              int k_p, void* buf_out, wa_stream_t stream);

/*
 * Compressed DRAM tier, NVFP4 form ([WA] HKV tier L2 with FP4 pages): per
 * (token, head) row of head_dim values, g = amax(|row|) / 2688 (fp32), per
 * block of 16 values an E4M3 scale sb = E4M3 RNE of amax(|block|) / (6 g), and
 * per value the E2M1 round-to-nearest-even (saturating at 6) of x / (sb * g);
 * each quotient and product one IEEE fp32 operation.  Decoding writes
 * bf16 RNE(value(code) * (value(sb) * g)).  A zero row has g = 0, zero block
 * scales and codes 0.  head_dim must be 64, 128 or 256 (WA_ERR_SHAPE); all
 * pointers 16-byte aligned (WA_ERR_ALIGN).  Codes and scales may be device
 * memory or pinned host memory (read or written through the device mapping).
 *
 * wa_nvfp4_encode       : x bf16 [n_tokens][n_heads][head_dim] -> codes uint8
 *                         [n_tokens][n_heads][head_dim/2] (two values per byte, the
 *                         even one in bits 0-3), block scales uint8 (E4M3 codes)
 *                         [n_tokens][n_heads][head_dim/16], row scales float32
 *                         [n_tokens][n_heads].
 * wa_nvfp4_decode       : the inverse, into out bf16 [n_tokens][n_heads][head_dim].
 * wa_gather_pages_nvfp4 : out[s*page_tokens + t] = decode(page idx_dev[s], token t) over
 *                         pages of page_tokens tokens in the three arrays above;
 *                         idx_dev device int32 [k_p]; a bad index zeroes the slot and
 *                         records WA_ERR_INDEX.
 */
wa_status wa_nvfp4_encode(const void* x, int n_tokens, int n_heads, int head_dim,
                          uint8_t* codes_out, uint8_t* bscales_out, float* rscales_out,
                          wa_stream_t stream);
wa_status wa_nvfp4_decode(const uint8_t* codes, const uint8_t* bscales, const float* rscales,
                          int n_tokens, int n_heads, int head_dim, void* out, wa_stream_t stream);
wa_status wa_gather_pages_nvfp4(const uint8_t* code_pages, const uint8_t* bscale_pages,
                                const float* rscale_pages, int n_pages, int page_tokens,
                                int n_heads, int head_dim, const int32_t* idx_dev, int k_p,
                                void* buf_out, wa_stream_t stream);

/*
 * KV cache manager around the path ([WA] HKV tiers L1/L2 and Fig. 2; [IX]
 * KV Cache Manager: append a clean block, range access, index-based selective
 * fetch, offload to main memory).  A host-side runtime over the calls above:
 *
 *   - pages of page_tokens tokens, pages_per_chunk per appended chunk, numbered
 *     in append order (chunk m owns pages m*ppc .. m*ppc + ppc - 1);
 *   - an HBM tier of hbm_pages page slots (K and V) and a pinned, device-mapped
 *     DRAM tier of host_pages slots; page summaries and prompt embeddings of
 *     every page stay in HBM;
 *   - the DRAM tier is inclusive: a page keeps its DRAM copy when promoted
 *     back to HBM (pages never change once appended), so evicting it again
 *     copies nothing;
 *   - dram_format 1 stores DRAM pages as FP8 E4M3 codes with per-(token, head)
 *     scales (the wa_fp8_encode format), 2 as NVFP4 (the wa_nvfp4_encode
 *     format); both need a bf16 cache with head_dim 64, 128 or 256.  A page read
 *     back from DRAM is decode(encode(page)), bit for bit, and stays so when
 *     promoted (its HBM copy is the decoded page);
 *   - append: pages to free HBM slots; when none is free the least recently
 *     used resident page leaves HBM: with no copy if it has a DRAM copy, else
 *     offloaded to the lowest free DRAM slot, or, with none free, to the slot of
 *     the most recently used page holding both copies (whose DRAM copy is
 *     dropped); summaries computed at insert;
 *   - offloads run on an internal copy stream from a device staging ring of
 *     pages_per_chunk + 4 pages, so they overlap the caller's later work;
 *     reads of a DRAM slot wait (device-side) for its copy to land;
 *   - retrieve: wa_select_pages over the cached pages, indices to the host (one
 *     synchronisation of `stream`), each page copied into the caller's buffer
 *     from HBM if it has an HBM copy, else from DRAM; pages found only in DRAM
 *     are promoted to HBM from the caller's buffer (a promotion that finds no
 *     DRAM slot for its victim gives up the promoted page's own DRAM copy);
 *   - window: the last n tokens of the sequence, contiguous (range access).
 * The LRU clock ticks once per append and per retrieval (ties: lower page).
 * Every call of one cache must use the same stream (its copies are ordered
 * against that stream).  dry_run != 0 makes a cache with no device memory and
 * no CUDA calls whose placement decisions can be driven with wa_cache_touch
 * (host-logic tests).  Not thread-safe; one cache per layer.
 */
typedef struct wa_cache wa_cache;

typedef struct {
  int n_heads, head_dim;
  wa_dtype dtype;
  int page_tokens;      /* tokens per page */
  int pages_per_chunk;  /* pages per appended chunk */
  int prompt_dim;       /* prompt embedding size; 0: no prompt stage */
  int hbm_pages;        /* HBM tier capacity (pages, >= 1) */
  int host_pages;       /* pinned DRAM tier capacity (pages, >= 0) */
  int max_chunks;       /* chunks the cache can hold */
  int dry_run;          /* 1: placement only, no device memory or copies */
  int dram_format;      /* DRAM tier: 0 the cache's dtype, 1 FP8 E4M3 codes + scales,
                           2 NVFP4 (wa_nvfp4_encode format) */
} wa_cache_config;

typedef struct {
  int n_pages, n_chunks;
  int in_hbm, in_host;                        /* pages with an HBM / a DRAM copy */
  long long offloads, promotions;             /* page copies HBM -> DRAM, DRAM -> HBM */
  long long bytes_h2d, bytes_d2h, bytes_d2d;  /* K+V bytes moved (dry run: planned); DRAM
                                                 bytes in the tier's format, staging
                                                 copies not counted */
  long long evictions;                        /* HBM copies dropped with no copy */
  long long reclaims;                         /* DRAM copies dropped to free a slot */
} wa_cache_stats;

/* Errors: WA_ERR_INVALID_ARG (also an unknown dram_format), WA_ERR_DTYPE (a
 * compressed dram_format with a non-bf16 dtype), WA_ERR_SHAPE (head rows not
 * whole 16-byte vectors; a compressed dram_format with head_dim not 64, 128 or
 * 256), WA_ERR_OOM (allocation failed). */
wa_status wa_cache_create(const wa_cache_config* cfg, wa_cache** out);
/* Synchronizes the device (unless dry_run) and frees the cache. */
wa_status wa_cache_destroy(wa_cache* cache);
/* Empties the cache for a new sequence, keeping its memory (synchronizes the
 * device unless dry_run). */
wa_status wa_cache_reset(wa_cache* cache);
/* k, v: device [pages_per_chunk*page_tokens][n_heads][head_dim] of dtype (page
 * major); prompt: device float32 [prompt_dim] (NULL if prompt_dim == 0).
 * WA_ERR_OOM when both tiers or max_chunks are full. */
wa_status wa_cache_append_chunk(wa_cache* cache, const void* k, const void* v, const float* prompt,
                                wa_stream_t stream);
/* q: device [n_q][n_heads][head_dim]; prompt_cur: device float32 [prompt_dim] or
 * NULL (no prompt stage: every page is a candidate); k_buf, v_buf: device
 * [k_p*page_tokens][n_heads][head_dim]; idx_out: host int32 [k_p] (ascending). */
wa_status wa_cache_retrieve(wa_cache* cache, const void* q, int n_q, const float* prompt_cur,
                            int k_p, void* k_buf, void* v_buf, int32_t* idx_out,
                            wa_stream_t stream);
/* k_out, v_out: device [n_tokens][n_heads][head_dim]: the last n_tokens tokens. */
wa_status wa_cache_window(wa_cache* cache, int n_tokens, void* k_out, void* v_out,
                          wa_stream_t stream);
/* Dry-run caches only: use pages as one retrieval would (LRU and promotion). */
wa_status wa_cache_touch(wa_cache* cache, const int32_t* pages, int n);
/* Where a read of the page goes: tier 0 (HBM) with its HBM slot if it has an
 * HBM copy, else tier 1 with its DRAM slot.  WA_ERR_INDEX for unknown pages. */
wa_status wa_cache_page_location(const wa_cache* cache, int page, int* tier, int* slot);
/* Both copies of a page: its HBM slot and its DRAM slot, -1 where it has none. */
wa_status wa_cache_page_slots(const wa_cache* cache, int page, int* hbm_slot, int* host_slot);
/* Make `stream` wait (device-side, no host synchronisation) for every offload
 * copy issued so far, e.g. to time a loop whole or before reading DRAM slots on
 * the host.  A no-op for dry-run caches. */
wa_status wa_cache_wait_copies(wa_cache* cache, wa_stream_t stream);
wa_status wa_cache_get_stats(const wa_cache* cache, wa_cache_stats* out);

/*
 * Synchronize `stream`, then read and clear this device's status word.
 * Returns WA_OK, WA_ERR_INDEX (a gather index was out of range),
 * WA_ERR_TIMEOUT (a kernel wait gave up; the kernel returned early and its
 * outputs are invalid) or WA_ERR_CUDA (the stream reported an error).
 */
wa_status wa_check(wa_stream_t stream);

/* Free this device's scratch arena (after a device synchronize). */
wa_status wa_shutdown(void);

/*
 * Upper limit, in nanoseconds, of each bounded wait inside the kernels that
 * pipeline copies and tensor-core work (wa_block_attn, wa_linear_branch,
 * wa_sparse_attn) for launches made after this call; 0 restores the default
 * of 4 s.  A wait that reaches the limit records WA_ERR_TIMEOUT in the status
 * word; the kernel then waits (with fixed limits of its own) for its copies
 * and MMAs in flight, frees its tensor memory and returns, so the context
 * stays usable.  Process-wide; not a property of any one stream.
 */
wa_status wa_set_wait_limit_ns(unsigned long long ns);

/*
 * Host-side fault injection for tests of the error paths; off by default and
 * process-wide.  No mode makes a GPU fault, trap or hang.
 *   WA_FAULT_NONE  : normal operation.
 *   WA_FAULT_ALLOC : any allocation the library would make (the scratch arena,
 *                    a cache's buffers) reports failure: the call returns
 *                    WA_ERR_OOM and enqueues nothing.  An arena that already
 *                    exists is used as before.
 *   WA_FAULT_COPY  : page copies from pinned host memory (wa_gather_pages with
 *                    host indices) report failure: WA_ERR_CUDA, nothing enqueued.
 *   WA_FAULT_WAIT  : wa_block_attn's copy producer withholds the query tiles,
 *                    so every wait on them runs out at the wait limit: the
 *                    launch returns WA_OK and wa_check() then WA_ERR_TIMEOUT.
 * The environment variable WA_FAULT (alloc | copy | wait) sets the mode when
 * the library is loaded.  Unknown modes return WA_ERR_INVALID_ARG.
 */
typedef enum { WA_FAULT_NONE = 0, WA_FAULT_ALLOC = 1, WA_FAULT_COPY = 2, WA_FAULT_WAIT = 3 } wa_fault;
wa_status wa_set_fault(int mode);

/* Size in bytes of the current device's scratch arena (0 when none has been
 * allocated yet, or after wa_shutdown); bytes_out is host memory. */
wa_status wa_scratch_bytes(size_t* bytes_out);

#ifdef __cplusplus
}
#endif

#endif /* WA_H_ */
