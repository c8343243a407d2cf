// libwa C ABI: argument validation, per-device scratch arena, dispatch.
//
// Every entry point validates on the host and returns a status before any
// launch; no C++ exception escapes (all code here is exception-free).
#include <atomic>
#include <math.h>
#include <mutex>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "wa_internal.cuh"

namespace wa {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceArena {
  char* base = nullptr;   // Ctrl block followed by data
  size_t data_bytes = 0;
};

std::mutex g_mu;
DeviceArena g_arena[kMaxDevices];

constexpr size_t ctrl_bytes() { return (sizeof(Ctrl) + 255) & ~size_t(255); }

constexpr unsigned long long kDefaultWaitNs = 4000000000ull;   // 4 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

int fault_from_env() {
  const char* e = getenv("WA_FAULT");
  if (!e) return WA_FAULT_NONE;
  if (!strcmp(e, "alloc")) return WA_FAULT_ALLOC;
  if (!strcmp(e, "copy")) return WA_FAULT_COPY;
  if (!strcmp(e, "wait")) return WA_FAULT_WAIT;
  return WA_FAULT_NONE;
}
std::atomic<int> g_fault{fault_from_env()};

}  // namespace

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int fault_mode() { return g_fault.load(std::memory_order_relaxed); }

wa_status get_scratch(size_t bytes, Scratch* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceArena& a = g_arena[dev];
  if (a.base == nullptr || a.data_bytes < bytes) {
    if (fault_mode() == WA_FAULT_ALLOC) return WA_ERR_OOM;
    size_t want = bytes < (size_t(1) << 20) ? (size_t(1) << 20) : bytes;
    if (a.base != nullptr) {
      // Earlier launches may still read the old arena.
      if (cudaDeviceSynchronize() != cudaSuccess) return WA_ERR_CUDA;
      cudaFree(a.base);
      a.base = nullptr;
      a.data_bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, ctrl_bytes() + want) != cudaSuccess) {
      cudaGetLastError();
      return WA_ERR_OOM;
    }
    if (cudaMemset(p, 0, ctrl_bytes()) != cudaSuccess) {
      cudaFree(p);
      return WA_ERR_CUDA;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
      cudaFree(p);
      return WA_ERR_CUDA;
    }
    a.base = static_cast<char*>(p);
    a.data_bytes = want;
  }
  out->ctrl = reinterpret_cast<Ctrl*>(a.base);
  out->data = a.base + ctrl_bytes();
  out->bytes = a.data_bytes;
  return WA_OK;
}

wa_status get_ctrl(Ctrl** out) {
  Scratch s;
  wa_status st = get_scratch(0, &s);
  if (st != WA_OK) return st;
  *out = s.ctrl;
  return WA_OK;
}

}  // namespace wa

using namespace wa;

namespace {

inline size_t esize(wa_dtype dt) { return dt == WA_BF16 ? 2 : 4; }
inline bool dtype_ok(wa_dtype dt) { return dt == WA_BF16 || dt == WA_F32; }

// Row of n_heads*head_dim elements must be whole 16-byte vectors.
inline bool row_ok(int n_heads, int head_dim, wa_dtype dt) {
  if (n_heads <= 0 || head_dim <= 0) return false;
  long long row = (long long)n_heads * head_dim;
  return (row * (long long)esize(dt)) % 16 == 0;
}

}  // namespace

extern "C" {

const char* wa_strerror(wa_status s) {
  switch (s) {
    case WA_OK: return "WA_OK";
    case WA_ERR_INVALID_ARG: return "WA_ERR_INVALID_ARG: invalid argument";
    case WA_ERR_SHAPE: return "WA_ERR_SHAPE: unsupported shape";
    case WA_ERR_DTYPE: return "WA_ERR_DTYPE: unsupported element type";
    case WA_ERR_ALIGN: return "WA_ERR_ALIGN: pointer not 16-byte aligned";
    case WA_ERR_INDEX: return "WA_ERR_INDEX: page index out of range";
    case WA_ERR_OOM: return "WA_ERR_OOM: scratch allocation failed";
    case WA_ERR_CUDA: return "WA_ERR_CUDA: CUDA runtime error";
    case WA_ERR_TIMEOUT: return "WA_ERR_TIMEOUT: a device wait exceeded its limit";
    case WA_ERR_UNIMPLEMENTED: return "WA_ERR_UNIMPLEMENTED";
  }
  return "WA_ERR_UNKNOWN";
}

const char* wa_version(void) { return "wa 0.1.0 sm_103a"; }

wa_status wa_page_summarize(const void* k_pages, wa_dtype dt, int n_pages, int page_tokens,
                            int n_heads, int head_dim, float* kbar_out, wa_stream_t stream) {
  if (!dtype_ok(dt)) return WA_ERR_DTYPE;
  if (!k_pages || !kbar_out || n_pages <= 0 || page_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if ((long long)n_heads * head_dim > 8192) return WA_ERR_SHAPE;
  if (!aligned16(k_pages) || !aligned16(kbar_out)) return WA_ERR_ALIGN;
  return launch_page_summarize(k_pages, dt, n_pages, page_tokens, n_heads * head_dim, kbar_out,
                               (cudaStream_t)stream);
}

wa_status wa_select_pages(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                          const float* kbar, int n_pages, const float* prompt_cur,
                          const float* prompt_chunks, int n_chunks, int prompt_dim,
                          int pages_per_chunk, int k_p, int32_t* idx_out, float* scores_out,
                          int32_t* chunk_out, wa_stream_t stream) {
  if (!dtype_ok(dt)) return WA_ERR_DTYPE;
  if (!q || !kbar || !idx_out || n_q <= 0 || n_pages <= 0 || k_p <= 0 || n_chunks < 0)
    return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if ((long long)n_heads * head_dim > 8192) return WA_ERR_SHAPE;
  int n_cand = n_pages;
  if (n_chunks > 0) {
    if (!prompt_cur || !prompt_chunks || prompt_dim <= 0 || pages_per_chunk <= 0)
      return WA_ERR_INVALID_ARG;
    if ((long long)n_chunks * pages_per_chunk > n_pages) return WA_ERR_INVALID_ARG;
    n_cand = pages_per_chunk;
  }
  if (k_p > n_cand || k_p > 1024) return WA_ERR_INVALID_ARG;
  if (n_cand > 8192) return WA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(kbar)) return WA_ERR_ALIGN;
  return launch_select_pages(q, dt, n_q, n_heads, head_dim, kbar, n_pages, prompt_cur,
                             prompt_chunks, n_chunks, prompt_dim, pages_per_chunk, k_p, idx_out,
                             scores_out, chunk_out, (cudaStream_t)stream);
}

wa_status wa_select_pages_per_head(const void* q, wa_dtype dt, int n_q, int n_heads, int head_dim,
                                   const float* kbar, int n_pages, const float* prompt_cur,
                                   const float* prompt_chunks, int n_chunks, int prompt_dim,
                                   int pages_per_chunk, int k_p, int32_t* idx_out,
                                   float* scores_out, int32_t* chunk_out, wa_stream_t stream) {
  if (!dtype_ok(dt)) return WA_ERR_DTYPE;
  if (!q || !kbar || !idx_out || n_q <= 0 || n_pages <= 0 || k_p <= 0 || n_chunks < 0)
    return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if ((long long)n_heads * head_dim > 8192) return WA_ERR_SHAPE;
  int n_cand = n_pages;
  if (n_chunks > 0) {
    if (!prompt_cur || !prompt_chunks || prompt_dim <= 0 || pages_per_chunk <= 0)
      return WA_ERR_INVALID_ARG;
    if ((long long)n_chunks * pages_per_chunk > n_pages) return WA_ERR_INVALID_ARG;
    n_cand = pages_per_chunk;
  }
  if (k_p > n_cand || k_p > 1024) return WA_ERR_INVALID_ARG;
  if (n_cand > 8192) return WA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(kbar)) return WA_ERR_ALIGN;
  return launch_select_pages(q, dt, n_q, n_heads, head_dim, kbar, n_pages, prompt_cur,
                             prompt_chunks, n_chunks, prompt_dim, pages_per_chunk, k_p, idx_out,
                             scores_out, chunk_out, (cudaStream_t)stream, 1);
}

wa_status wa_gather_pages_per_head(const void* k_pages, const void* v_pages, wa_dtype dt,
                                   int n_pages, int page_tokens, int n_heads, int head_dim,
                                   const int32_t* idx_dev, int k_p, void* k_buf, void* v_buf,
                                   wa_stream_t stream) {
  if (!dtype_ok(dt)) return WA_ERR_DTYPE;
  if (!k_pages || !k_buf || !idx_dev || n_pages <= 0 || page_tokens <= 0 || k_p <= 0)
    return WA_ERR_INVALID_ARG;
  if ((v_pages == nullptr) != (v_buf == nullptr)) return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if ((head_dim * esize(dt)) % 16 != 0) return WA_ERR_SHAPE;
  if (!aligned16(k_pages) || !aligned16(k_buf) || (v_pages && (!aligned16(v_pages) ||
      !aligned16(v_buf))))
    return WA_ERR_ALIGN;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, k_pages) != cudaSuccess) {
    cudaGetLastError();
    return WA_ERR_INVALID_ARG;
  }
  if (attr.type != cudaMemoryTypeDevice) return WA_ERR_INVALID_ARG;
  return launch_gather_per_head(k_pages, v_pages, n_pages, page_tokens, n_heads,
                                (size_t)head_dim * esize(dt), idx_dev, k_p, k_buf, v_buf,
                                (cudaStream_t)stream);
}

wa_status wa_gather_pages(const void* k_pages, const void* v_pages, wa_dtype dt, int n_pages,
                          int page_tokens, int n_heads, int head_dim, const int32_t* idx_dev,
                          const int32_t* idx_host, int k_p, void* k_buf, void* v_buf,
                          wa_stream_t stream) {
  if (!dtype_ok(dt)) return WA_ERR_DTYPE;
  if (!k_pages || !k_buf || n_pages <= 0 || page_tokens <= 0 || k_p <= 0)
    return WA_ERR_INVALID_ARG;
  if ((v_pages == nullptr) != (v_buf == nullptr)) return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if (!aligned16(k_pages) || !aligned16(k_buf) || (v_pages && (!aligned16(v_pages) ||
      !aligned16(v_buf))))
    return WA_ERR_ALIGN;
  const size_t page_bytes = (size_t)page_tokens * n_heads * head_dim * esize(dt);
  cudaStream_t s = (cudaStream_t)stream;

  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, k_pages) != cudaSuccess) {
    cudaGetLastError();
    return WA_ERR_INVALID_ARG;
  }
  if (attr.type == cudaMemoryTypeHost) {
    // DRAM tier: pinned host pages, copy engine, host-side indices.
    if (v_pages) {
      cudaPointerAttributes av;
      if (cudaPointerGetAttributes(&av, v_pages) != cudaSuccess || av.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return WA_ERR_INVALID_ARG;
      }
    }
    if (!idx_host) {
      // device indices: the copy kernel reads the pinned pages through their
      // device mapping (GPU loads over the CPU-GPU link); no host round trip
      if (!idx_dev) return WA_ERR_INVALID_ARG;
      const void* kd = attr.devicePointer;
      const void* vd = nullptr;
      if (v_pages) {
        cudaPointerAttributes av;
        if (cudaPointerGetAttributes(&av, v_pages) != cudaSuccess) {
          cudaGetLastError();
          return WA_ERR_INVALID_ARG;
        }
        vd = av.devicePointer;
        if (!vd) return WA_ERR_INVALID_ARG;
      }
      if (!kd) return WA_ERR_INVALID_ARG;
      if (!aligned16(kd) || (vd && !aligned16(vd))) return WA_ERR_ALIGN;
      return launch_gather_device(kd, vd, page_bytes, n_pages, idx_dev, k_p, k_buf, v_buf, s);
    }
    for (int i = 0; i < k_p; ++i)
      if (idx_host[i] < 0 || idx_host[i] >= n_pages) return WA_ERR_INDEX;
    if (fault_mode() == WA_FAULT_COPY) return WA_ERR_CUDA;
    for (int i = 0; i < k_p; ++i) {
      const char* ks = static_cast<const char*>(k_pages) + (size_t)idx_host[i] * page_bytes;
      if (cudaMemcpyAsync(static_cast<char*>(k_buf) + (size_t)i * page_bytes, ks, page_bytes,
                          cudaMemcpyHostToDevice, s) != cudaSuccess)
        return WA_ERR_CUDA;
      if (v_pages) {
        const char* vs = static_cast<const char*>(v_pages) + (size_t)idx_host[i] * page_bytes;
        if (cudaMemcpyAsync(static_cast<char*>(v_buf) + (size_t)i * page_bytes, vs, page_bytes,
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
          return WA_ERR_CUDA;
      }
    }
    return WA_OK;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return WA_ERR_INVALID_ARG;
  if (!idx_dev) return WA_ERR_INVALID_ARG;
  return launch_gather_device(k_pages, v_pages, page_bytes, n_pages, idx_dev, k_p, k_buf, v_buf,
                              s);
}

wa_status wa_block_attn(const void* q, int n_q, const void* k_main, const void* v_main, int n_main,
                        const void* k_loc, const void* v_loc, int n_loc, wa_dtype dt,
                        int n_heads, int head_dim, float scale, void* o, wa_dtype o_dt,
                        float* lse, wa_stream_t stream) {
  if (!dtype_ok(dt) || !dtype_ok(o_dt)) return WA_ERR_DTYPE;
  if (dt == WA_F32 && o_dt != WA_F32) return WA_ERR_DTYPE;
  if (!q || !o || n_q <= 0 || n_main < 0 || n_loc < 0 || n_main + n_loc <= 0)
    return WA_ERR_INVALID_ARG;
  if (n_main > 0 && (!k_main || !v_main)) return WA_ERR_INVALID_ARG;
  if (n_loc > 0 && (!k_loc || !v_loc)) return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(o) || (n_main > 0 && (!aligned16(k_main) || !aligned16(v_main))) ||
      (n_loc > 0 && (!aligned16(k_loc) || !aligned16(v_loc))))
    return WA_ERR_ALIGN;
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)head_dim);
  cudaStream_t s = (cudaStream_t)stream;
  if (dt == WA_F32) {
    if (head_dim > 256 || head_dim % 4 != 0) return WA_ERR_SHAPE;
    return launch_attn_f32((const float*)q, n_q, (const float*)k_main, (const float*)v_main,
                           n_main, (const float*)k_loc, (const float*)v_loc, n_loc, n_heads,
                           head_dim, scale, (float*)o, lse, s);
  }
  if (head_dim != 128) return WA_ERR_SHAPE;
  if ((long long)n_heads * 128 > 16384) return WA_ERR_SHAPE;
  return launch_attn_tc(q, n_q, k_main, v_main, n_main, k_loc, v_loc, n_loc, n_heads, scale, o,
                        o_dt == WA_F32, lse, 0, nullptr, nullptr, 0, s);
}

wa_status wa_gather_attn(const void* q, int n_q, const void* k_pages, const void* v_pages,
                         int n_pages, int page_tokens, const int32_t* idx_dev, int k_p,
                         int per_head, void* k_buf, void* v_buf, const void* k_loc,
                         const void* v_loc, int n_loc, wa_dtype dt, int n_heads, int head_dim,
                         float scale, void* o, wa_dtype o_dt, float* lse, wa_stream_t stream) {
  if (!dtype_ok(dt) || !dtype_ok(o_dt)) return WA_ERR_DTYPE;
  if (dt == WA_F32 && o_dt != WA_F32) return WA_ERR_DTYPE;
  if (!q || !o || !k_pages || !v_pages || !idx_dev || n_q <= 0 || n_pages <= 0 ||
      page_tokens <= 0 || k_p <= 0 || n_loc < 0)
    return WA_ERR_INVALID_ARG;
  if ((k_buf == nullptr) != (v_buf == nullptr)) return WA_ERR_INVALID_ARG;
  if (n_loc > 0 && (!k_loc || !v_loc)) return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if (dt == WA_BF16 && (head_dim != 128 || (long long)n_heads * 128 > 16384 || page_tokens % 8 != 0))
    return WA_ERR_SHAPE;
  if (dt == WA_F32 && (head_dim > 256 || head_dim % 4 != 0)) return WA_ERR_SHAPE;
  if ((long long)n_pages * page_tokens > 0x7fffffffLL || (long long)k_p * page_tokens > 0x7fffffffLL)
    return WA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_pages) || !aligned16(v_pages) ||
      (k_buf && (!aligned16(k_buf) || !aligned16(v_buf))) ||
      (n_loc > 0 && (!aligned16(k_loc) || !aligned16(v_loc))))
    return WA_ERR_ALIGN;
  const void* const banks[2] = {k_pages, v_pages};
  for (const void* pages : banks) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, pages) != cudaSuccess) {
      cudaGetLastError();
      return WA_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
      return WA_ERR_INVALID_ARG;
  }
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)head_dim);
  PagedKV pk;
  pk.k_pages = k_pages;
  pk.v_pages = v_pages;
  pk.n_pages = n_pages;
  pk.page_tokens = page_tokens;
  pk.idx = idx_dev;
  pk.idx_stride = per_head ? k_p : 0;
  if (dt == WA_F32)
    return launch_attn_f32((const float*)q, n_q, (const float*)k_buf, (const float*)v_buf,
                           k_p * page_tokens, (const float*)k_loc, (const float*)v_loc, n_loc,
                           n_heads, head_dim, scale, (float*)o, lse, (cudaStream_t)stream, &pk);
  return launch_attn_tc(q, n_q, k_buf, v_buf, k_p * page_tokens, k_loc, v_loc, n_loc, n_heads,
                        scale, o, o_dt == WA_F32, lse, 0, nullptr, nullptr, 0,
                        (cudaStream_t)stream, nullptr, &pk);
}

// Device-usable address of p: device memory as is, pinned host memory through
// its device mapping; NULL if neither.
static const void* device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

static bool fp8_shape_ok(int n_heads, int head_dim) {
  return n_heads > 0 && (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

wa_status wa_fp8_encode(const void* x, int n_tokens, int n_heads, int head_dim, uint8_t* codes_out,
                        float* scales_out, wa_stream_t stream) {
  if (!x || !codes_out || !scales_out || n_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (!fp8_shape_ok(n_heads, head_dim)) return WA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(codes_out) || !aligned16(scales_out)) return WA_ERR_ALIGN;
  void* c = const_cast<void*>(device_view(codes_out));
  float* sc = static_cast<float*>(const_cast<void*>(device_view(scales_out)));
  if (!c || !sc || !device_view(x)) return WA_ERR_INVALID_ARG;
  return launch_fp8_encode(x, (size_t)n_tokens * n_heads, head_dim, c, sc, (cudaStream_t)stream);
}

wa_status wa_fp8_decode(const uint8_t* codes, const float* scales, int n_tokens, int n_heads,
                        int head_dim, void* out, wa_stream_t stream) {
  if (!codes || !scales || !out || n_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (!fp8_shape_ok(n_heads, head_dim)) return WA_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(out)) return WA_ERR_ALIGN;
  const void* c = device_view(codes);
  const float* sc = static_cast<const float*>(device_view(scales));
  if (!c || !sc) return WA_ERR_INVALID_ARG;
  const size_t rows = (size_t)n_tokens * n_heads;
  return launch_fp8_decode(c, sc, nullptr, 1, rows, rows, head_dim, out, (cudaStream_t)stream);
}

wa_status wa_gather_pages_fp8(const uint8_t* code_pages, const float* scale_pages, int n_pages,
                              int page_tokens, int n_heads, int head_dim, const int32_t* idx_dev,
                              int k_p, void* buf_out, wa_stream_t stream) {
  if (!code_pages || !scale_pages || !idx_dev || !buf_out || n_pages <= 0 || page_tokens <= 0 ||
      k_p <= 0)
    return WA_ERR_INVALID_ARG;
  if (!fp8_shape_ok(n_heads, head_dim)) return WA_ERR_SHAPE;
  if (!aligned16(code_pages) || !aligned16(scale_pages) || !aligned16(buf_out))
    return WA_ERR_ALIGN;
  const void* c = device_view(code_pages);
  const float* sc = static_cast<const float*>(device_view(scale_pages));
  if (!c || !sc) return WA_ERR_INVALID_ARG;
  const size_t page_rows = (size_t)page_tokens * n_heads;
  return launch_fp8_decode(c, sc, idx_dev, n_pages, page_rows, page_rows * k_p, head_dim, buf_out,
                           (cudaStream_t)stream);
}

wa_status wa_nvfp4_encode(const void* x, int n_tokens, int n_heads, int head_dim,
                          uint8_t* codes_out, uint8_t* bscales_out, float* rscales_out,
                          wa_stream_t stream) {
  if (!x || !codes_out || !bscales_out || !rscales_out || n_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (!fp8_shape_ok(n_heads, head_dim)) return WA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(codes_out) || !aligned16(bscales_out) || !aligned16(rscales_out))
    return WA_ERR_ALIGN;
  void* c = const_cast<void*>(device_view(codes_out));
  void* b = const_cast<void*>(device_view(bscales_out));
  float* r = static_cast<float*>(const_cast<void*>(device_view(rscales_out)));
  if (!c || !b || !r || !device_view(x)) return WA_ERR_INVALID_ARG;
  return launch_nvfp4_encode(x, (size_t)n_tokens * n_heads, head_dim, c, b, r,
                             (cudaStream_t)stream);
}

wa_status wa_nvfp4_decode(const uint8_t* codes, const uint8_t* bscales, const float* rscales,
                          int n_tokens, int n_heads, int head_dim, void* out, wa_stream_t stream) {
  if (!codes || !bscales || !rscales || !out || n_tokens <= 0) return WA_ERR_INVALID_ARG;
  if (!fp8_shape_ok(n_heads, head_dim)) return WA_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(bscales) || !aligned16(rscales) || !aligned16(out))
    return WA_ERR_ALIGN;
  const void* c = device_view(codes);
  const void* b = device_view(bscales);
  const float* r = static_cast<const float*>(device_view(rscales));
  if (!c || !b || !r) return WA_ERR_INVALID_ARG;
  const size_t rows = (size_t)n_tokens * n_heads;
  return launch_nvfp4_decode(c, b, r, nullptr, 1, rows, rows, head_dim, out, (cudaStream_t)stream);
}

wa_status wa_gather_pages_nvfp4(const uint8_t* code_pages, const uint8_t* bscale_pages,
                                const float* rscale_pages, int n_pages, int page_tokens,
                                int n_heads, int head_dim, const int32_t* idx_dev, int k_p,
                                void* buf_out, wa_stream_t stream) {
  if (!code_pages || !bscale_pages || !rscale_pages || !idx_dev || !buf_out || n_pages <= 0 ||
      page_tokens <= 0 || k_p <= 0)
    return WA_ERR_INVALID_ARG;
  if (!fp8_shape_ok(n_heads, head_dim)) return WA_ERR_SHAPE;
  if (!aligned16(code_pages) || !aligned16(bscale_pages) || !aligned16(rscale_pages) ||
      !aligned16(buf_out))
    return WA_ERR_ALIGN;
  const void* c = device_view(code_pages);
  const void* b = device_view(bscale_pages);
  const float* r = static_cast<const float*>(device_view(rscale_pages));
  if (!c || !b || !r) return WA_ERR_INVALID_ARG;
  const size_t page_rows = (size_t)page_tokens * n_heads;
  return launch_nvfp4_decode(c, b, r, idx_dev, n_pages, page_rows, page_rows * k_p, head_dim,
                             buf_out, (cudaStream_t)stream);
}

wa_status wa_block_means_segments(int n_seg, const void* const* xs, const int* n_rows,
                                  const int* blocks, wa_dtype dt, int n_heads, int head_dim,
                                  float* const* means_out, wa_stream_t stream) {
  if (!dtype_ok(dt)) return WA_ERR_DTYPE;
  if (n_seg < 1 || n_seg > 3 || !xs || !n_rows || !blocks || !means_out) return WA_ERR_INVALID_ARG;
  if (!row_ok(n_heads, head_dim, dt)) return WA_ERR_SHAPE;
  if ((long long)n_heads * head_dim > 8192) return WA_ERR_SHAPE;
  for (int i = 0; i < n_seg; ++i) {
    if (!xs[i] || !means_out[i] || n_rows[i] <= 0 || blocks[i] <= 0) return WA_ERR_INVALID_ARG;
    if ((n_rows[i] + (long long)blocks[i] - 1) / blocks[i] > 4000) return WA_ERR_SHAPE;
    if (!aligned16(xs[i]) || !aligned16(means_out[i])) return WA_ERR_ALIGN;
  }
  return launch_block_means(n_seg, xs, n_rows, blocks, dt, n_heads * head_dim, means_out,
                            (cudaStream_t)stream);
}

wa_status wa_block_means(const void* x, wa_dtype dt, int n_rows, int block, int n_heads,
                         int head_dim, float* means_out, wa_stream_t stream) {
  return wa_block_means_segments(1, &x, &n_rows, &block, dt, n_heads, head_dim, &means_out,
                                 stream);
}

wa_status wa_sparse_select(const float* qbar, int n_qb, const float* kbar, int n_kb, int n_heads,
                           int head_dim, float scale, const float* tau, int32_t* sel_out,
                           int32_t* count_out, float* gini_out, float* mass_out,
                           wa_stream_t stream) {
  if (!qbar || !kbar || !sel_out || !count_out || n_qb <= 0 || n_kb <= 0 || n_heads <= 0 ||
      head_dim <= 0)
    return WA_ERR_INVALID_ARG;
  if (head_dim > 256 || head_dim % 4 != 0 || n_qb > sparse_select_max_qb() || n_kb > (1 << 20))
    return WA_ERR_SHAPE;
  if (!aligned16(qbar) || !aligned16(kbar)) return WA_ERR_ALIGN;
  if (sparse_select_smem(n_qb, n_kb, head_dim) > 227 * 1024) return WA_ERR_SHAPE;
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)head_dim);
  return launch_sparse_select(qbar, n_qb, kbar, n_kb, n_heads, head_dim, scale, tau, sel_out,
                              count_out, gini_out, mass_out, (cudaStream_t)stream);
}

wa_status wa_sparse_attn(const void* q, int n_q, const void* k_main, const void* v_main, int n_main,
                         const void* k_loc, const void* v_loc, int n_loc, int block_main,
                         int block_loc, const int32_t* sel, const int32_t* count, wa_dtype dt,
                         int n_heads, int head_dim, float scale, void* o, wa_dtype o_dt,
                         float* lse, wa_stream_t stream) {
  if (!dtype_ok(dt) || !dtype_ok(o_dt)) return WA_ERR_DTYPE;
  if (dt != WA_BF16) return WA_ERR_DTYPE;
  if (!q || !o || !sel || !count || n_q <= 0 || n_main < 0 || n_loc < 0 || n_main + n_loc <= 0)
    return WA_ERR_INVALID_ARG;
  if (n_main > 0 && (!k_main || !v_main)) return WA_ERR_INVALID_ARG;
  if (n_loc > 0 && (!k_loc || !v_loc)) return WA_ERR_INVALID_ARG;
  if (block_main < 1 || block_main > 128 || block_loc < 1 || block_loc > 128) return WA_ERR_SHAPE;
  if ((n_main + (long long)block_main - 1) / block_main +
          (n_loc + (long long)block_loc - 1) / block_loc > 12000)
    return WA_ERR_SHAPE;
  if (head_dim != 128 || n_heads <= 0 || (long long)n_heads * 128 > 16384) return WA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(o) || (n_main > 0 && (!aligned16(k_main) || !aligned16(v_main))) ||
      (n_loc > 0 && (!aligned16(k_loc) || !aligned16(v_loc))))
    return WA_ERR_ALIGN;
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)head_dim);
  SparseBlocks sb;
  sb.sel = sel;
  sb.count = count;
  sb.b_main = block_main;
  sb.b_loc = block_loc;
  sb.stride = (n_main + block_main - 1) / block_main + (n_loc + block_loc - 1) / block_loc;
  return launch_attn_tc(q, n_q, k_main, v_main, n_main, k_loc, v_loc, n_loc, n_heads, scale, o,
                        o_dt == WA_F32, lse, 0, nullptr, nullptr, 0, (cudaStream_t)stream, &sb);
}

wa_status wa_linear_branch(const void* q, int n_q, const void* k_main, const void* v_main,
                           int n_main, const void* k_loc, const void* v_loc, int n_loc,
                           const void* e_k, const void* e_v, int rank, wa_dtype dt, int n_heads,
                           int head_dim, float scale, const float* w_attn, const float* w_lin,
                           int accumulate, void* o, wa_dtype o_dt, wa_stream_t stream) {
  if (!dtype_ok(dt) || !dtype_ok(o_dt)) return WA_ERR_DTYPE;
  if (dt != WA_BF16) return WA_ERR_DTYPE;
  if (!q || !o || !e_k || !e_v || n_q <= 0 || n_main < 0 || n_loc < 0 || n_main + n_loc <= 0)
    return WA_ERR_INVALID_ARG;
  if (n_main > 0 && (!k_main || !v_main)) return WA_ERR_INVALID_ARG;
  if (n_loc > 0 && (!k_loc || !v_loc)) return WA_ERR_INVALID_ARG;
  if (head_dim != 128 || n_heads <= 0 || (long long)n_heads * 128 > 16384) return WA_ERR_SHAPE;
  if (rank <= 0 || rank % 128 != 0 || rank > 512) return WA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(o) || !aligned16(e_k) || !aligned16(e_v) ||
      (n_main > 0 && (!aligned16(k_main) || !aligned16(v_main))) ||
      (n_loc > 0 && (!aligned16(k_loc) || !aligned16(v_loc))))
    return WA_ERR_ALIGN;
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)head_dim);
  return launch_linear_branch(q, n_q, k_main, v_main, n_main, k_loc, v_loc, n_loc, e_k, e_v, rank,
                              n_heads, scale, w_attn, w_lin, accumulate, o, o_dt == WA_F32,
                              (cudaStream_t)stream);
}

wa_status wa_check(wa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return WA_ERR_CUDA;
  Ctrl* ctrl = nullptr;
  wa_status st = get_ctrl(&ctrl);
  if (st != WA_OK) return st;
  int h = 0;
  if (cudaMemcpy(&h, &ctrl->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return WA_ERR_CUDA;
  if (h != 0) {
    int zero = 0;
    if (cudaMemcpy(&ctrl->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return WA_ERR_CUDA;
  }
  if (h & kStatusTimeout) return WA_ERR_TIMEOUT;
  if (h & kStatusIndex) return WA_ERR_INDEX;
  return WA_OK;
}

wa_status wa_set_wait_limit_ns(unsigned long long ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
  return WA_OK;
}

wa_status wa_set_fault(int mode) {
  if (mode < WA_FAULT_NONE || mode > WA_FAULT_WAIT) return WA_ERR_INVALID_ARG;
  g_fault.store(mode, std::memory_order_relaxed);
  return WA_OK;
}

wa_status wa_scratch_bytes(size_t* bytes_out) {
  if (!bytes_out) return WA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return WA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  *bytes_out = g_arena[dev].base ? g_arena[dev].data_bytes : 0;
  return WA_OK;
}

wa_status wa_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  wa_status rc = WA_OK;
  for (int d = 0; d < kMaxDevices; ++d) {
    if (!g_arena[d].base) continue;
    if (cudaSetDevice(d) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) rc = WA_ERR_CUDA;
    cudaFree(g_arena[d].base);
    g_arena[d].base = nullptr;
    g_arena[d].data_bytes = 0;
  }
  cudaSetDevice(cur);
  return rc;
}

}  // extern "C"
