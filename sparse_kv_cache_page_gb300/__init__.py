"""Python binding of libwa (page-retrieval sparse attention on GB300).

Argument marshalling only: each function checks tensor shapes, takes raw
pointers and the current CUDA stream, and calls the C entry point of the same
name in ``lib/libwa.so``.  Every step of the path runs in the library's CUDA
kernels; there is no fallback -- if the library is missing or a call fails,
an exception is raised.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "WaError",
    "lib_path",
    "load",
    "wa_page_summarize",
    "wa_select_pages",
    "wa_gather_pages",
    "wa_select_pages_per_head",
    "wa_gather_pages_per_head",
    "wa_block_attn",
    "wa_gather_attn",
    "wa_linear_branch",
    "wa_block_means",
    "wa_sparse_select",
    "wa_sparse_attn",
    "WaCache",
    "wa_fp8_encode",
    "wa_fp8_decode",
    "wa_gather_pages_fp8",
    "wa_nvfp4_encode",
    "wa_nvfp4_decode",
    "wa_gather_pages_nvfp4",
    "wa_block_means_segments",
    "wa_check",
    "wa_shutdown",
    "wa_version",
    "EXPORTED_SYMBOLS",
]

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

WA_F32, WA_BF16 = 0, 1

# Every symbol include/wa.h declares.
EXPORTED_SYMBOLS = ("wa_strerror", "wa_version", "wa_page_summarize", "wa_select_pages",
                    "wa_select_pages_noalloc", "wa_gather_pages", "wa_block_attn",
                    "wa_gather_attn",
                    "wa_linear_branch", "wa_block_means", "wa_block_means_segments",
                    "wa_sparse_select", "wa_sparse_attn",
                    "wa_select_pages_per_head", "wa_gather_pages_per_head", "wa_cache_create",
                    "wa_cache_destroy", "wa_cache_reset", "wa_cache_append_chunk",
                    "wa_cache_retrieve",
                    "wa_cache_window", "wa_cache_touch", "wa_cache_page_location",
                    "wa_cache_get_stats", "wa_cache_page_slots", "wa_cache_wait_copies",
                    "wa_fp8_encode", "wa_fp8_decode", "wa_nvfp4_encode", "wa_nvfp4_decode",
                    "wa_gather_pages_nvfp4",
                    "wa_gather_pages_fp8", "wa_check", "wa_shutdown", "wa_set_wait_limit_ns",
                    "wa_set_fault", "wa_scratch_bytes")


class _CacheConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_heads", "head_dim", "dtype", "page_tokens",
                                             "pages_per_chunk", "prompt_dim", "hbm_pages",
                                             "host_pages", "max_chunks", "dry_run",
                                             "dram_format")]


class _CacheStats(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int) for n in ("n_pages", "n_chunks", "in_hbm", "in_host")]
                + [(n, ctypes.c_longlong) for n in ("offloads", "promotions", "bytes_h2d",
                                                    "bytes_d2h", "bytes_d2d", "evictions",
                                                    "reclaims")])


class WaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def lib_path() -> str:
    return os.path.join(HERE, "lib", "libwa.so")


def load():
    """Load lib/libwa.so (built by ``build.build()``) and declare signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with sparse_kv_cache_page_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "wa_strerror": (ctypes.c_char_p, [I]),
        "wa_version": (ctypes.c_char_p, []),
        "wa_page_summarize": (I, [P, I, I, I, I, I, P, P]),
        "wa_select_pages": (I, [P, I, I, I, I, P, I, P, P, I, I, I, I, P, P, P, P]),
        "wa_gather_pages": (I, [P, P, I, I, I, I, I, P, P, I, P, P, P]),
        "wa_select_pages_per_head": (I, [P, I, I, I, I, P, I, P, P, I, I, I, I, P, P, P, P]),
        "wa_gather_pages_per_head": (I, [P, P, I, I, I, I, I, P, I, P, P, P]),
        "wa_block_attn": (I, [P, I, P, P, I, P, P, I, I, I, I, F, P, I, P, P]),
        "wa_gather_attn": (I, [P, I, P, P, I, I, P, I, I, P, P, P, P, I, I, I, I, F, P, I, P, P]),
        "wa_linear_branch": (I, [P, I, P, P, I, P, P, I, P, P, I, I, I, I, F, P, P, I, P, I, P]),
        "wa_block_means": (I, [P, I, I, I, I, I, P, P]),
        "wa_block_means_segments": (I, [I, P, P, P, I, I, I, P, P]),
        "wa_sparse_select": (I, [P, I, P, I, I, I, F, P, P, P, P, P, P]),
        "wa_sparse_attn": (I, [P, I, P, P, I, P, P, I, I, I, P, P, I, I, I, F, P, I, P, P]),
        "wa_cache_create": (I, [ctypes.POINTER(_CacheConfig), ctypes.POINTER(P)]),
        "wa_cache_destroy": (I, [P]),
        "wa_cache_reset": (I, [P]),
        "wa_cache_append_chunk": (I, [P, P, P, P, P]),
        "wa_cache_retrieve": (I, [P, P, I, P, I, P, P, P, P]),
        "wa_cache_window": (I, [P, I, P, P, P]),
        "wa_cache_touch": (I, [P, P, I]),
        "wa_cache_page_location": (I, [P, I, ctypes.POINTER(I), ctypes.POINTER(I)]),
        "wa_cache_get_stats": (I, [P, ctypes.POINTER(_CacheStats)]),
        "wa_cache_page_slots": (I, [P, I, ctypes.POINTER(I), ctypes.POINTER(I)]),
        "wa_cache_wait_copies": (I, [P, P]),
        "wa_fp8_encode": (I, [P, I, I, I, P, P, P]),
        "wa_fp8_decode": (I, [P, P, I, I, I, P, P]),
        "wa_gather_pages_fp8": (I, [P, P, I, I, I, I, P, I, P, P]),
        "wa_nvfp4_encode": (I, [P, I, I, I, P, P, P, P]),
        "wa_nvfp4_decode": (I, [P, P, P, I, I, I, P, P]),
        "wa_gather_pages_nvfp4": (I, [P, P, P, I, I, I, I, P, I, P, P]),
        "wa_check": (I, [P]),
        "wa_shutdown": (I, []),
        "wa_set_wait_limit_ns": (I, [ctypes.c_ulonglong]),
        "wa_set_fault": (I, [I]),
        "wa_scratch_bytes": (I, [ctypes.POINTER(ctypes.c_size_t)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return WA_BF16
    if t.dtype == torch.float32:
        return WA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ok(fn: str, st: int):
    if st != 0:
        raise WaError(fn, st, load().wa_strerror(st).decode())


def _need(cond: bool, what: str):
    if not cond:
        raise ValueError(what)


def _buf(t, dtype, numel: int, what: str):
    """A buffer the library reads or writes through a plain pointer: present,
    contiguous, of `dtype` and exactly `numel` elements (the C ABI cannot see
    sizes, so a short buffer would be overrun)."""
    _need(t is not None and t.is_contiguous() and t.dtype == dtype and t.numel() == numel,
          f"{what} must be contiguous {dtype} with {numel} elements")


def wa_version() -> str:
    return load().wa_version().decode()


def wa_page_summarize(k_pages: torch.Tensor, kbar_out: torch.Tensor, stream=None):
    """kbar_out[j,h,:] = mean_t k_pages[j,t,h,:]; k_pages [n_pages][P][H][d]."""
    _need(k_pages.dim() == 4 and k_pages.is_contiguous(), "k_pages must be contiguous [n][P][H][d]")
    n, p, h, d = k_pages.shape
    _need(kbar_out.shape == (n, h, d) and kbar_out.dtype == torch.float32
          and kbar_out.is_contiguous(), "kbar_out must be float32 [n][H][d]")
    _ok("wa_page_summarize", load().wa_page_summarize(_ptr(k_pages), _dt(k_pages), n, p, h, d,
                                                      _ptr(kbar_out), _stream(stream)))


def wa_select_pages(q: torch.Tensor, kbar: torch.Tensor, prompt_cur, prompt_chunks,
                    pages_per_chunk: int, k_p: int, idx_out: torch.Tensor,
                    scores_out=None, chunk_out=None, stream=None):
    """Prompt-stage top-1 chunk (skipped when prompt_chunks is None) and
    page-stage top-k_p; writes ascending page indices to idx_out (int32)."""
    _need(q.dim() == 3 and q.is_contiguous(), "q must be contiguous [n_q][H][d]")
    n_q, h, d = q.shape
    _need(kbar.dim() == 3 and kbar.shape[1:] == (h, d) and kbar.dtype == torch.float32,
          "kbar must be float32 [n_pages][H][d]")
    _need(idx_out.dtype == torch.int32 and idx_out.numel() >= k_p, "idx_out must be int32 [k_p]")
    n_chunks, pdim = 0, 0
    if prompt_chunks is not None:
        n_chunks, pdim = prompt_chunks.shape
        _need(prompt_cur is not None and prompt_cur.numel() == pdim
              and prompt_chunks.dtype == torch.float32 and prompt_cur.dtype == torch.float32,
              "prompt embeddings must be float32")
    _ok("wa_select_pages", load().wa_select_pages(
        _ptr(q), _dt(q), n_q, h, d, _ptr(kbar), kbar.shape[0], _ptr(prompt_cur),
        _ptr(prompt_chunks), n_chunks, pdim, pages_per_chunk, k_p, _ptr(idx_out),
        _ptr(scores_out), _ptr(chunk_out), _stream(stream)))


def wa_gather_pages(k_pages: torch.Tensor, v_pages, idx_dev, idx_host, k_buf: torch.Tensor,
                    v_buf, stream=None):
    """k_buf[s*P + t] = k_pages[idx[s]][t] (likewise v).  Device pages use
    idx_dev (device int32); pinned host pages use idx_host (host int32)."""
    _need(k_pages.dim() == 4 and k_pages.is_contiguous(), "k_pages must be contiguous [n][P][H][d]")
    n, p, h, d = k_pages.shape
    k_p = (idx_dev if idx_dev is not None else idx_host).numel()
    _buf(k_buf, k_pages.dtype, k_p * p * h * d, "k_buf")
    _need((v_pages is None) == (v_buf is None), "v_pages and v_buf go together")
    if v_pages is not None:
        _buf(v_pages, k_pages.dtype, k_pages.numel(), "v_pages")
        _buf(v_buf, k_pages.dtype, k_p * p * h * d, "v_buf")
    idx = idx_dev if idx_dev is not None else idx_host
    _need(idx.dtype == torch.int32 and idx.is_contiguous(), "page indices must be contiguous int32")
    _ok("wa_gather_pages", load().wa_gather_pages(
        _ptr(k_pages), _ptr(v_pages), _dt(k_pages), n, p, h, d, _ptr(idx_dev), _ptr(idx_host),
        k_p, _ptr(k_buf), _ptr(v_buf), _stream(stream)))


def wa_select_pages_per_head(q: torch.Tensor, kbar: torch.Tensor, prompt_cur, prompt_chunks,
                             pages_per_chunk: int, k_p: int, idx_out: torch.Tensor,
                             scores_out=None, chunk_out=None, stream=None):
    """Prompt-stage top-1 chunk, then a top-k_p page set per head (scored on
    that head's slice); idx_out int32 [H][k_p], ascending per head."""
    _need(q.dim() == 3 and q.is_contiguous(), "q must be contiguous [n_q][H][d]")
    n_q, h, d = q.shape
    _need(kbar.dim() == 3 and kbar.shape[1:] == (h, d) and kbar.dtype == torch.float32,
          "kbar must be float32 [n_pages][H][d]")
    _need(idx_out.dtype == torch.int32 and idx_out.numel() >= h * k_p,
          "idx_out must be int32 [H][k_p]")
    n_chunks, pdim = 0, 0
    if prompt_chunks is not None:
        n_chunks, pdim = prompt_chunks.shape
        _need(prompt_cur is not None and prompt_cur.numel() == pdim
              and prompt_chunks.dtype == torch.float32 and prompt_cur.dtype == torch.float32,
              "prompt embeddings must be float32")
    _ok("wa_select_pages_per_head", load().wa_select_pages_per_head(
        _ptr(q), _dt(q), n_q, h, d, _ptr(kbar), kbar.shape[0], _ptr(prompt_cur),
        _ptr(prompt_chunks), n_chunks, pdim, pages_per_chunk, k_p, _ptr(idx_out),
        _ptr(scores_out), _ptr(chunk_out), _stream(stream)))


def wa_gather_pages_per_head(k_pages: torch.Tensor, v_pages, idx_dev: torch.Tensor,
                             k_buf: torch.Tensor, v_buf, stream=None):
    """k_buf[s*P + t][h] = k_pages[idx_dev[h][s]][t][h] (likewise v); device pages."""
    _need(k_pages.dim() == 4 and k_pages.is_contiguous(), "k_pages must be contiguous [n][P][H][d]")
    n, p, h, d = k_pages.shape
    _need(idx_dev.dim() == 2 and idx_dev.shape[0] == h and idx_dev.dtype == torch.int32,
          "idx_dev must be int32 [H][k_p]")
    k_p = idx_dev.shape[1]
    _need(idx_dev.is_contiguous(), "idx_dev must be contiguous")
    _buf(k_buf, k_pages.dtype, k_p * p * h * d, "k_buf")
    _need((v_pages is None) == (v_buf is None), "v_pages and v_buf go together")
    if v_pages is not None:
        _buf(v_pages, k_pages.dtype, k_pages.numel(), "v_pages")
        _buf(v_buf, k_pages.dtype, k_p * p * h * d, "v_buf")
    _ok("wa_gather_pages_per_head", load().wa_gather_pages_per_head(
        _ptr(k_pages), _ptr(v_pages), _dt(k_pages), n, p, h, d, _ptr(idx_dev), k_p, _ptr(k_buf),
        _ptr(v_buf), _stream(stream)))


def _rows(t):
    return 0 if t is None else t.shape[0]


def _kv_pair(k, v, h: int, d: int, dtype, what: str):
    """Keys and values of one segment: both absent, or both contiguous
    [rows][H][d] of `dtype` with the same row count."""
    _need((k is None) == (v is None), f"{what}: keys and values go together")
    if k is not None:
        _need(k.dim() == 3 and k.shape[1:] == (h, d) and v.shape == k.shape,
              f"{what}: keys and values must be [rows][H][d] with the same rows")
        _buf(k, dtype, k.numel(), f"{what} keys")
        _buf(v, dtype, v.numel(), f"{what} values")


def wa_block_attn(q: torch.Tensor, k_main, v_main, k_loc, v_loc, o: torch.Tensor, lse=None,
                  scale: float = 0.0, stream=None):
    """o = softmax(q [k_main; k_loc]^T * scale) [v_main; v_loc]; lse [H][n_q] optional.
    o may be float32 (the fp32 result) or the input dtype."""
    _need(q.dim() == 3 and q.is_contiguous() and o.shape == q.shape and o.is_contiguous(),
          "q and o must be contiguous [n_q][H][d]")
    n_q, h, d = q.shape
    _need(o.dtype in (torch.float32, q.dtype), "o must be float32 or the input dtype")
    _kv_pair(k_main, v_main, h, d, q.dtype, "main segment")
    _kv_pair(k_loc, v_loc, h, d, q.dtype, "local segment")
    if lse is not None:
        _buf(lse, torch.float32, h * n_q, "lse")
    _ok("wa_block_attn", load().wa_block_attn(
        _ptr(q), n_q, _ptr(k_main), _ptr(v_main), _rows(k_main), _ptr(k_loc), _ptr(v_loc),
        _rows(k_loc), _dt(q), h, d, float(scale), _ptr(o), _dt(o), _ptr(lse), _stream(stream)))


def wa_gather_attn(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                   idx_dev: torch.Tensor, k_loc, v_loc, o: torch.Tensor, k_buf=None, v_buf=None,
                   lse=None, scale: float = 0.0, stream=None):
    """Gather and attention in one launch: k_buf[s*P + t] = k_pages[idx[s]][t]
    (idx int32 [k_p]; or [H][k_p], a page set per head), likewise v, and o as
    wa_block_attn over [k_buf; k_loc], [v_buf; v_loc].  k_buf/v_buf may be None
    (attention only)."""
    _need(q.dim() == 3 and q.is_contiguous() and o.shape == q.shape and o.is_contiguous(),
          "q and o must be contiguous [n_q][H][d]")
    n_q, h, d = q.shape
    _need(o.dtype in (torch.float32, q.dtype), "o must be float32 or the input dtype")
    _need(k_pages.dim() == 4 and k_pages.shape[2:] == (h, d) and v_pages.shape == k_pages.shape,
          "k_pages, v_pages must be [n_pages][P][H][d]")
    n, p = k_pages.shape[:2]
    _buf(k_pages, q.dtype, k_pages.numel(), "k_pages")
    _buf(v_pages, q.dtype, v_pages.numel(), "v_pages")
    _need(idx_dev.dtype == torch.int32 and idx_dev.is_contiguous() and idx_dev.dim() in (1, 2),
          "idx_dev must be contiguous int32 [k_p] or [H][k_p]")
    per_head = idx_dev.dim() == 2
    _need(not per_head or idx_dev.shape[0] == h, "a page set per head needs idx_dev [H][k_p]")
    k_p = idx_dev.shape[-1]
    _need((k_buf is None) == (v_buf is None), "k_buf and v_buf go together")
    if k_buf is not None:
        _buf(k_buf, q.dtype, k_p * p * h * d, "k_buf")
        _buf(v_buf, q.dtype, k_p * p * h * d, "v_buf")
    _kv_pair(k_loc, v_loc, h, d, q.dtype, "local segment")
    if lse is not None:
        _buf(lse, torch.float32, h * n_q, "lse")
    _ok("wa_gather_attn", load().wa_gather_attn(
        _ptr(q), n_q, _ptr(k_pages), _ptr(v_pages), n, p, _ptr(idx_dev), k_p, int(per_head),
        _ptr(k_buf), _ptr(v_buf), _ptr(k_loc), _ptr(v_loc), _rows(k_loc), _dt(q), h, d,
        float(scale), _ptr(o), _dt(o), _ptr(lse), _stream(stream)))


def wa_linear_branch(q: torch.Tensor, k_main, v_main, k_loc, v_loc, e_k: torch.Tensor,
                     e_v: torch.Tensor, o: torch.Tensor, w_attn=None, w_lin=None,
                     accumulate: bool = True, scale: float = 0.0, stream=None):
    """Linformer branch; o = w_attn*o + w_lin*O_lin (accumulate) or o = O_lin."""
    _need(q.dim() == 3 and q.is_contiguous() and o.shape == q.shape and o.is_contiguous(),
          "q and o must be contiguous [n_q][H][d]")
    n_q, h, d = q.shape
    _need(o.dtype in (torch.float32, q.dtype), "o must be float32 or the input dtype")
    _kv_pair(k_main, v_main, h, d, q.dtype, "main segment")
    _kv_pair(k_loc, v_loc, h, d, q.dtype, "local segment")
    _need(e_k.dim() == 3 and e_k.shape[:2] == (h, _rows(k_main) + _rows(k_loc))
          and e_v.shape == e_k.shape, "e_k, e_v must be [H][n_main + n_loc][rank]")
    rank = e_k.shape[-1]
    _buf(e_k, q.dtype, e_k.numel(), "e_k")
    _buf(e_v, q.dtype, e_v.numel(), "e_v")
    for w, name in ((w_attn, "w_attn"), (w_lin, "w_lin")):
        if w is not None:
            _buf(w, torch.float32, h, name)
    _ok("wa_linear_branch", load().wa_linear_branch(
        _ptr(q), n_q, _ptr(k_main), _ptr(v_main), _rows(k_main), _ptr(k_loc), _ptr(v_loc),
        _rows(k_loc), _ptr(e_k), _ptr(e_v), rank, _dt(q), h, d, float(scale), _ptr(w_attn),
        _ptr(w_lin), int(bool(accumulate)), _ptr(o), _dt(o), _stream(stream)))


def wa_block_means(x: torch.Tensor, block: int, means_out: torch.Tensor, stream=None):
    """means_out[b,h,:] = mean of x rows [b*block, min((b+1)*block, n)) (ragged last block)."""
    _need(x.dim() == 3 and x.is_contiguous(), "x must be contiguous [n][H][d]")
    n, h, d = x.shape
    nb = (n + block - 1) // block
    _need(means_out.shape == (nb, h, d) and means_out.dtype == torch.float32
          and means_out.is_contiguous(), "means_out must be float32 [ceil(n/block)][H][d]")
    _ok("wa_block_means", load().wa_block_means(_ptr(x), _dt(x), n, int(block), h, d,
                                                _ptr(means_out), _stream(stream)))


def wa_block_means_segments(segments, stream=None):
    """Block means of up to three row sets in one launch: segments is a list of
    (x [n][H][d], block, means_out float32 [ceil(n/block)][H][d]); every set's
    means equal wa_block_means on that set alone, bit for bit."""
    _need(1 <= len(segments) <= 3, "one to three segments")
    x0 = segments[0][0]
    _need(x0.dim() == 3, "x must be [n][H][d]")
    h, d = x0.shape[1:]
    for x, block, out in segments:
        _need(x.dim() == 3 and x.shape[1:] == (h, d) and x.dtype == x0.dtype and x.is_contiguous(),
              "every x must be contiguous [n][H][d] with the same H, d and dtype")
        _need(int(block) > 0, "block must be positive")
        nb = (x.shape[0] + int(block) - 1) // int(block)
        _buf(out, torch.float32, nb * h * d, "means_out")
    n = len(segments)
    xs = (ctypes.c_void_p * n)(*[x.data_ptr() for x, _, _ in segments])
    rows = (ctypes.c_int * n)(*[x.shape[0] for x, _, _ in segments])
    blocks = (ctypes.c_int * n)(*[int(b) for _, b, _ in segments])
    outs = (ctypes.c_void_p * n)(*[o.data_ptr() for _, _, o in segments])
    _ok("wa_block_means_segments", load().wa_block_means_segments(
        n, xs, rows, blocks, _dt(x0), h, d, outs, _stream(stream)))


def wa_sparse_select(qbar: torch.Tensor, kbar: torch.Tensor, sel_out: torch.Tensor,
                     count_out: torch.Tensor, tau=None, gini_out=None, mass_out=None,
                     scale: float = 0.0, stream=None):
    """HSA block selection: per head, the fewest key blocks (by pooled mass)
    whose cumulative mass reaches tau_h (= 1 - Gini when tau is None)."""
    _need(qbar.dim() == 3 and kbar.dim() == 3 and qbar.dtype == torch.float32
          and kbar.dtype == torch.float32 and qbar.is_contiguous() and kbar.is_contiguous(),
          "qbar/kbar must be contiguous float32 [n][H][d]")
    n_qb, h, d = qbar.shape
    n_kb = kbar.shape[0]
    _need(sel_out.shape == (h, n_kb) and sel_out.dtype == torch.int32 and count_out.numel() == h
          and count_out.dtype == torch.int32, "sel_out int32 [H][n_kb], count_out int32 [H]")
    _ok("wa_sparse_select", load().wa_sparse_select(
        _ptr(qbar), n_qb, _ptr(kbar), n_kb, h, d, float(scale), _ptr(tau), _ptr(sel_out),
        _ptr(count_out), _ptr(gini_out), _ptr(mass_out), _stream(stream)))


def wa_sparse_attn(q: torch.Tensor, k_main, v_main, k_loc, v_loc, sel: torch.Tensor,
                   count: torch.Tensor, o: torch.Tensor, block_main: int = 128,
                   block_loc: int = 64, lse=None, scale: float = 0.0, stream=None):
    """Attention restricted, per head, to the kept key blocks sel[h][:count[h]]."""
    _need(q.dim() == 3 and q.is_contiguous() and o.shape == q.shape and o.is_contiguous(),
          "q and o must be contiguous [n_q][H][d]")
    n_q, h, d = q.shape
    _ok("wa_sparse_attn", load().wa_sparse_attn(
        _ptr(q), n_q, _ptr(k_main), _ptr(v_main), _rows(k_main), _ptr(k_loc), _ptr(v_loc),
        _rows(k_loc), int(block_main), int(block_loc), _ptr(sel), _ptr(count), _dt(q), h, d,
        float(scale), _ptr(o), _dt(o), _ptr(lse), _stream(stream)))


def wa_fp8_encode(x: torch.Tensor, codes_out: torch.Tensor, scales_out: torch.Tensor, stream=None):
    """FP8 E4M3 codes and per-(token, head) scales of a bf16 [n][H][d] tensor;
    codes uint8 [n][H][d] and scales float32 [n][H] on the device or pinned."""
    _need(x.dim() == 3, "x must be [n][H][d]")
    n, h, d = x.shape
    _buf(x, torch.bfloat16, n * h * d, "x")
    _buf(codes_out, torch.uint8, n * h * d, "codes_out")
    _buf(scales_out, torch.float32, n * h, "scales_out")
    _ok("wa_fp8_encode", load().wa_fp8_encode(_ptr(x), n, h, d, _ptr(codes_out), _ptr(scales_out),
                                              _stream(stream)))


def wa_fp8_decode(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None):
    """out bf16 [n][H][d] = decode(codes uint8 [n][H][d], scales float32 [n][H])."""
    _need(out.dim() == 3, "out must be [n][H][d]")
    n, h, d = out.shape
    _buf(out, torch.bfloat16, n * h * d, "out")
    _buf(codes, torch.uint8, n * h * d, "codes")
    _buf(scales, torch.float32, n * h, "scales")
    _ok("wa_fp8_decode", load().wa_fp8_decode(_ptr(codes), _ptr(scales), n, h, d, _ptr(out),
                                              _stream(stream)))


def wa_gather_pages_fp8(code_pages: torch.Tensor, scale_pages: torch.Tensor, idx_dev: torch.Tensor,
                        buf_out: torch.Tensor, stream=None):
    """buf_out[s*P + t] = decode(code_pages[idx[s]][t]) (bf16); pages on the
    device or in pinned host memory."""
    _need(code_pages.dim() == 4, "code_pages must be [n][P][H][d]")
    n, p, h, d = code_pages.shape
    _buf(code_pages, torch.uint8, n * p * h * d, "code_pages")
    _buf(scale_pages, torch.float32, n * p * h, "scale_pages")
    _need(idx_dev.dtype == torch.int32 and idx_dev.is_contiguous(), "idx_dev must be contiguous int32")
    _buf(buf_out, torch.bfloat16, idx_dev.numel() * p * h * d, "buf_out")
    _ok("wa_gather_pages_fp8", load().wa_gather_pages_fp8(
        _ptr(code_pages), _ptr(scale_pages), n, p, h, d, _ptr(idx_dev), idx_dev.numel(),
        _ptr(buf_out), _stream(stream)))


def wa_nvfp4_encode(x: torch.Tensor, codes_out: torch.Tensor, bscales_out: torch.Tensor,
                    rscales_out: torch.Tensor, stream=None):
    """NVFP4 form of a bf16 [n][H][d] tensor: E2M1 codes uint8 [n][H][d/2], E4M3
    block scales uint8 [n][H][d/16], fp32 row scales [n][H]; on the device or pinned."""
    _need(x.dim() == 3 and x.shape[2] % 16 == 0, "x must be [n][H][d], d a multiple of 16")
    n, h, d = x.shape
    _buf(x, torch.bfloat16, n * h * d, "x")
    _buf(codes_out, torch.uint8, n * h * d // 2, "codes_out")
    _buf(bscales_out, torch.uint8, n * h * d // 16, "bscales_out")
    _buf(rscales_out, torch.float32, n * h, "rscales_out")
    _ok("wa_nvfp4_encode", load().wa_nvfp4_encode(_ptr(x), n, h, d, _ptr(codes_out),
                                                  _ptr(bscales_out), _ptr(rscales_out),
                                                  _stream(stream)))


def wa_nvfp4_decode(codes: torch.Tensor, bscales: torch.Tensor, rscales: torch.Tensor,
                    out: torch.Tensor, stream=None):
    """out bf16 [n][H][d] = decode of the NVFP4 form (codes, block scales, row scales)."""
    _need(out.dim() == 3 and out.shape[2] % 16 == 0, "out must be [n][H][d], d a multiple of 16")
    n, h, d = out.shape
    _buf(out, torch.bfloat16, n * h * d, "out")
    _buf(codes, torch.uint8, n * h * d // 2, "codes")
    _buf(bscales, torch.uint8, n * h * d // 16, "bscales")
    _buf(rscales, torch.float32, n * h, "rscales")
    _ok("wa_nvfp4_decode", load().wa_nvfp4_decode(_ptr(codes), _ptr(bscales), _ptr(rscales), n, h,
                                                  d, _ptr(out), _stream(stream)))


def wa_gather_pages_nvfp4(code_pages: torch.Tensor, bscale_pages: torch.Tensor,
                          rscale_pages: torch.Tensor, idx_dev: torch.Tensor, buf_out: torch.Tensor,
                          stream=None):
    """buf_out[s*P + t] = decode of page idx[s], token t (bf16); code pages
    [n][P][H][d/2], block scales [n][P][H][d/16], row scales [n][P][H], on the
    device or in pinned host memory."""
    _need(code_pages.dim() == 4, "code_pages must be [n][P][H][d/2]")
    n, p, h, half = code_pages.shape
    d = 2 * half
    _need(d % 16 == 0, "d must be a multiple of 16")
    _buf(code_pages, torch.uint8, n * p * h * half, "code_pages")
    _buf(bscale_pages, torch.uint8, n * p * h * (d // 16), "bscale_pages")
    _buf(rscale_pages, torch.float32, n * p * h, "rscale_pages")
    _need(idx_dev.dtype == torch.int32 and idx_dev.is_contiguous(), "idx_dev must be contiguous int32")
    _buf(buf_out, torch.bfloat16, idx_dev.numel() * p * h * d, "buf_out")
    _ok("wa_gather_pages_nvfp4", load().wa_gather_pages_nvfp4(
        _ptr(code_pages), _ptr(bscale_pages), _ptr(rscale_pages), n, p, h, 2 * half,
        _ptr(idx_dev), idx_dev.numel(), _ptr(buf_out), _stream(stream)))


class WaCache:
    """KV cache manager (libwa wa_cache_*): HBM and inclusive pinned-DRAM page
    tiers (optionally FP8 or NVFP4 in DRAM), summaries at insert, retrieval with LRU
    eviction, overlapped offloads and promotion, window access.  ``dry_run``
    caches plan placements without any CUDA work."""

    def __init__(self, n_heads: int, head_dim: int, page_tokens: int, pages_per_chunk: int,
                 hbm_pages: int, host_pages: int, max_chunks: int, prompt_dim: int = 0,
                 dtype=torch.bfloat16, dry_run: bool = False, dram_format: str = "native"):
        """dram_format: "native" (the cache's dtype), "fp8" or "nvfp4"."""
        fmt = {"native": 0, "bf16": 0, "fp8": 1, "nvfp4": 2}.get(dram_format)
        _need(fmt is not None, "dram_format must be 'native', 'fp8' or 'nvfp4'")
        cfg = _CacheConfig(n_heads, head_dim, WA_BF16 if dtype == torch.bfloat16 else WA_F32,
                           page_tokens, pages_per_chunk, prompt_dim, hbm_pages, host_pages,
                           max_chunks, int(bool(dry_run)), fmt)
        h = ctypes.c_void_p()
        _ok("wa_cache_create", load().wa_cache_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h
        self.cfg = cfg

    def close(self):
        if self._h:
            _ok("wa_cache_destroy", load().wa_cache_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:   # interpreter shutdown
            pass

    def reset(self):
        """Empty the cache for a new sequence; the tiers' memory is kept."""
        _ok("wa_cache_reset", load().wa_cache_reset(self._h))

    def append(self, k, v, prompt=None, stream=None):
        _ok("wa_cache_append_chunk", load().wa_cache_append_chunk(
            self._h, _ptr(k), _ptr(v), _ptr(prompt),
            None if self.cfg.dry_run else _stream(stream)))

    def retrieve(self, q: torch.Tensor, prompt_cur, k_p: int, k_buf: torch.Tensor,
                 v_buf: torch.Tensor, stream=None):
        """Indices (ascending) of the k_p pages copied into k_buf / v_buf."""
        idx = (ctypes.c_int32 * k_p)()
        _ok("wa_cache_retrieve", load().wa_cache_retrieve(
            self._h, _ptr(q), q.shape[0], _ptr(prompt_cur), k_p, _ptr(k_buf), _ptr(v_buf),
            ctypes.cast(idx, ctypes.c_void_p), _stream(stream)))
        return list(idx)

    def window(self, n_tokens: int, k_out: torch.Tensor, v_out: torch.Tensor, stream=None):
        _ok("wa_cache_window", load().wa_cache_window(self._h, n_tokens, _ptr(k_out), _ptr(v_out),
                                                      _stream(stream)))

    def touch(self, pages):
        arr = (ctypes.c_int32 * len(pages))(*pages)
        _ok("wa_cache_touch", load().wa_cache_touch(self._h, ctypes.cast(arr, ctypes.c_void_p),
                                                    len(pages)))

    def location(self, page: int):
        t, s = ctypes.c_int(), ctypes.c_int()
        _ok("wa_cache_page_location", load().wa_cache_page_location(
            self._h, page, ctypes.byref(t), ctypes.byref(s)))
        return t.value, s.value

    def slots(self, page: int):
        """(HBM slot, DRAM slot) of a page, -1 where it has no copy."""
        h, x = ctypes.c_int(), ctypes.c_int()
        _ok("wa_cache_page_slots", load().wa_cache_page_slots(
            self._h, page, ctypes.byref(h), ctypes.byref(x)))
        return h.value, x.value

    def wait_copies(self, stream=None):
        """Make the stream wait for every offload copy issued so far."""
        _ok("wa_cache_wait_copies", load().wa_cache_wait_copies(
            self._h, None if self.cfg.dry_run else _stream(stream)))

    def stats(self) -> dict:
        st = _CacheStats()
        _ok("wa_cache_get_stats", load().wa_cache_get_stats(self._h, ctypes.byref(st)))
        return {n: getattr(st, n) for n, _ in _CacheStats._fields_}


def wa_check(stream=None):
    """Synchronize the stream and raise if a kernel recorded an error."""
    _ok("wa_check", load().wa_check(_stream(stream)))


def wa_shutdown():
    _ok("wa_shutdown", load().wa_shutdown())


# Fault-injection modes of wa_set_fault (host side; none faults a GPU).
WA_FAULT_NONE, WA_FAULT_ALLOC, WA_FAULT_COPY, WA_FAULT_WAIT = 0, 1, 2, 3


def wa_set_wait_limit_ns(ns: int):
    """Limit of each bounded device wait for later launches (0 = the 4 s default)."""
    _ok("wa_set_wait_limit_ns", load().wa_set_wait_limit_ns(int(ns)))


def wa_set_fault(mode: int):
    """Process-wide host-side fault injection (WA_FAULT_* above)."""
    _ok("wa_set_fault", load().wa_set_fault(int(mode)))


def wa_scratch_bytes() -> int:
    """Bytes of the current device's scratch arena (0 if none is allocated)."""
    n = ctypes.c_size_t(0)
    _ok("wa_scratch_bytes", load().wa_scratch_bytes(ctypes.byref(n)))
    return int(n.value)
