"""Thin ctypes binding of libbsa (include/bsa.h).

Argument marshalling only: every step of the attention runs in the CUDA
library. Tensor arguments may be torch tensors (their data pointers are
passed), raw integer addresses, or None for the optional outputs. The
library must have been built (``dynamic_block_sparse_causal_gb300.build``);
importing the binding without it raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

BSA_BF16 = 0
BSA_FP8_E4M3 = 1

STATUS = {
    0: "BSA_OK", 1: "BSA_ERR_INVALID_ARG", 2: "BSA_ERR_UNSUPPORTED", 3: "BSA_ERR_CUDA",
    4: "BSA_ERR_TIMEOUT", 5: "BSA_ERR_NO_MEMORY", 6: "BSA_ERR_BAD_SEQLENS",
}

_lib = None


class BsaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """Load libbsa.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libbsa.so is missing ({LIB_PATH}); build it first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    L.bsa_prefill_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp, vp]
    L.bsa_prefill_fwd.restype = i32
    L.bsa_prefill_fwd_chunked.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                          vp, vp, vp, vp]
    L.bsa_prefill_fwd_chunked.restype = i32
    L.bsa_prefill_fwd_paged.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, i32, i32, i32, i32, i32,
                                        f32, i32, vp, vp, vp, vp]
    L.bsa_prefill_fwd_paged.restype = i32
    L.bsa_skip_bitmap_words_chunked.argtypes = [ctypes.POINTER(ctypes.c_int32),
                                                ctypes.POINTER(ctypes.c_int32), i32, i32]
    L.bsa_skip_bitmap_words_chunked.restype = i64
    L.bsa_prefill_fwd_noalloc.argtypes = L.bsa_prefill_fwd.argtypes
    L.bsa_prefill_fwd_noalloc.restype = i32
    L.bsa_set_fp8_scales.argtypes = [vp, vp, vp]
    L.bsa_set_fp8_scales.restype = i32
    L.bsa_quantize_fp8.argtypes = [vp, i64, i32, i32, vp, vp, vp]
    L.bsa_quantize_fp8.restype = i32
    L.bsa_skip_bitmap_words.argtypes = [ctypes.POINTER(ctypes.c_int32), i32, i32]
    L.bsa_skip_bitmap_words.restype = i64
    L.bsa_get_device_status.argtypes = [vp]
    L.bsa_get_device_status.restype = i32
    L.bsa_status_string.argtypes = [i32]
    L.bsa_status_string.restype = ctypes.c_char_p
    L.bsa_version.argtypes = []
    L.bsa_version.restype = i32
    L.bsa_release.argtypes = []
    L.bsa_release.restype = None
    L.bsa_release_stream.argtypes = [vp]
    L.bsa_release_stream.restype = i32
    L.bsa_get_noalloc_status.argtypes = [vp]
    L.bsa_get_noalloc_status.restype = i32
    L.bsa_debug_fault_drill.argtypes = [i32, i64]
    L.bsa_debug_fault_drill.restype = i32
    L.bsa_decode_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, i32, f32, vp,
                                 vp, vp, vp]
    L.bsa_decode_fwd.restype = i32
    L.bsa_block_importance.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i64, vp, vp, vp]
    L.bsa_block_importance.restype = i32
    L.bsa_top_p_select.argtypes = [vp, vp, i32, i64, f32, vp, vp, vp, vp]
    L.bsa_top_p_select.restype = i32
    L.bsa_importance_blocks.argtypes = [ctypes.POINTER(ctypes.c_int32), i32]
    L.bsa_importance_blocks.restype = i64
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def prefill_fwd(q, k, v, cu_seqlens, n_seqs, Hq, Hkv, d, causal, lam, dtype, out, lse,
                skip_bitmap, stream=None) -> int:
    """bsa_prefill_fwd; returns the status code."""
    return lib().bsa_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(n_seqs),
                                 int(Hq), int(Hkv), int(d), int(causal), float(lam), int(dtype),
                                 _ptr(out), _ptr(lse), _ptr(skip_bitmap), _stream(stream))


def prefill_fwd_chunked(q, k, v, cu_seqlens_q, cu_seqlens_k, n_seqs, Hq, Hkv, d, causal, lam,
                        dtype, out, lse, skip_bitmap, stream=None) -> int:
    """bsa_prefill_fwd_chunked: queries are the last positions of their sequence."""
    return lib().bsa_prefill_fwd_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q),
                                         _ptr(cu_seqlens_k), int(n_seqs), int(Hq), int(Hkv),
                                         int(d), int(causal), float(lam), int(dtype), _ptr(out),
                                         _ptr(lse), _ptr(skip_bitmap), _stream(stream))


def prefill_fwd_paged(q, k_cache, v_cache, page_table, max_pages_per_seq, num_pages, cu_seqlens_q,
                      cu_seqlens_k, n_seqs, Hq, Hkv, d, causal, lam, dtype, out, lse, skip_bitmap,
                      stream=None) -> int:
    """bsa_prefill_fwd_paged: keys/values from 128-token pages via a page table."""
    return lib().bsa_prefill_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                       int(max_pages_per_seq), int(num_pages), _ptr(cu_seqlens_q),
                                       _ptr(cu_seqlens_k), int(n_seqs), int(Hq), int(Hkv), int(d),
                                       int(causal), float(lam), int(dtype), _ptr(out), _ptr(lse),
                                       _ptr(skip_bitmap), _stream(stream))


def prefill_fwd_noalloc(q, k, v, cu_seqlens, n_seqs, Hq, Hkv, d, causal, lam, dtype, out, lse,
                        skip_bitmap, stream=None) -> int:
    """bsa_prefill_fwd_noalloc: same call, scratch from a fixed array in the
    library instead of an allocation (for callers that may not allocate)."""
    return lib().bsa_prefill_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(n_seqs),
                                         int(Hq), int(Hkv), int(d), int(causal), float(lam),
                                         int(dtype), _ptr(out), _ptr(lse), _ptr(skip_bitmap),
                                         _stream(stream))


def set_fp8_scales(q_scale, k_scale, v_scale) -> int:
    return lib().bsa_set_fp8_scales(_ptr(q_scale), _ptr(k_scale), _ptr(v_scale))


def quantize_fp8(x, tokens, H, d, x_e4m3, scale, stream=None) -> int:
    return lib().bsa_quantize_fp8(_ptr(x), int(tokens), int(H), int(d), _ptr(x_e4m3),
                                  _ptr(scale), _stream(stream))


def skip_bitmap_words(cu_seqlens_host, Hq) -> int:
    import numpy as np
    cu = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
    return lib().bsa_skip_bitmap_words(cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       int(cu.shape[0] - 1), int(Hq))


def skip_bitmap_words_chunked(cu_seqlens_q_host, cu_seqlens_k_host, Hq) -> int:
    import numpy as np
    cq = np.ascontiguousarray(cu_seqlens_q_host, dtype=np.int32)
    ck = np.ascontiguousarray(cu_seqlens_k_host, dtype=np.int32)
    if cq.shape != ck.shape:
        return -1
    P = ctypes.POINTER(ctypes.c_int32)
    return lib().bsa_skip_bitmap_words_chunked(cq.ctypes.data_as(P), ck.ctypes.data_as(P),
                                               int(cq.shape[0] - 1), int(Hq))


def decode_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, n_seqs, max_seqlen_q, total_k, Hq, Hkv, d,
               causal, lam, out, lse, skip_bitmap, stream=None) -> int:
    """bsa_decode_fwd: a few new queries per sequence against all earlier keys (split-KV)."""
    return lib().bsa_decode_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                int(n_seqs), int(max_seqlen_q), int(total_k), int(Hq), int(Hkv),
                                int(d), int(causal), float(lam), _ptr(out), _ptr(lse),
                                _ptr(skip_bitmap), _stream(stream))


def block_importance(q, k, cu_seqlens, n_seqs, Hq, Hkv, d, n_window, causal, total_blocks,
                     scores, mean_scores, stream=None) -> int:
    """bsa_block_importance: per-head block scores of the last n_window queries."""
    return lib().bsa_block_importance(_ptr(q), _ptr(k), _ptr(cu_seqlens), int(n_seqs), int(Hq),
                                      int(Hkv), int(d), int(n_window), int(causal),
                                      int(total_blocks), _ptr(scores), _ptr(mean_scores),
                                      _stream(stream))


def top_p_select(scores, cu_seqlens, n_seqs, total_blocks, p, order, n_selected, keep,
                 stream=None) -> int:
    """bsa_top_p_select: per-sequence block order by score and the top-p count."""
    return lib().bsa_top_p_select(_ptr(scores), _ptr(cu_seqlens), int(n_seqs), int(total_blocks),
                                  float(p), _ptr(order), _ptr(n_selected), _ptr(keep),
                                  _stream(stream))


def importance_blocks(cu_seqlens_host) -> int:
    import numpy as np
    cu = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
    return lib().bsa_importance_blocks(cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       int(cu.shape[0] - 1))


def get_device_status(stream=None) -> int:
    return lib().bsa_get_device_status(_stream(stream))


def get_noalloc_status(stream=None) -> int:
    """bsa_get_noalloc_status: device-side status of the no-allocation calls."""
    return lib().bsa_get_noalloc_status(_stream(stream))


def release_stream(stream=None) -> int:
    """bsa_release_stream: free the scratch kept for one stream."""
    return lib().bsa_release_stream(_stream(stream))


def status_string(status: int) -> str:
    return lib().bsa_status_string(int(status)).decode()


def version() -> int:
    return lib().bsa_version()


def release() -> None:
    lib().bsa_release()


def debug_fault_drill(drop_k_load: int, wait_limit_ns: int) -> int:
    return lib().bsa_debug_fault_drill(int(drop_k_load), int(wait_limit_ns))


def check(status: int, what: str = "bsa") -> None:
    if status != 0:
        raise BsaError(status, what)
