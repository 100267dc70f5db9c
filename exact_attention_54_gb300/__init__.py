"""GB300-native exact attention: FlashAttention-2 forward (dense and packed
varlen, causal or not, with per-row LSE) and split-KV decoding with a
log-sum-exp merge, as hand-written sm_103a kernels behind the C ABI declared in
include/fa.h.

This module is the thin Python binding over libfa.so: the functions named like
the C entry points (``fa_fwd``, ``fa_fwd_varlen``, ``fa_decode_splitkv``,
``fa_splitkv_merge``) only marshal torch CUDA tensors into pointers and sizes
and check the returned status. ``flash_attention``, ``flash_attention_varlen``
and ``flash_decode`` additionally allocate the outputs (and the decode
workspace) with torch. Every step of the computation runs in the library's
kernels; there is no fallback. If libfa.so is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["FAError", "fa_fwd", "fa_fwd_varlen", "fa_decode_splitkv", "fa_decode_paged_splitkv", "fa_splitkv_merge",
           "fa_decode_splitkv_fused", "fa_decode_paged_splitkv_fused", "fa_bwd", "fa_bwd_workspace_bytes",
           "fa_bwd_varlen", "fa_bwd_varlen_workspace_bytes", "fa_check_device_error", "fa_status_string",
           "fa_test_withhold_load",
           "flash_attention", "flash_attention_varlen", "flash_attention_bwd", "flash_attention_varlen_bwd",
           "flash_decode", "flash_decode_paged", "library_path", "load_library", "EXPORTED_SYMBOLS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libfa.so")
_lock = threading.Lock()
_lib = None

FA_FP16, FA_BF16 = 0, 1
FA_MAX_SPLITS = 1024
EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_varlen", "fa_decode_splitkv", "fa_decode_paged_splitkv", "fa_splitkv_merge",
                    "fa_decode_splitkv_fused", "fa_decode_paged_splitkv_fused", "fa_bwd", "fa_bwd_workspace_bytes",
                    "fa_bwd_varlen", "fa_bwd_varlen_workspace_bytes", "fa_check_device_error", "fa_status_string",
                    "fa_version", "fa_test_withhold_load")


class FAError(RuntimeError):
    """A libfa entry point returned a non-zero status."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libfa.so (declares the argument types of every entry point)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built: run exact_attention_54_gb300.build.build() "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
        lib.fa_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_splitkv_merge.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
        lib.fa_decode_splitkv_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_decode_paged_splitkv_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                                      f, i, vp]
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, i, f, i, vp]
        lib.fa_test_withhold_load.argtypes = [i, ctypes.c_ulonglong]
        lib.fa_bwd.restype = ctypes.c_int
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp, vp, i, i, i, i, i,
                                      i, i, i, f, i, vp]
        lib.fa_bwd_varlen.restype = ctypes.c_int
        lib.fa_bwd_varlen_workspace_bytes.argtypes = [i, i, i]
        lib.fa_bwd_varlen_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_check_device_error.argtypes = [vp]
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        for name in ("fa_fwd", "fa_fwd_varlen", "fa_decode_splitkv", "fa_splitkv_merge", "fa_decode_splitkv_fused",
                     "fa_decode_paged_splitkv_fused", "fa_check_device_error", "fa_version"):
            getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise FAError(fn, status, fa_status_string(status))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: expected float16 or bfloat16")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need_contig(*ts):
    for t in ts:
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


# ------------------------------------------------------------- entry points --

def fa_fwd(q, k, v, o, lse, causal: bool, scale: float | None = None, stream=None):
    """Dense forward: q, o [B,H,Sq,D]; k, v [B,H,Sk,D]; lse [B,H,Sq] fp32."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    _need_contig(q, k, v, o, lse)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Sk, D, int(bool(causal)),
                               float(scale), _dtype_code(q), _stream(stream))
    _check("fa_fwd", st)


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal: bool,
                  scale: float | None = None, stream=None):
    """Packed forward: q, o [total_q,H,D]; k, v [total_k,H,D]; lse [H,total_q];
    cu_seqlens_* int32 CUDA tensors of length num_seqs+1."""
    Tq, H, D = q.shape
    Tk = k.shape[0]
    _need_contig(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                                      _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, Tq, Tk, int(max_seqlen_q), H,
                                      D, int(bool(causal)), float(scale), _dtype_code(q), _stream(stream))
    _check("fa_fwd_varlen", st)


def fa_decode_splitkv(q, k, v, o_part, m_part, l_part, num_splits: int, scale: float | None = None, stream=None):
    """Phase 1: q [B,H,1,D] (or [B,H,D]); k, v [B,H,Sk,D]; o_part [B,H,S,D],
    m_part and l_part [B,H,S] fp32."""
    B, H, Sk, D = k.shape
    _need_contig(q, k, v, o_part, m_part, l_part)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o_part), _ptr(m_part), _ptr(l_part),
                                          B, H, Sk, D, int(num_splits), float(scale), _dtype_code(k),
                                          _stream(stream))
    _check("fa_decode_splitkv", st)


def fa_decode_paged_splitkv(q, k_cache, v_cache, block_table, seq_lens, o_part, m_part, l_part, num_splits: int,
                            scale: float | None = None, stream=None):
    """Phase 1 over a paged cache: q [B,H,1,D]; k_cache, v_cache
    [num_blocks,H,block_size,D]; block_table [B,max_blocks] and seq_lens [B]
    int32 CUDA tensors; partials as in fa_decode_splitkv."""
    B, H = q.shape[0], q.shape[1]
    num_blocks, _, block_size, D = k_cache.shape
    _need_contig(q, k_cache, v_cache, block_table, seq_lens, o_part, m_part, l_part)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    lib = load_library()
    fn = lib.fa_decode_paged_splitkv
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    fn.restype = ctypes.c_int
    _check("fa_decode_paged_splitkv",
           fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(o_part), _ptr(m_part),
              _ptr(l_part), B, H, D, num_blocks, block_size, block_table.shape[1], int(num_splits), float(scale),
              _dtype_code(q), _stream(stream)))


def fa_splitkv_merge(o_part, m_part, l_part, o, lse, stream=None):
    """Phase 2: partials from phase 1 -> o [B,H,1,D] (16-bit), lse [B,H] fp32."""
    B, H, S, D = o_part.shape
    _need_contig(o_part, m_part, l_part, o, lse)
    st = load_library().fa_splitkv_merge(_ptr(o_part), _ptr(m_part), _ptr(l_part), _ptr(o), _ptr(lse), B, H, D,
                                         S, _dtype_code(o), _stream(stream))
    _check("fa_splitkv_merge", st)


def fa_decode_splitkv_fused(q, k, v, o, lse, o_part, m_part, l_part, counters, num_splits: int,
                            scale: float | None = None, stream=None):
    """Both decode phases in one launch. Arguments as fa_decode_splitkv plus
    o [B,H,1,D], lse [B,H] and counters, an int32 [B*H] CUDA tensor that is
    zero before the first call and is left zero by every completed call."""
    B, H, Sk, D = k.shape
    _need_contig(q, k, v, o, lse, o_part, m_part, l_part, counters)
    if counters.dtype != torch.int32:
        raise TypeError("counters must be int32")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_decode_splitkv_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(o_part),
                                                _ptr(m_part), _ptr(l_part), _ptr(counters), B, H, Sk, D,
                                                int(num_splits), float(scale), _dtype_code(k), _stream(stream))
    _check("fa_decode_splitkv_fused", st)


def fa_decode_paged_splitkv_fused(q, k_cache, v_cache, block_table, seq_lens, o, lse, o_part, m_part, l_part,
                                  counters, num_splits: int, scale: float | None = None, stream=None):
    """Both decode phases over a paged cache in one launch (arguments as
    fa_decode_paged_splitkv plus o, lse and counters as fa_decode_splitkv_fused)."""
    B, H = q.shape[0], q.shape[1]
    num_blocks, _, block_size, D = k_cache.shape
    _need_contig(q, k_cache, v_cache, block_table, seq_lens, o, lse, o_part, m_part, l_part, counters)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32 or counters.dtype != torch.int32:
        raise TypeError("block_table, seq_lens and counters must be int32")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_decode_paged_splitkv_fused(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(o), _ptr(lse), _ptr(o_part),
        _ptr(m_part), _ptr(l_part), _ptr(counters), B, H, D, num_blocks, block_size, block_table.shape[1],
        int(num_splits), float(scale), _dtype_code(q), _stream(stream))
    _check("fa_decode_paged_splitkv_fused", st)


def fa_bwd_workspace_bytes(B: int, H: int, Sq: int, D: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, Sq, D))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal: bool, scale: float | None = None, stream=None):
    """Backward pass: q, o, dout, dq [B,H,Sq,D]; k, v, dk, dv [B,H,Sk,D];
    lse [B,H,Sq] fp32 from the forward; workspace a CUDA tensor of at least
    fa_bwd_workspace_bytes(B, H, Sq, D) bytes."""
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    _need_contig(q, k, v, o, dout, lse, dq, dk, dv, workspace)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, Sq,
                               Sk, D, int(bool(causal)), float(scale), _dtype_code(q), _stream(stream))
    _check("fa_bwd", st)


def fa_bwd_varlen_workspace_bytes(total_q: int, H: int, D: int) -> int:
    return int(load_library().fa_bwd_varlen_workspace_bytes(total_q, H, D))


def fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, causal: bool, scale: float | None = None, stream=None):
    """Backward pass over packed sequences: q, o, dout, dq [total_q,H,D]; k, v,
    dk, dv [total_k,H,D]; lse [H,total_q] fp32 from fa_fwd_varlen;
    cu_seqlens_* int32 CUDA tensors of length num_seqs+1; workspace a CUDA
    tensor of at least fa_bwd_varlen_workspace_bytes(total_q, H, D) bytes."""
    Tq, H, D = q.shape
    Tk = k.shape[0]
    _need_contig(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens_q, cu_seqlens_k)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    st = load_library().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                      _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, Tq, Tk,
                                      int(max_seqlen_q), int(max_seqlen_k), H, D, int(bool(causal)), float(scale),
                                      _dtype_code(q), _stream(stream))
    _check("fa_bwd_varlen", st)


def fa_test_withhold_load(load: int, wait_limit_ns: int = 0):
    """Test support: make CTA 0 of later prefill launches withhold one tile
    load so that their bounded wait runs out (see include/fa.h); (0, 0) turns
    it off."""
    _check("fa_test_withhold_load", load_library().fa_test_withhold_load(int(load), int(wait_limit_ns)))


def fa_check_device_error(stream=None):
    """Synchronise the stream and raise if a kernel abandoned a barrier wait."""
    _check("fa_check_device_error", load_library().fa_check_device_error(_stream(stream)))


# ------------------------------------------------------ allocating helpers --

def flash_attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Returns (o, lse) for dense [B,H,S,D] CUDA tensors."""
    B, H, Sq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def flash_attention_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, stream=None,
                        workspace=None):
    """Returns (dq, dk, dv) for dense [B,H,S,D] CUDA tensors, given the
    forward's o and lse."""
    B, H, Sq, D = q.shape
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, Sq, D) // 4, dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal, scale, stream)
    return dq, dk, dv


def flash_attention_varlen_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                               max_seqlen_k: int, causal: bool = False, scale: float | None = None, stream=None,
                               workspace=None):
    """Returns (dq, dk, dv) for packed sequences, given fa_fwd_varlen's o and lse."""
    Tq, H, D = q.shape
    if workspace is None:
        workspace = torch.empty(fa_bwd_varlen_workspace_bytes(Tq, H, D) // 4, dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  max_seqlen_k, causal, scale, stream)
    return dq, dk, dv


def flash_attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal: bool = False,
                           scale: float | None = None, stream=None):
    """Returns (o [total_q,H,D], lse [H,total_q]) for packed sequences."""
    Tq, H, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(H, Tq, dtype=torch.float32, device=q.device)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, causal, scale, stream)
    return o, lse


def _decode_workspace(B, H, S, D, device, fused):
    ws = (torch.empty(B, H, S, D, dtype=torch.float32, device=device),
          torch.empty(B, H, S, dtype=torch.float32, device=device),
          torch.empty(B, H, S, dtype=torch.float32, device=device))
    return ws + (torch.zeros(B * H, dtype=torch.int32, device=device),) if fused else ws


def flash_decode_paged(q, k_cache, v_cache, block_table, seq_lens, num_splits: int, scale: float | None = None,
                       stream=None, workspace=None, fused: bool = False):
    """Split-KV decoding over a paged cache (phase 1 + phase 2). Returns
    (o [B,H,1,D], lse [B,H]). ``workspace`` may pass preallocated (o_part,
    m_part, l_part), plus the int32 [B*H] counters when ``fused``."""
    B, H = q.shape[0], q.shape[1]
    D = k_cache.shape[3]
    if workspace is None:
        workspace = _decode_workspace(B, H, num_splits, D, q.device, fused)
    o = torch.empty(B, H, 1, D, dtype=q.dtype, device=q.device)
    lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    if fused:
        fa_decode_paged_splitkv_fused(q, k_cache, v_cache, block_table, seq_lens, o, lse, *workspace, num_splits,
                                      scale, stream)
        return o, lse
    o_part, m_part, l_part = workspace[:3]
    fa_decode_paged_splitkv(q, k_cache, v_cache, block_table, seq_lens, o_part, m_part, l_part, num_splits, scale,
                            stream)
    fa_splitkv_merge(o_part, m_part, l_part, o, lse, stream)
    return o, lse


def flash_decode(q, k, v, num_splits: int, scale: float | None = None, stream=None, workspace=None,
                 fused: bool = False):
    """Split-KV decoding (phase 1 + phase 2). Returns (o [B,H,1,D], lse [B,H]).
    ``workspace`` may pass preallocated (o_part, m_part, l_part), plus the
    int32 [B*H] counters when ``fused`` (one launch instead of two)."""
    B, H, Sk, D = k.shape
    if workspace is None:
        workspace = _decode_workspace(B, H, num_splits, D, k.device, fused)
    o = torch.empty(B, H, 1, D, dtype=k.dtype, device=k.device)
    lse = torch.empty(B, H, dtype=torch.float32, device=k.device)
    if fused:
        fa_decode_splitkv_fused(q, k, v, o, lse, *workspace, num_splits, scale, stream)
        return o, lse
    o_part, m_part, l_part = workspace[:3]
    fa_decode_splitkv(q, k, v, o_part, m_part, l_part, num_splits, scale, stream)
    fa_splitkv_merge(o_part, m_part, l_part, o, lse, stream)
    return o, lse


def fa_decode_noalloc(q, k, v, o, lse, num_splits: int, scale: float | None = None, stream=None):
    """Split-KV decoding (both phases) with no device allocation and no
    workspace argument, for callers that cannot allocate device memory when
    they call in. The partials use a fixed device array built into the
    library (FA_NOALLOC_SCRATCH_FLOATS floats); concurrent calls whose GPU work
    overlaps race on it. q [B,H,1,D]; k, v [B,H,Sk,D]; o [B,H,1,D]; lse [B,H]."""
    lib = load_library()
    fn = lib.fa_decode_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    fn.restype = ctypes.c_int
    B, H, Sk, D = k.shape
    _need_contig(q, k, v, o, lse)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    _check("fa_decode_noalloc", fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sk, D, int(num_splits),
                                   float(scale), _dtype_code(k), _stream(stream)))
