"""Exact-attention oracle (fp64, CPU).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path may not.
It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``attention_ref.c`` (plain C, fp64, materialises S and
P); this module compiles it with gcc, widens inputs to float64 arrays and lays
out the outputs. Each function names the passage it follows.

Parity pins live in tests/test_oracle.py: torch's fp64
scaled_dot_product_attention and logsumexp on tiny shapes, closed forms and
invariants, the split/merge identity, block-diagonal SDPA for the varlen
bookkeeping, torch fp64 autograd and central finite differences of the
oracle's own forward for the backward pass, and mutation tests that plant
mistakes in a copy of the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def compile_source(src: str, out: str) -> str:
    """gcc -O2 (no fast-math) a C oracle source into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile attention_ref.c into oracle/_build/liboracle.so when stale."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _f64(x) -> np.ndarray:
    """Exact widening of the given values (fp16/bf16/fp32 tensors or arrays) to fp64."""
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU, values unchanged
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_attention.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, _ip, ctypes.c_int, ctypes.c_int]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_splitkv_partials.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
        lib.oracle_splitkv_partials.restype = ctypes.c_int
        lib.oracle_splitkv_merge.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, _dp, _dp]
        lib.oracle_splitkv_merge.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                             ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def attention(self, q, k, v, causal: bool, scale: float, rows=None, nthreads: int | None = None):
        """Exact attention for tensors laid out [..., S, D] (leading dims = heads).

        The plain definition: S = scale*QK^T, keys k > q hidden when causal,
        row softmax, P V, LSE = m + ln l (attention_ref.c cites the passages).
        ``rows`` restricts the query rows evaluated (the same rows in every
        head). Returns (o, lse) float64 arrays [..., nrows, D] and [..., nrows].
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        lead = q.shape[:-2]
        Sq, D = q.shape[-2:]
        Sk = k.shape[-2]
        if k.shape[:-2] != lead or v.shape != k.shape or k.shape[-1] != D:
            raise ValueError("shape mismatch between q, k and v")
        BH = int(np.prod(lead)) if lead else 1
        if rows is None:
            nrows, rows_ptr, rows_arr = Sq, None, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
            nrows = int(rows_arr.size)
            rows_ptr = rows_arr.ctypes.data_as(_ip)
        o = np.zeros((BH, nrows, D), np.float64)
        lse = np.zeros((BH, nrows), np.float64)
        rc = self.lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), BH, Sq, Sk, D,
                                       int(bool(causal)), float(scale), rows_ptr, nrows,
                                       nthreads or default_threads())
        del rows_arr
        if rc != 0:
            raise ValueError(f"oracle_attention failed ({rc})")
        return o.reshape(*lead, nrows, D), lse.reshape(*lead, nrows)

    def attention_bwd(self, q, k, v, dout, causal: bool, scale: float, nthreads: int | None = None):
        """Gradients (dq, dk, dv) of sum(O * dout) for O = attention(q, k, v)
        ("Adaptive High-Performance Attention Kernels in CUDA", Advanced
        Production Features 2: S and P recomputed, D_i = sum_k dO_ik O_ik,
        dS = P (dP - D); dV = P^T dO, dP = dO V^T, dQ = scale dS K,
        dK = scale dS^T Q). Tensors laid out [..., S, D]; float64 results."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        lead = q.shape[:-2]
        Sq, D = q.shape[-2:]
        Sk = k.shape[-2]
        if k.shape[:-2] != lead or v.shape != k.shape or dout.shape != q.shape or k.shape[-1] != D:
            raise ValueError("shape mismatch between q, k, v and dout")
        BH = int(np.prod(lead)) if lead else 1
        dq = np.zeros((BH, Sq, D), np.float64)
        dk = np.zeros((BH, Sk, D), np.float64)
        dv = np.zeros((BH, Sk, D), np.float64)
        rc = self.lib.oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                           BH, Sq, Sk, D, int(bool(causal)), float(scale),
                                           nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_attention_bwd failed ({rc})")
        return dq.reshape(*lead, Sq, D), dk.reshape(*lead, Sk, D), dv.reshape(*lead, Sk, D)

    def attention_varlen(self, q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float,
                         nthreads: int | None = None, seqs=None):
        """Packed variable-length attention ("Adaptive High-Performance Attention
        Kernels in CUDA", Advanced Production Features 3: tokens flattened to
        [total_tokens, H, d], sequences delimited by cumulative lengths).

        Each sequence is an independent exact attention over its own keys, with
        causal positions counted from the sequence start. Returns o
        [total_q, H, D] and lse [H, total_q] (per-head contiguous) as float64;
        ``seqs`` limits the work to those sequence indices (others stay 0).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        cq = [int(x) for x in np.asarray(cu_seqlens_q).tolist()]
        ck = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
        Tq, H, D = q.shape
        o = np.zeros((Tq, H, D), np.float64)
        lse = np.zeros((H, Tq), np.float64)
        for i in (range(len(cq) - 1) if seqs is None else seqs):
            q0, q1, k0, k1 = cq[i], cq[i + 1], ck[i], ck[i + 1]
            if q1 == q0:
                continue
            oi, li = self.attention(q[q0:q1].transpose(1, 0, 2), k[k0:k1].transpose(1, 0, 2),
                                    v[k0:k1].transpose(1, 0, 2), causal, scale, nthreads=nthreads)
            o[q0:q1] = oi.transpose(1, 0, 2)
            lse[:, q0:q1] = li
        return o, lse

    def attention_bwd_varlen(self, q, k, v, dout, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float,
                             nthreads: int | None = None):
        """Gradients of packed variable-length attention (attention_varlen)
        with respect to q, k, v for the upstream gradient dout ("Adaptive
        High-Performance Attention Kernels in CUDA", Advanced Production
        Features 2 and 3). Each sequence is an independent exact attention over
        its own keys, so its gradients are those of its own block, computed by
        attention_bwd; causal positions count from each sequence's start.
        Tokens laid out [total, H, D]; returns float64 dq [total_q, H, D] and
        dk, dv [total_k, H, D]. Keys of a sequence without queries, and queries
        of a sequence without keys, get zero gradients."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        cq = [int(x) for x in np.asarray(cu_seqlens_q).tolist()]
        ck = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for i in range(len(cq) - 1):
            q0, q1, k0, k1 = cq[i], cq[i + 1], ck[i], ck[i + 1]
            if q1 == q0 or k1 == k0:
                continue
            g = self.attention_bwd(*(x.transpose(1, 0, 2) for x in (q[q0:q1], k[k0:k1], v[k0:k1], dout[q0:q1])),
                                   causal, scale, nthreads=nthreads)
            dq[q0:q1], dk[k0:k1], dv[k0:k1] = (x.transpose(1, 0, 2) for x in g)
        return dq, dk, dv

    def splitkv_partials(self, q, k, v, num_splits: int, scale: float):
        """Split-K decoding phase 1 for q [..., 1, D] (or [..., D]) and k, v [..., Sk, D].

        Returns o_part [..., S, D] (unnormalised), m_part [..., S], l_part [..., S].
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        Sk, D = k.shape[-2:]
        lead = k.shape[:-2]
        q = q.reshape(-1, D)
        k = k.reshape(-1, Sk, D)
        v = v.reshape(-1, Sk, D)
        BH = k.shape[0]
        if q.shape[0] != BH:
            raise ValueError("q and k disagree on the number of heads")
        o_part = np.zeros((BH, num_splits, D), np.float64)
        m_part = np.zeros((BH, num_splits), np.float64)
        l_part = np.zeros((BH, num_splits), np.float64)
        for h in range(BH):
            qh, kh, vh = (np.ascontiguousarray(x[h]) for x in (q, k, v))
            rc = self.lib.oracle_splitkv_partials(_ptr(qh), _ptr(kh), _ptr(vh), Sk, D, float(scale),
                                                  num_splits, _ptr(o_part[h]), _ptr(m_part[h]),
                                                  _ptr(l_part[h]))
            if rc != 0:
                raise ValueError(f"oracle_splitkv_partials failed ({rc})")
        return (o_part.reshape(*lead, num_splits, D), m_part.reshape(*lead, num_splits),
                l_part.reshape(*lead, num_splits))

    def splitkv_merge(self, o_part, m_part, l_part):
        """Split-K decoding phase 2: log-sum-exp merge of the partials.

        o_part [..., S, D], m_part/l_part [..., S] -> o [..., D], lse [...].
        """
        o_part, m_part, l_part = _f64(o_part), _f64(m_part), _f64(l_part)
        S, D = o_part.shape[-2:]
        lead = o_part.shape[:-2]
        op = o_part.reshape(-1, S, D)
        mp = m_part.reshape(-1, S)
        lp = l_part.reshape(-1, S)
        n = op.shape[0]
        o = np.zeros((n, D), np.float64)
        lse = np.zeros((n,), np.float64)
        for h in range(n):
            a, b, c = (np.ascontiguousarray(x[h]) for x in (op, mp, lp))
            rc = self.lib.oracle_splitkv_merge(_ptr(a), _ptr(b), _ptr(c), S, D, _ptr(o[h]),
                                               _ptr(lse[h:h + 1]))
            if rc != 0:
                raise ValueError(f"oracle_splitkv_merge failed ({rc})")
        return o.reshape(*lead, D), lse.reshape(*lead)

    def paged_gather(self, cache, block_table, seq_lens):
        """Contiguous keys (or values) of every sequence from a paged cache
        ("Adaptive High-Performance Attention Kernels in CUDA", Advanced
        Production Features 4: physical pages [num_blocks, H, block_size, d],
        logical position p of sequence b lives in page block_table[b][p //
        block_size] at offset p % block_size). Returns a list of [H, L_b, d]
        float64 arrays."""
        cache = _f64(cache)
        bt = np.asarray(block_table).astype(np.int64)
        lens = [int(x) for x in np.asarray(seq_lens).tolist()]
        bs = cache.shape[2]
        out = []
        for b, L in enumerate(lens):
            pages = [cache[bt[b, p // bs], :, p % bs, :] for p in range(L)]  # each [H, d]
            out.append(np.stack(pages, axis=1) if pages else np.zeros((cache.shape[1], 0, cache.shape[3])))
        return out

    def decode_paged(self, q, k_cache, v_cache, block_table, seq_lens, scale: float):
        """Single-query attention per (sequence, head) over the keys a block
        table maps into a paged cache: gather, then exact attention. q is
        [B, H, 1, d]; returns o [B, H, 1, d] and lse [B, H, 1] (a sequence of
        length 0 gives o = 0 and lse = -inf)."""
        q = _f64(q)
        ks = self.paged_gather(k_cache, block_table, seq_lens)
        vs = self.paged_gather(v_cache, block_table, seq_lens)
        B, H, _, D = q.shape
        o = np.zeros((B, H, 1, D))
        lse = np.full((B, H, 1), -np.inf)
        for b in range(B):
            if ks[b].shape[1] == 0:
                continue
            o[b], lse[b] = self.attention(q[b], ks[b], vs[b], False, scale)
        return o, lse

    def decode(self, q, k, v, scale: float, nthreads: int | None = None):
        """Single-query attention (Sq = 1) computed without splitting: the
        result the split/merge pair must reproduce."""
        return self.attention(q, k, v, False, scale, nthreads=nthreads)


def get() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def attention(*a, **kw):
    return get().attention(*a, **kw)


def attention_varlen(*a, **kw):
    return get().attention_varlen(*a, **kw)


def splitkv_partials(*a, **kw):
    return get().splitkv_partials(*a, **kw)


def splitkv_merge(*a, **kw):
    return get().splitkv_merge(*a, **kw)


def decode(*a, **kw):
    return get().decode(*a, **kw)


def decode_paged(*a, **kw):
    return get().decode_paged(*a, **kw)


def attention_bwd(*a, **kw):
    return get().attention_bwd(*a, **kw)


def attention_bwd_varlen(*a, **kw):
    return get().attention_bwd_varlen(*a, **kw)
