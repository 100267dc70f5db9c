"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with
  * a library routine computing the same special case (torch's fp64
    scaled_dot_product_attention and logsumexp on tiny shapes, block-diagonal
    SDPA for packed sequences), or
  * a closed form or invariant of exact attention (rows of P summing to 1,
    a single key, all-equal scores, causal row 0, two keys, score shift,
    permutation equivariance), or
  * the split-K decoding identity (phase 1 + phase 2 equal full attention), or
  * for the backward pass: torch fp64 autograd through SDPA, central finite
    differences of the oracle's own forward, and gradient invariants.
tests/test_oracle_mutants.py plants mistakes in copies of the C source and
checks that every one of them trips at least one pin here.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

TOL = 1e-12


def _rand(shape, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def _masked_scores(q, k, scale, causal):
    s = scale * (q @ k.transpose(-1, -2))
    if causal:
        Sq, Sk = s.shape[-2:]
        keep = torch.ones(Sq, Sk, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, float("-inf"))
    return s


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


def pin_sdpa(orc):
    """torch SDPA (fp64, is_causal = top-left tril mask) and logsumexp on tiny shapes."""
    seed = 0
    for D in (1, 4, 64):
        for Sq in (1, 2, 3, 17):
            for Sk in (1, 2, 3, 17):
                for causal in (False, True):
                    seed += 1
                    q, k, v = _rand((2, Sq, D), seed), _rand((2, Sk, D), seed + 500), _rand((2, Sk, D), seed + 900)
                    scale = 0.3 + 0.1 * (seed % 7)
                    o, lse = orc.attention(q, k, v, causal, scale)
                    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
                    ref_lse = torch.logsumexp(_masked_scores(q, k, scale, causal), dim=-1)
                    _close(o, ref.numpy(), what=f"O D={D} Sq={Sq} Sk={Sk} causal={causal}")
                    _close(lse, ref_lse.numpy(), what=f"LSE D={D} Sq={Sq} Sk={Sk} causal={causal}")


def pin_rows_sum_to_one(orc):
    """With V = 1 every output equals the row sum of P, which must be 1."""
    for causal in (False, True):
        q, k = _rand((3, 19, 8), 11), _rand((3, 23, 8), 12)
        v = torch.ones(3, 23, 8, dtype=torch.float64)
        o, _ = orc.attention(q, k, v, causal, 0.7)
        _close(o, np.ones_like(o), what=f"row sums causal={causal}")


def pin_single_key(orc):
    """Sk = 1: O = V[0] and LSE = scale * q . k0 for every query."""
    q, k, v = _rand((2, 5, 16), 21), _rand((2, 1, 16), 22), _rand((2, 1, 16), 23)
    scale = 0.25
    o, lse = orc.attention(q, k, v, False, scale)
    _close(o, v.expand(2, 5, 16).numpy(), what="single key O")
    _close(lse, (scale * (q @ k.transpose(-1, -2)))[..., 0].numpy(), what="single key LSE")


def pin_equal_scores(orc):
    """K = 0 makes every score 0: O = mean of the visible V rows, LSE = ln(#visible)."""
    Sk, D = 9, 6
    q, v = _rand((2, Sk, D), 31), _rand((2, Sk, D), 32)
    k = torch.zeros(2, Sk, D, dtype=torch.float64)
    o, lse = orc.attention(q, k, v, False, 1.3)
    _close(o, v.mean(dim=1, keepdim=True).expand(2, Sk, D).numpy(), what="equal scores O")
    _close(lse, np.full((2, Sk), math.log(Sk)), what="equal scores LSE")
    o, lse = orc.attention(q, k, v, True, 1.3)
    counts = torch.arange(1, Sk + 1, dtype=torch.float64)
    prefix_mean = torch.cumsum(v, dim=1) / counts[None, :, None]
    _close(o, prefix_mean.numpy(), what="equal scores causal O")
    _close(lse, np.log(counts.numpy())[None, :].repeat(2, 0), what="equal scores causal LSE")


def pin_causal_row0(orc):
    """Causal row 0 sees only key 0: O[0] = V[0], LSE[0] = scale * q0 . k0."""
    q, k, v = _rand((4, 12, 32), 41), _rand((4, 12, 32), 42), _rand((4, 12, 32), 43)
    scale = 1 / math.sqrt(32)
    o, lse = orc.attention(q, k, v, True, scale)
    _close(o[:, 0], v[:, 0].numpy(), what="causal row 0 O")
    _close(lse[:, 0], (scale * (q[:, 0] * k[:, 0]).sum(-1)).numpy(), what="causal row 0 LSE")


def pin_two_keys(orc):
    """Two keys: O = sigmoid(s0 - s1) V0 + sigmoid(s1 - s0) V1, LSE = log(e^s0 + e^s1)."""
    q, k, v = _rand((1, 7, 5), 51), _rand((1, 2, 5), 52), _rand((1, 2, 5), 53)
    scale = 0.9
    o, lse = orc.attention(q, k, v, False, scale)
    for i in range(7):
        s0 = scale * float((q[0, i] * k[0, 0]).sum())
        s1 = scale * float((q[0, i] * k[0, 1]).sum())
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        _close(o[0, i], (w0 * v[0, 0] + w1 * v[0, 1]).numpy(), what="two keys O")
        mx = max(s0, s1)
        _close(lse[0, i], mx + math.log(math.exp(s0 - mx) + math.exp(s1 - mx)), what="two keys LSE")


def pin_shift(orc):
    """Adding the same c to every score of a row leaves O alone and shifts LSE by c.
    The shift is built by appending one dimension: q' = [q, 1], k' = [k, c/scale]
    (and a zero column to V, so O keeps its first D columns)."""
    q, k, v = _rand((2, 6, 7), 61), _rand((2, 10, 7), 62), _rand((2, 10, 7), 63)
    scale, c = 0.5, 3.75
    o, lse = orc.attention(q, k, v, False, scale)
    q2 = torch.cat([q, torch.ones(2, 6, 1, dtype=torch.float64)], -1)
    k2 = torch.cat([k, torch.full((2, 10, 1), c / scale, dtype=torch.float64)], -1)
    v2 = torch.cat([v, torch.zeros(2, 10, 1, dtype=torch.float64)], -1)
    o2, lse2 = orc.attention(q2, k2, v2, False, scale)
    _close(o2[..., :7], o, what="shift O")
    _close(lse2, lse + c, what="shift LSE")


def pin_permutation(orc):
    """Non-causal attention is invariant to permuting the (key, value) pairs and
    equivariant to permuting the queries."""
    q, k, v = _rand((3, 11, 9), 71), _rand((3, 13, 9), 72), _rand((3, 13, 9), 73)
    o, lse = orc.attention(q, k, v, False, 0.6)
    pk = torch.randperm(13, generator=torch.Generator().manual_seed(5))
    pq = torch.randperm(11, generator=torch.Generator().manual_seed(6))
    o2, lse2 = orc.attention(q, k[:, pk], v[:, pk], False, 0.6)
    _close(o2, o, what="key permutation O")
    _close(lse2, lse, what="key permutation LSE")
    o3, lse3 = orc.attention(q[:, pq], k, v, False, 0.6)
    _close(o3, o[:, pq.numpy()], what="query permutation O")
    _close(lse3, lse[:, pq.numpy()], what="query permutation LSE")


def pin_rows_subset(orc):
    """Evaluating a subset of rows gives exactly those rows of the full result."""
    q, k, v = _rand((2, 40, 8), 81), _rand((2, 40, 8), 82), _rand((2, 40, 8), 83)
    rows = [0, 7, 39, 13, 13]
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.4)
        os_, ls_ = orc.attention(q, k, v, causal, 0.4, rows=rows)
        _close(os_, o[:, rows], tol=0.0, what="row subset O")
        _close(ls_, lse[:, rows], tol=0.0, what="row subset LSE")


def pin_partials_definition(orc):
    """Phase-1 partials: m_s is the largest scaled score in partition s,
    O_s / l_s is exact attention over that partition's keys and
    m_s + ln l_s its LSE (checked with torch SDPA / logsumexp); an empty
    partition has m = -inf, l = 0, O = 0."""
    D = 8
    for Sk, S in ((100, 32), (17, 5), (64, 4), (7, 7)):
        q, k, v = _rand((3, 1, D), 91 + Sk), _rand((3, Sk, D), 92 + Sk), _rand((3, Sk, D), 93 + Sk)
        scale = 1 / math.sqrt(D)
        op, mp, lp = orc.splitkv_partials(q, k, v, S, scale)
        P = -(-Sk // S)
        for s in range(S):
            lo, hi = s * P, min(s * P + P, Sk)
            if lo >= hi:
                assert np.all(mp[:, s] == -np.inf) and np.all(lp[:, s] == 0) and np.all(op[:, s] == 0)
                continue
            ks, vs = k[:, lo:hi], v[:, lo:hi]
            scores = scale * (q @ ks.transpose(-1, -2))[:, 0]
            _close(mp[:, s], scores.max(-1).values.numpy(), what="partial max")
            ref = F.scaled_dot_product_attention(q, ks, vs, scale=scale)[:, 0]
            _close(op[:, s] / lp[:, s, None], ref.numpy(), what="partial O/l")
            _close(mp[:, s] + np.log(lp[:, s]), torch.logsumexp(scores, -1).numpy(), what="partial LSE")


def pin_merge_identity(orc):
    """Phase 2 applied to phase 1 equals full attention (uneven, single and empty partitions)."""
    D = 16
    for Sk, S in ((100, 32), (17, 5), (256, 1), (7, 7), (300, 8)):
        q, k, v = _rand((4, 1, D), 101 + Sk), _rand((4, Sk, D), 102 + Sk), _rand((4, Sk, D), 103 + Sk)
        scale = 1 / math.sqrt(D)
        op, mp, lp = orc.splitkv_partials(q, k, v, S, scale)
        o, lse = orc.splitkv_merge(op, mp, lp)
        ref = F.scaled_dot_product_attention(q, k, v, scale=scale)[:, 0]
        ref_lse = torch.logsumexp(scale * (q @ k.transpose(-1, -2))[:, 0], -1)
        _close(o, ref.numpy(), what=f"merge O Sk={Sk} S={S}")
        _close(lse, ref_lse.numpy(), what=f"merge LSE Sk={Sk} S={S}")


def pin_varlen_block_diag(orc):
    """Packed sequences equal SDPA over the whole packed stream with a
    block-diagonal mask (causal inside each block); LSE is laid out [H, T]."""
    lengths = [5, 1, 17, 9]
    H, D = 3, 8
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = _rand((T, H, D), 111), _rand((T, H, D), 112), _rand((T, H, D), 113)
    scale = 0.45
    for causal in (False, True):
        o, lse = orc.attention_varlen(q, k, v, cu, cu, causal, scale)
        seg = torch.repeat_interleave(torch.arange(len(lengths)), torch.tensor(lengths))
        pos = torch.cat([torch.arange(n) for n in lengths])
        keep = seg[:, None] == seg[None, :]
        if causal:
            keep &= pos[None, :] <= pos[:, None]
        qh, kh, vh = (x.transpose(0, 1) for x in (q, k, v))  # [H, T, D]
        ref = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=keep, scale=scale).transpose(0, 1)
        s = (scale * qh @ kh.transpose(-1, -2)).masked_fill(~keep, float("-inf"))
        _close(o, ref.numpy(), what=f"varlen O causal={causal}")
        _close(lse, torch.logsumexp(s, -1).numpy(), what=f"varlen LSE causal={causal}")


def pin_paged_gather(orc):
    """A paged cache built by scattering dense K/V into randomly permuted pages
    (and sharing one prefix page between two sequences) gives exactly the
    dense single-query attention of each sequence; a length-0 sequence gives
    O = 0, LSE = -inf."""
    H, D, bs = 2, 8, 4
    lens = [9, 4, 0, 13]
    g = torch.Generator().manual_seed(121)
    nblk = sum(-(-L // bs) for L in lens) + 3
    perm = torch.randperm(nblk, generator=g).tolist()
    kc = torch.zeros(nblk, H, bs, D, dtype=torch.float64)
    vc = torch.zeros(nblk, H, bs, D, dtype=torch.float64)
    maxb = max(-(-L // bs) for L in lens)
    bt = torch.zeros(len(lens), maxb, dtype=torch.int32)
    q = _rand((len(lens), H, 1, D), 122)
    dense = []
    nxt = 0
    for b, L in enumerate(lens):
        k, v = _rand((H, L, D), 123 + b), _rand((H, L, D), 223 + b)
        if b == 3:  # share sequence 0's first page (same key/value content)
            k[:, :bs], v[:, :bs] = dense[0][0][:, :bs], dense[0][1][:, :bs]
        dense.append((k, v))
        for i in range(-(-L // bs)):
            if b == 3 and i == 0:
                bt[b, i] = bt[0, 0]
                continue
            page = perm[nxt]
            nxt += 1
            bt[b, i] = page
            n = min(bs, L - i * bs)
            kc[page, :, :n] = k[:, i * bs:i * bs + n]
            vc[page, :, :n] = v[:, i * bs:i * bs + n]
    o, lse = orc.decode_paged(q, kc, vc, bt, torch.tensor(lens, dtype=torch.int32), 0.35)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(o[b] == 0) and np.all(lse[b] == -np.inf)
            continue
        k, v = dense[b]
        ref = F.scaled_dot_product_attention(q[b], k, v, scale=0.35)
        _close(o[b], ref.numpy(), what=f"paged O seq {b}")
        _close(lse[b, :, 0], torch.logsumexp(0.35 * (q[b] @ k.transpose(-1, -2))[:, 0], -1).numpy(),
               what=f"paged LSE seq {b}")


def _sdpa_grads(q, k, v, do, causal, scale):
    q, k, v = (t.clone().requires_grad_() for t in (q, k, v))
    o = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    o.backward(do)
    return q.grad, k.grad, v.grad


def pin_bwd_autograd(orc):
    """dq, dk, dv against torch fp64 autograd through scaled_dot_product_attention
    (is_causal = top-left tril mask) on tiny shapes, Sq != Sk included."""
    seed = 3000
    for D in (1, 4, 16):
        for Sq, Sk in ((1, 1), (2, 3), (3, 2), (5, 5), (9, 17), (17, 9)):
            for causal in (False, True):
                seed += 1
                q, do = _rand((2, Sq, D), seed), _rand((2, Sq, D), seed + 1)
                k, v = _rand((2, Sk, D), seed + 2), _rand((2, Sk, D), seed + 3)
                scale = 0.25 + 0.1 * (seed % 5)
                got = orc.attention_bwd(q, k, v, do, causal, scale)
                ref = _sdpa_grads(q, k, v, do, causal, scale)
                for name, a, b in zip(("dq", "dk", "dv"), got, ref):
                    _close(a, b.numpy(), 1e-11, f"{name} D={D} Sq={Sq} Sk={Sk} causal={causal}")


def pin_bwd_finite_differences(orc):
    """Every element of dq, dk, dv equals the central difference of
    L = sum(O * dO) computed with the oracle's forward (an independent code
    path), on a tiny case, causal and not."""
    h = 1e-6
    for causal in (False, True):
        q, k, v = _rand((1, 3, 3), 41).numpy(), _rand((1, 4, 3), 42).numpy(), _rand((1, 4, 3), 43).numpy()
        do = _rand((1, 3, 3), 44).numpy()
        scale = 0.7
        grads = orc.attention_bwd(q, k, v, do, causal, scale)

        def loss(qq, kk, vv):
            return float(np.sum(orc.attention(qq, kk, vv, causal, scale)[0] * do))

        for idx, (x, g) in enumerate(zip((q, k, v), grads)):
            for pos in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[pos] += h
                xm[pos] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[idx], args_m[idx] = xp, xm
                fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
                assert abs(fd - g[pos]) <= 1e-7, f"{'qkv'[idx]}{pos} causal={causal}: fd {fd} vs {g[pos]}"


def pin_bwd_invariants(orc):
    """sum_j dK_j = 0 (every row of dS sums to zero); sum_j dV_j = sum_i dO_i
    (every row of P sums to one); adding one vector to every key changes no
    probability, so dQ and dV are unchanged."""
    for causal in (False, True):
        q, do = _rand((2, 7, 5), 51), _rand((2, 7, 5), 52)
        k, v = _rand((2, 9, 5), 53), _rand((2, 9, 5), 54)
        dq, dk, dv = orc.attention_bwd(q, k, v, do, causal, 0.6)
        _close(dk.sum(axis=1), np.zeros((2, 5)), 1e-12, f"sum dK causal={causal}")
        _close(dv.sum(axis=1), do.sum(dim=1).numpy(), 1e-12, f"sum dV causal={causal}")
        shift = _rand((1, 1, 5), 55)
        dq2, _, dv2 = orc.attention_bwd(q, k + shift, v, do, causal, 0.6)
        _close(dq2, dq, 1e-11, f"dq under key shift causal={causal}")
        _close(dv2, dv, 1e-11, f"dv under key shift causal={causal}")


def pin_bwd_varlen_block_diag(orc):
    """Packed-sequence gradients equal torch fp64 autograd through SDPA over
    the whole packed stream with a block-diagonal mask (top-left causal inside
    each block), with query and key lengths that differ per sequence so that
    positions counted from the wrong start would show; a sequence with no
    queries gets zero key gradients."""
    Lq, Lk = [3, 2, 0, 4, 1], [5, 2, 3, 6, 1]
    H, D = 2, 4
    cq = np.concatenate([[0], np.cumsum(Lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(Lk)]).astype(np.int32)
    Tq, Tk = sum(Lq), sum(Lk)
    q, do = _rand((Tq, H, D), 131), _rand((Tq, H, D), 132)
    k, v = _rand((Tk, H, D), 133), _rand((Tk, H, D), 134)
    scale = 0.55
    seg_q = torch.repeat_interleave(torch.arange(len(Lq)), torch.tensor(Lq))
    seg_k = torch.repeat_interleave(torch.arange(len(Lk)), torch.tensor(Lk))
    pos_q = torch.cat([torch.arange(n) for n in Lq])
    pos_k = torch.cat([torch.arange(n) for n in Lk])
    for causal in (False, True):
        got = orc.attention_bwd_varlen(q, k, v, do, cq, ck, causal, scale)
        keep = seg_q[:, None] == seg_k[None, :]
        if causal:
            keep &= pos_k[None, :] <= pos_q[:, None]
        qh, kh, vh = (x.transpose(0, 1).clone().requires_grad_(True) for x in (q, k, v))
        o = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=keep, scale=scale)
        (o * do.transpose(0, 1)).sum().backward()
        for name, a, b in zip(("dq", "dk", "dv"), got, (qh.grad, kh.grad, vh.grad)):
            _close(a, b.transpose(0, 1).numpy(), 1e-11, f"varlen {name} causal={causal}")
        # sequence 2 has keys [ck[2], ck[3]) and no queries: no gradient reaches them
        assert np.all(got[1][ck[2]:ck[3]] == 0) and np.all(got[2][ck[2]:ck[3]] == 0)


PINS = [pin_sdpa, pin_rows_sum_to_one, pin_single_key, pin_equal_scores, pin_causal_row0,
        pin_two_keys, pin_shift, pin_permutation, pin_rows_subset, pin_partials_definition,
        pin_merge_identity, pin_varlen_block_diag, pin_paged_gather, pin_bwd_autograd,
        pin_bwd_finite_differences, pin_bwd_invariants, pin_bwd_varlen_block_diag]
