"""Mutation check of the oracle's pins.

Each case copies the committed C oracle, plants one plausible mistake in the
copy (a dropped term, a wrong sign or index, a transposed operand, a wrong
mask), compiles it on the CPU and requires that at least one pin rejects it.
The committed oracle itself is never modified.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

MUTANTS = [
    ("dropped scale", "S[(size_t)r * Sk + j] = scale * dot;", "S[(size_t)r * Sk + j] = dot;"),
    ("mask hides the past", "for (int j = i + 1; j < Sk; ++j) S[(size_t)r * Sk + j] = -INFINITY;",
     "for (int j = 0; j < i && j < Sk; ++j) S[(size_t)r * Sk + j] = -INFINITY;"),
    ("mask hides the diagonal", "for (int j = i + 1; j < Sk; ++j) S[(size_t)r * Sk + j] = -INFINITY;",
     "for (int j = i; j < Sk; ++j) S[(size_t)r * Sk + j] = -INFINITY;"),
    ("K used as V", "acc += P[(size_t)r * Sk + j] * v[(size_t)j * D + d];",
     "acc += P[(size_t)r * Sk + j] * k[(size_t)j * D + d];"),
    ("transposed scores", "dot += q[(size_t)i * D + d] * k[(size_t)j * D + d];",
     "dot += q[(size_t)(j % Sq) * D + d] * k[(size_t)(i % Sk) * D + d];"),
    ("dropped last dimension", "for (int d = 0; d < D; ++d) dot += q[(size_t)i * D + d]",
     "for (int d = 0; d < D - 1; ++d) dot += q[(size_t)i * D + d]"),
    ("no normalisation", "P[(size_t)r * Sk + j] /= l;", "P[(size_t)r * Sk + j] /= 1.0;"),
    ("LSE without the max", "lse[r] = m + log(l);", "lse[r] = log(l);"),
    ("softmax without max subtraction", "P[(size_t)r * Sk + j] = exp(S[(size_t)r * Sk + j] - m);",
     "P[(size_t)r * Sk + j] = exp(S[(size_t)r * Sk + j]);"),
    ("partition size rounded down", "const int P = (Sk + num_splits - 1) / num_splits;",
     "const int P = Sk / num_splits;"),
    ("partial max unscaled", "if (scale * dot > m) m = scale * dot;", "if (dot > m) m = dot;"),
    ("merge weight without max", "acc += exp(m_part[s] - mg) / lg * o_part[(size_t)s * D + d];",
     "acc += 1.0 / lg * o_part[(size_t)s * D + d];"),
    ("merge LSE sign", "*lse = mg + log(lg);", "*lse = mg - log(lg);"),
    ("merge sum unweighted", "lg += exp(m_part[s] - mg) * l_part[s];", "lg += l_part[s];"),
    ("bwd drops D_i", "dS[(size_t)i * Sk + j] = Pi[j] * (dp - Di);", "dS[(size_t)i * Sk + j] = Pi[j] * dp;"),
    ("bwd D_i from dO.dO", "Di += dout[(size_t)i * D + d] * acc;",
     "Di += dout[(size_t)i * D + d] * dout[(size_t)i * D + d];"),
    ("bwd dP against K", "dp += dout[(size_t)i * D + d] * v[(size_t)j * D + d];",
     "dp += dout[(size_t)i * D + d] * k[(size_t)j * D + d];"),
    ("bwd dQ unscaled", "dq[(size_t)i * D + d] = scale * acc;", "dq[(size_t)i * D + d] = acc;"),
    ("bwd dQ against V", "acc += dS[(size_t)i * Sk + j] * k[(size_t)j * D + d];",
     "acc += dS[(size_t)i * Sk + j] * v[(size_t)j * D + d];"),
    ("bwd dK from P", "dk[(size_t)j * D + d] += ds_ij * q[(size_t)i * D + d];",
     "dk[(size_t)j * D + d] += p_ij * q[(size_t)i * D + d];"),
    ("bwd dV from dS", "dv[(size_t)j * D + d] += p_ij * dout[(size_t)i * D + d];",
     "dv[(size_t)j * D + d] += ds_ij * dout[(size_t)i * D + d];"),
    ("bwd dK unscaled", "for (size_t x = 0; x < (size_t)Sk * D; ++x) dk[x] *= scale;",
     "for (size_t x = 0; x < (size_t)Sk * D; ++x) dk[x] *= 1.0;"),
    ("bwd mask direction", "Pi[j] = (causal && j > i) ? -INFINITY : scale * qk;",
     "Pi[j] = (causal && j < i) ? -INFINITY : scale * qk;"),
    ("bwd softmax unnormalised", "for (int j = 0; j < Sk; ++j) Pi[j] /= l;", "for (int j = 0; j < Sk; ++j) Pi[j] /= 1.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    mutant = oracle.Oracle(oracle.compile_source(path, os.path.join(tmp_path, "libmutant.so")))
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin rejects the mutant '{name}'"


class _VarlenBwdMutant:
    """The committed oracle with one mistake planted in its packed-sequence
    backward (which composes per-sequence calls in Python, not C)."""

    def __init__(self, base, kind):
        self.base, self.kind = base, kind

    def __getattr__(self, name):
        return getattr(self.base, name)

    def attention_bwd_varlen(self, q, k, v, dout, cq, ck, causal, scale, nthreads=None):
        import numpy as np
        q, k, v, dout = (oracle._f64(x) for x in (q, k, v, dout))
        if self.kind == "one block":  # sequences not separated
            g = self.base.attention_bwd(*(x.transpose(1, 0, 2) for x in (q, k, v, dout)), causal, scale)
            return tuple(x.transpose(1, 0, 2) for x in g)
        cq, ck = [int(x) for x in cq], [int(x) for x in ck]
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for i in range(len(cq) - 1):
            q0, q1, k0, k1 = cq[i], cq[i + 1], ck[i], ck[i + 1]
            if q1 == q0 or k1 == k0:
                continue
            if self.kind == "keys at query offsets":
                k0, k1 = q0, min(q0 + (k1 - k0), k.shape[0])
            g = self.base.attention_bwd(*(x.transpose(1, 0, 2) for x in (q[q0:q1], k[k0:k1], v[k0:k1], dout[q0:q1])),
                                        causal, scale)
            g = [x.transpose(1, 0, 2) for x in g]
            dq[q0:q1] = g[0]
            if self.kind == "key gradients at query offsets":
                n = min(k1 - k0, dk.shape[0] - q0)
                dk[q0:q0 + n], dv[q0:q0 + n] = g[1][:n], g[2][:n]
            else:
                dk[k0:k1], dv[k0:k1] = g[1], g[2]
        return dq, dk, dv


@pytest.mark.parametrize("kind", ["one block", "keys at query offsets", "key gradients at query offsets"])
def test_varlen_bwd_pin_rejects_mutant(kind):
    from oracle_pins import pin_bwd_varlen_block_diag
    with pytest.raises(AssertionError):
        pin_bwd_varlen_block_diag(_VarlenBwdMutant(oracle.get(), kind))
