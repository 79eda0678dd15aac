"""The fp64 oracle against its pins (CPU only), plus planted-mistake checks.

The oracle is what every GPU parity test compares against, so it is pinned to
things other than itself first: finite differences, a hand-derived worked
example, closed forms, invariants, an independent library forward and
structural reductions (see ``tests/oracle_pins.py``).  The mutation test then
plants plausible mistakes in a copy of the C source and checks that each one
fails at least one pin.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle_pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle_mod, pin):
    pin(oracle_mod.default())


def test_thread_count_does_not_change_bits(oracle_mod):
    rng = np.random.default_rng(40)
    q = rng.standard_normal((2, 33, 4, 8))
    k = rng.standard_normal((2, 33, 2, 8))
    v = rng.standard_normal((2, 33, 2, 8))
    do = rng.standard_normal((2, 33, 4, 8))
    a = oracle_mod.backward(q, k, v, do, 0.35, True, nthreads=1)
    b = oracle_mod.backward(q, k, v, do, 0.35, True, nthreads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_rejects_bad_shapes(oracle_mod):
    rng = np.random.default_rng(41)
    q = rng.standard_normal((1, 4, 3, 2))
    k = rng.standard_normal((1, 4, 2, 2))   # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle_mod.forward(q, k, k, 1.0)
    q = rng.standard_normal((1, 4, 2, 2))
    k = rng.standard_normal((1, 4, 1, 2))
    with pytest.raises(ValueError):
        oracle_mod.backward_sampled(q, k, k, q, 1.0, qrows=[(0, 4, 0)])  # row out of range


# Each mutant replaces one exact snippet of fa_oracle.c.
MUTANTS = {
    "dS sign of D": ("ds = pij * (dropout_factor(p, b, h, i, j) * dprob(p, b, h, i, j) - dv);",
                     "ds = pij * (dropout_factor(p, b, h, i, j) * dprob(p, b, h, i, j) + dv);"),
    "dS drops D in dK": ("double ds = pij * (f * dprob(p, b, h, i, j) - dvec_g[g][i]);",
                         "double ds = pij * f * dprob(p, b, h, i, j);"),
    "dK without scale": ("for (int d = 0; d < D; ++d) dk_out[d] *= p->scale;", ""),
    "dQ without scale": ("for (int d = 0; d < D; ++d) dq_out[d] *= p->scale;", ""),
    "dV uses dS": ("dv_out[d] += pij * f * doi[d];", "dv_out[d] += ds * doi[d];"),
    "dK uses dO": ("dk_out[d] += ds * qi[d];", "dk_out[d] += ds * doi[d];"),
    "top-left causal": ("if (p->causal && j > i + diag) return 0;",
                        "if (p->causal && j > i) return 0;"),
    "causal off by one": ("if (p->causal && j > i + diag) return 0;",
                          "if (p->causal && j >= i + diag) return 0;"),
    "GQA head mapping": ("int hk = h / p->G;\n    double s = p->scale",
                         "int hk = h % p->Hkv;\n    double s = p->scale"),
    "window left off by one": ("j < i + diag - p->ext.window_left", "j <= i + diag - p->ext.window_left"),
    "window right off by one": ("j > i + diag + p->ext.window_right",
                                "j >= i + diag + p->ext.window_right"),
    "window top-left aligned": ("j > i + diag + p->ext.window_right", "j > i + p->ext.window_right"),
    "ALiBi sign": ("s -= slope *", "s += slope *"),
    "ALiBi signed distance": ("s -= slope * (double)(dist < 0 ? -dist : dist);",
                              "s -= slope * (double)dist;"),
    "ALiBi top-left aligned": ("int dist = i + (seq_len_k(p, b) - seq_len_q(p, b)) - j;",
                               "int dist = i - j;"),
    "ALiBi ignores the batch stride": ("p->ext.alibi[(long)b * p->ext.alibi_bstride + h]",
                                       "p->ext.alibi[h]"),
    "seqused_k ignored": ("return p->ext.seqused_k ? p->ext.seqused_k[b] : stored_len_k(p, b);",
                          "return stored_len_k(p, b);"),
    "bias sign": ("s += p->ext.bias[", "s -= p->ext.bias["),
    "bias transposed": ("(long)i * p->ext.bias_rs + j];", "(long)j * p->ext.bias_rs + i];"),
    "bias ignores the head stride": ("(long)h * p->ext.bias_hs +", "0 +"),
    "bias scaled": ("        s += p->ext.bias[", "        s += p->scale * p->ext.bias["),
    "Philox key bump sign": ("k0 += 0x9E3779B9u;", "k0 -= 0x9E3779B9u;"),
    "Philox word order": ("c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;",
                          "c[0] = n2; c[1] = n1; c[2] = n0; c[3] = n3;"),
    "dropout without the keep scale": ("return 256.0 / (256.0 - p->ext.dropout_t);", "return 1.0;"),
    "dropout counter query / key swapped": (
        "unsigned int ctr[4] = {(unsigned int)j >> 4, (unsigned int)i,",
        "unsigned int ctr[4] = {(unsigned int)i >> 4, (unsigned int)j,"),
    "dropout mask missing from dS": ("double ds = pij * (f * dprob(p, b, h, i, j) - dvec_g[g][i]);",
                                     "double ds = pij * (dprob(p, b, h, i, j) - dvec_g[g][i]);"),
    "dropout mask missing from dV": ("dv_out[d] += pij * f * doi[d];", "dv_out[d] += pij * doi[d];"),
    "seqused_q ignored": ("return p->ext.seqused_q ? p->ext.seqused_q[b] : stored_len_q(p, b);",
                          "return stored_len_q(p, b);"),
    "Dv from q": ("return dot(doi, o_scratch, p->Dv);", "return dot(doi, p->q + row_q(p, b, i, h), p->Dv);"),
    "dP over the query / key dim": ("p->v + row_v(p, b, j, hk), p->Dv);", "p->v + row_v(p, b, j, hk), p->D);"),
    "dV rows at the key stride": ("dv + row_v(&p, b, j, hk));", "dv + row_k(&p, b, j, hk));"),
    "O rows at the query stride": ("row_forward(&p, b, h, i, o + row_o(&p, b, i, h));",
                                   "row_forward(&p, b, h, i, o + row_q(&p, b, i, h));"),
    "dV summed over D columns": ("for (int d = 0; d < Dv; ++d) dv_out[d] += pij * f * doi[d];",
                                 "for (int d = 0; d < D; ++d) dv_out[d] += pij * f * doi[d];"),
    "value dim taken as D": ("p->Dv = p->ext.head_dim_v > 0 ? p->ext.head_dim_v : D;", "p->Dv = D;"),
    "preprocess skips the LSE guard": ("if (lse == -INFINITY) lse = 0.0; /* get_validated_lse */", ""),
    "LSE drops max shift": ("double lse = m + log(sum);", "double lse = log(sum);"),
    "score without scale": ("double s = p->scale * dot(", "double s = dot("),
    "varlen lse index": ("if (p->cu_q) return (long)h * p->total_q + p->cu_q[b] + s;",
                         "if (p->cu_q) return (long)h * p->total_q + s;"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(old) == 1, "mutant snippet must match exactly once: %r" % old
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle_mod.compile_library(str(mpath), str(tmp_path / "libmutant.so"), openmp=False)
    # a subprocess, so that a mutant that crashes counts as caught without
    # taking the test run down
    res = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), lib],
                         capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        return
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, "planted mistake %r passed every pin" % name
