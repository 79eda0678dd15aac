"""The five benchmark workloads at full size, in the same launch configuration
the benchmark times (fa_fwd for O / LSE, then fa_bwd), against the fp64
oracle on sampled output rows: dQ rows (b, s, h) and dK / dV rows (b, s, hk)
spread over the sequence, the first and last positions included.  The oracle
recomputes its own fp64 forward for these rows (no oracle input comes from the
GPU).  Deterministic workloads are also run twice and compared bit for bit."""
import numpy as np
import pytest
import torch

from attention_backward_preprocess_gb300.workloads import WORKLOAD_ORDER, WORKLOADS, generate
from gpu_util import check_bar, to64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _rows(rng, n, lengths, heads, groups=None):
    """n (b, s, head) triples; always includes the first and last position."""
    out = []
    B = len(lengths)
    for t in range(n):
        b = int(rng.integers(B)) if groups is None else groups[t % len(groups)][0]
        L = lengths[b]
        if L == 0:
            continue
        s = 0 if t == 0 else (L - 1 if t == 1 else int(rng.integers(L)))
        h = int(rng.integers(heads)) if groups is None else groups[t % len(groups)][1]
        out.append((b, s, h))
    return out


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_full_size_workload(fa, oracle_mod, cuda_device, name):
    w = WORKLOADS[name]
    x = generate(w, "cpu")
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    kw, cu_np = {}, None
    if w.varlen is not None:
        kw = dict(cu_seqlens_q=x["cu_q"].to(dev), cu_seqlens_k=x["cu_k"].to(dev),
                  max_seqlen_q=x["max_len"], max_seqlen_k=x["max_len"])
        lengths = x["lengths"]
        cu_np = x["cu_q"].numpy()
    else:
        lengths = [w.Sq] * w.B
    o, lse = fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, **kw)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal=w.causal, softmax_scale=w.softmax_scale,
                           deterministic=w.deterministic, **kw)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    if w.deterministic:
        dq2, dk2, dv2 = fa.fa_bwd(q, k, v, o, do, lse, causal=w.causal,
                                  softmax_scale=w.softmax_scale, deterministic=True, **kw)
        torch.cuda.synchronize()
        for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert fa.device_status() == fa.FA_OK
    rng = np.random.default_rng(7)
    big = w.Sq * w.Sk * w.Hq // w.Hkv >= 8192 * 8192
    qrows = _rows(rng, 32, lengths, w.Hq)
    groups = [(0, 0)] if big else [(0, 0), (len(lengths) - 1, w.Hkv - 1)]
    krows = _rows(rng, 16 if big else 24, lengths, w.Hkv, groups=groups)
    rq, rk, rv = oracle_mod.backward_sampled(
        to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["dout"]), w.softmax_scale, w.causal,
        cu_q=cu_np, cu_k=cu_np, qrows=qrows, krows=krows)

    def pick(t, rows, heads_dim):
        out = []
        for (b, s, h) in rows:
            if w.varlen is not None:
                out.append(t[int(cu_np[b]) + s, h])
            else:
                out.append(t[b, s, h])
        return torch.stack(out)

    check_bar(pick(dq, qrows, w.Hq), rq, name + " dq rows")
    check_bar(pick(dk, krows, w.Hkv), rk, name + " dk rows")
    check_bar(pick(dv, krows, w.Hkv), rv, name + " dv rows")
