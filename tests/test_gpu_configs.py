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


# Extensions at full size (fa_fwd_ext / fa_bwd_ext).  The oracle runs the
# forward of sequence 0 and the query heads of kv head 0 (fp64), rounds O to the
# input dtype and LSE to fp32, and the backward of that group is checked on
# sampled rows with those same rounded O / LSE as input on both sides (the
# other heads take the GPU forward's output: no oracle row depends on them).
# Exact inputs matter with dropout: a row that sees one key has dS = s dP - D
# = 0 exactly in fp64, but not with O rounded.  The GPU forward's O rows of the
# group are checked against the oracle's fp64 O.
EXT_FULL = [
    ("b2_hq32_hkv8_s8192_d128_causal_gqa", dict(window=(1024, -1), alibi=True)),
    ("b4_h16_s2048_d128_causal", dict(dropout=(0.1, 0x5EED, 3))),
    ("varlen16_h16_d64_fp16_causal", dict(window=(300, -1))),
]


@pytest.mark.parametrize("name,opt", EXT_FULL, ids=lambda v: v if isinstance(v, str) else "")
def test_full_size_extension(fa, oracle_mod, cuda_device, name, opt):
    w = WORKLOADS[name]
    G = w.Hq // w.Hkv
    x = generate(w, "cpu")
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    varlen = w.varlen is not None
    kw = {}
    if varlen:
        kw = dict(cu_seqlens_q=x["cu_q"].to(dev), cu_seqlens_k=x["cu_k"].to(dev),
                  max_seqlen_q=x["max_len"], max_seqlen_k=x["max_len"])
        L0 = x["lengths"][0]
        sl = lambda t, hs: t[0:L0, hs]
        cu_s = np.array([0, L0], dtype=np.int32)
    else:
        L0 = w.Sq
        sl = lambda t, hs: t[0:1, :, hs]
        cu_s = None
    gk, ok = {}, {}
    if "window" in opt:
        gk["window"] = ok["window"] = opt["window"]
    if opt.get("alibi"):
        slopes = np.array([2.0 ** (-8.0 * (h + 1) / w.Hq) for h in range(w.Hq)], dtype=np.float32)
        gk["alibi_slopes"] = torch.from_numpy(slopes).to(dev)
        ok["alibi"] = slopes[:G].astype(np.float64)
    if "dropout" in opt:
        pr, seed, off = opt["dropout"]
        gk["dropout"] = (pr, seed, off)
        ok["dropout"] = (min(255, int(np.float32(pr) * np.float32(256) + np.float32(0.5))), seed, off)
    # the group's inputs and the oracle's forward of it
    qs, ks, vs, dos = (to64(sl(x[n], slice(0, G) if n in ("q", "dout") else slice(0, 1)))
                       for n in ("q", "k", "v", "dout"))
    o64, lse64 = oracle_mod.forward(qs, ks, vs, w.softmax_scale, w.causal, cu_q=cu_s, cu_k=cu_s, **ok)
    o_r = torch.from_numpy(o64).to(w.torch_dtype)
    lse_r = torch.from_numpy(lse64).float()
    # GPU forward; its O rows of the group against the oracle's fp64 O
    o, lse = fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, **kw, **gk)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    check_bar(sl(o, slice(0, G)), o64, name + " o (group)")
    # GPU backward with the group's O / LSE replaced by the oracle's rounded ones
    o_in, lse_in = o.clone(), lse.clone()
    if varlen:
        o_in[0:L0, 0:G] = o_r.to(dev)
        lse_in[0:G, 0:L0] = lse_r.to(dev)
    else:
        o_in[0:1, :, 0:G] = o_r.to(dev)
        lse_in[0:1, 0:G] = lse_r.to(dev)
    dq, dk, dv = fa.fa_bwd(q, k, v, o_in, do, lse_in, causal=w.causal,
                           softmax_scale=w.softmax_scale, **kw, **gk)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    rng = np.random.default_rng(11)
    qrows = _rows(rng, 24, [L0], G)
    krows = _rows(rng, 12, [L0], 1)
    rq, rk, rv = oracle_mod.backward_sampled(
        qs, ks, vs, dos, w.softmax_scale, w.causal, o=to64(o_r), lse=to64(lse_r),
        cu_q=cu_s, cu_k=cu_s, qrows=qrows, krows=krows, **ok)

    def pick(t, rows):
        return torch.stack([t[s, h] if varlen else t[0, s, h] for (_, s, h) in rows])

    check_bar(pick(dq, qrows), rq, name + " dq rows")
    check_bar(pick(dk, krows), rk, name + " dk rows")
    check_bar(pick(dv, krows), rv, name + " dv rows")


def test_accumulator_past_2_31_elements(fa, oracle_mod, cuda_device):
    """The bench workload at B = 65: the fp32 dQ accumulator holds 65 x 32 x
    8192 rows x 128 = 2.18 G elements, past 2^31, so every index into it and
    into the outputs of the last sequences needs 64-bit arithmetic (about
    30 GB on the device).  Rows of the
    first and the last sequence are checked against the oracle, which takes
    that one sequence alone."""
    w = WORKLOADS["b2_hq32_hkv8_s8192_d128_causal_gqa"].with_(name="b65_hq32_hkv8_s8192", B=65)
    dev = torch.device("cuda")
    x = generate(w, dev)
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    lay = fa.workspace_layout(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    assert lay["rows"] * 128 > 2 ** 31
    o, lse = fa.fa_fwd(q, k, v, causal=True, softmax_scale=w.softmax_scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal=True, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    rng = np.random.default_rng(11)
    for b in (w.B - 1, 0):
        one = {n: x[n][b:b + 1].cpu() for n in ("q", "k", "v", "dout")}
        qrows = _rows(rng, 16, [w.Sq], w.Hq)
        krows = _rows(rng, 8, [w.Sk], w.Hkv, groups=[(0, w.Hkv - 1)])
        rq, rk, rv = oracle_mod.backward_sampled(
            to64(one["q"]), to64(one["k"]), to64(one["v"]), to64(one["dout"]), w.softmax_scale,
            True, qrows=qrows, krows=krows)
        got_q = torch.stack([dq[b, s, h] for (_, s, h) in qrows])
        got_k = torch.stack([dk[b, s, h] for (_, s, h) in krows])
        got_v = torch.stack([dv[b, s, h] for (_, s, h) in krows])
        check_bar(got_q, rq, "dq rows of sequence %d" % b)
        check_bar(got_k, rk, "dk rows of sequence %d" % b)
        check_bar(got_v, rv, "dv rows of sequence %d" % b)
    del q, k, v, do, o, lse, dq, dk, dv, x
    torch.cuda.empty_cache()
