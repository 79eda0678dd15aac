"""Head dims above 128 and a value head dim Dv different from the query / key
dim D, on the GPU against the fp64 oracle (which takes Dv from v's shape).

These run in the second backward kernel (dK / dV / dQ in 128-column halves,
32 queries per step).  Inputs are seeded and drawn here (Q, K, V, dO in that
order, N(0, 1)); O and LSE come from the oracle's fp64 forward, rounded as a
forward kernel would store them.
"""
import numpy as np
import pytest
import torch

from gpu_util import check_bar, to64

pytestmark = pytest.mark.gpu


def make_case(oracle_mod, B, Sq, Sk, Hq, Hkv, D, Dv, dtype=torch.bfloat16, causal=False,
              lengths=None, seed=0):
    g = torch.Generator().manual_seed(seed)
    if lengths is None:
        q = torch.randn((B, Sq, Hq, D), generator=g)
        k = torch.randn((B, Sk, Hkv, D), generator=g)
        v = torch.randn((B, Sk, Hkv, Dv), generator=g)
        do = torch.randn((B, Sq, Hq, Dv), generator=g)
        cu = None
    else:
        T = sum(lengths)
        q = torch.randn((T, Hq, D), generator=g)
        k = torch.randn((T, Hkv, D), generator=g)
        v = torch.randn((T, Hkv, Dv), generator=g)
        do = torch.randn((T, Hq, Dv), generator=g)
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v, do = (t.to(dtype) for t in (q, k, v, do))
    scale = 1.0 / np.sqrt(D)
    o64, lse64 = oracle_mod.forward(to64(q), to64(k), to64(v), scale, causal, cu_q=cu, cu_k=cu)
    x = dict(q=q, k=k, v=v, dout=do, o=torch.from_numpy(o64).to(dtype),
             lse=torch.from_numpy(lse64).float(), scale=scale, causal=causal, cu=cu,
             max_len=(max(lengths) if lengths else None))
    return x


def oracle_grads(oracle_mod, x, window=None):
    kw = {} if window is None else dict(window=window)
    return oracle_mod.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["dout"]),
                               x["scale"], x["causal"], o=to64(x["o"]), lse=to64(x["lse"]),
                               cu_q=x["cu"], cu_k=x["cu"], **kw)


def gpu_grads(fa, x, outs=None, **kw):
    g = {n: x[n].cuda() for n in ("q", "k", "v", "dout", "o", "lse")}
    vl = {}
    if x["cu"] is not None:
        cu = torch.from_numpy(x["cu"]).cuda()
        vl = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=x["max_len"],
                  max_seqlen_k=x["max_len"])
    if outs is not None:
        kw.update(dq=outs[0], dk=outs[1], dv=outs[2])
    r = fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], causal=x["causal"],
                  softmax_scale=x["scale"], **vl, **kw)
    torch.cuda.synchronize()
    return r


CASES = [
    # (B, Sq, Sk, Hq, Hkv, D, Dv, dtype, causal)
    (2, 300, 300, 4, 2, 192, 192, torch.bfloat16, True),      # D = 192, causal GQA
    (1, 200, 200, 2, 2, 256, 256, torch.float16, False),      # D = 256
    (1, 257, 257, 4, 1, 256, 256, torch.bfloat16, True),      # D = 256, causal, ragged
    (2, 190, 190, 2, 1, 192, 128, torch.bfloat16, True),      # Dqk = 192, Dv = 128
    (1, 160, 160, 2, 2, 96, 160, torch.bfloat16, False),      # Dv > Dqk
    (1, 130, 130, 2, 2, 128, 64, torch.float16, True),        # unequal, both <= 128
    (1, 100, 300, 2, 2, 256, 256, torch.bfloat16, True),      # Sq < Sk, bottom-right causal
    (1, 300, 100, 2, 1, 192, 128, torch.bfloat16, True),      # Sq > Sk: rows with no key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_sq%d_sk%d_hq%d_hkv%d_d%d_dv%d_%s%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "bf16" if c[7] == torch.bfloat16 else "fp16",
    "_causal" if c[8] else ""))
def test_wide_head_dims_match_oracle(fa, oracle_mod, cuda_device, case):
    B, Sq, Sk, Hq, Hkv, D, Dv, dtype, causal = case
    x = make_case(oracle_mod, B, Sq, Sk, Hq, Hkv, D, Dv, dtype, causal, seed=D + Dv + Sq)
    dq, dk, dv = gpu_grads(fa, x)
    assert dq.shape[-1] == D and dk.shape[-1] == D and dv.shape[-1] == Dv
    rq, rk, rv = oracle_grads(oracle_mod, x)
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")


@pytest.mark.parametrize("D,Dv", [(256, 256), (192, 128)])
def test_wide_varlen_matches_oracle(fa, oracle_mod, cuda_device, D, Dv):
    x = make_case(oracle_mod, 3, 0, 0, 4, 2, D, Dv, torch.bfloat16, True, lengths=[260, 1, 131],
                  seed=7)
    dq, dk, dv = gpu_grads(fa, x)
    rq, rk, rv = oracle_grads(oracle_mod, x)
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")


def test_wide_outputs_written_in_bounds_only(fa, oracle_mod, cuda_device):
    x = make_case(oracle_mod, 1, 150, 150, 2, 1, 192, 136, torch.bfloat16, True, seed=3)
    pad = 4096
    outs, bufs = [], []
    for t in (x["q"], x["k"], x["v"]):
        n = t.numel()
        buf = torch.full((n + 2 * pad,), -7.0, dtype=t.dtype, device="cuda")
        bufs.append(buf)
        outs.append(buf[pad:pad + n].view(t.shape))
    gpu_grads(fa, x, outs=outs)
    for buf in bufs:
        assert bool((buf[:pad] == -7.0).all()) and bool((buf[-pad:] == -7.0).all())
    for got, ref, name in zip(outs, oracle_grads(oracle_mod, x), ("dq", "dk", "dv")):
        check_bar(got, ref, name)


def test_wide_refusals(fa, oracle_mod, cuda_device):
    """What the wide kernel does not build is refused before any launch."""
    x = make_case(oracle_mod, 1, 64, 64, 2, 2, 192, 192, torch.bfloat16, True, seed=1)
    g = {n: x[n].cuda() for n in ("q", "k", "v", "dout", "o", "lse")}
    args = (g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"])
    for kw in (dict(deterministic=True), dict(alibi_slopes=torch.ones(2, device="cuda"))):
        with pytest.raises(fa.FaError) as e:
            fa.fa_bwd(*args, causal=True, **kw)
        assert e.value.status == fa.FA_ERR_UNSUPPORTED
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(g["q"], g["k"], g["v"], causal=True, alibi_slopes=torch.ones(2, device="cuda"))
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%d_sq%d_sk%d_hq%d_hkv%d_d%d_dv%d_%s%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "bf16" if c[7] == torch.bfloat16 else "fp16",
    "_causal" if c[8] else ""))
def test_wide_forward_matches_oracle(fa, oracle_mod, cuda_device, case):
    B, Sq, Sk, Hq, Hkv, D, Dv, dtype, causal = case
    x = make_case(oracle_mod, B, Sq, Sk, Hq, Hkv, D, Dv, dtype, causal, seed=D + Dv + Sq)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=causal,
                       softmax_scale=x["scale"])
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    assert o.shape[-1] == Dv
    check_bar(o, to64(x["o"]), "o")
    lg, lr = to64(lse), to64(x["lse"])
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert np.max(np.abs(lg[fin] - lr[fin])) < 1e-4


@pytest.mark.parametrize("D,Dv", [(256, 256), (192, 128)])
def test_wide_varlen_forward_then_backward(fa, oracle_mod, cuda_device, D, Dv):
    """The library's forward feeds its backward (as a training step does):
    both against the oracle's fp64 forward and backward on the same inputs."""
    x = make_case(oracle_mod, 3, 0, 0, 4, 2, D, Dv, torch.bfloat16, True, lengths=[200, 77, 131],
                  seed=9)
    cu = torch.from_numpy(x["cu"]).cuda()
    vl = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=x["max_len"], max_seqlen_k=x["max_len"])
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, causal=True, softmax_scale=x["scale"], **vl)
    torch.cuda.synchronize()
    check_bar(o, to64(x["o"]), "o")
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal=True, softmax_scale=x["scale"], **vl)
    torch.cuda.synchronize()
    rq, rk, rv = oracle_mod.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["dout"]),
                                     x["scale"], True, cu_q=x["cu"], cu_k=x["cu"])
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")


WINDOWS = [
    # (B, Sq, Sk, Hq, Hkv, D, Dv, causal, window, lengths)
    (1, 300, 300, 4, 2, 256, 256, True, (100, 0), None),
    (2, 260, 260, 2, 1, 192, 128, False, (64, 32), None),
    (1, 200, 330, 2, 2, 128, 256, True, (40, -1), None),
    (3, 0, 0, 4, 2, 256, 256, True, (70, 0), [260, 1, 131]),
]


@pytest.mark.parametrize("case", WINDOWS, ids=lambda c: "d%d_dv%d_w%d_%d%s" % (
    c[5], c[6], c[8][0], c[8][1], "_varlen" if c[9] else ""))
def test_wide_window_matches_oracle(fa, oracle_mod, cuda_device, case):
    """A left (and right) window at head dims above 128 or Dv != D: the
    forward against the oracle's fp64 forward, then the backward from the
    oracle's O / LSE against its gradients."""
    B, Sq, Sk, Hq, Hkv, D, Dv, causal, window, lengths = case
    x = make_case(oracle_mod, B, Sq, Sk, Hq, Hkv, D, Dv, torch.bfloat16, causal,
                  lengths=lengths, seed=D + Dv + window[0])
    # the inputs' O / LSE from the oracle's forward with the window
    o64, lse64 = oracle_mod.forward(to64(x["q"]), to64(x["k"]), to64(x["v"]), x["scale"], causal,
                                    cu_q=x["cu"], cu_k=x["cu"], window=window)
    x["o"] = torch.from_numpy(o64).to(torch.bfloat16)
    x["lse"] = torch.from_numpy(lse64).float()
    kw = dict(window=window)
    vl = {}
    if x["cu"] is not None:
        cu = torch.from_numpy(x["cu"]).cuda()
        vl = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=x["max_len"],
                  max_seqlen_k=x["max_len"])
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    o, lse = fa.fa_fwd(q, k, v, causal=causal, softmax_scale=x["scale"], **vl, **kw)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    check_bar(o, to64(x["o"]), "o")
    dq, dk, dv = gpu_grads(fa, x, **kw)
    assert fa.device_status() == fa.FA_OK
    rq, rk, rv = oracle_grads(oracle_mod, x, window=window)
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")
