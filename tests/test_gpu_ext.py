"""GPU forward and backward with the extensions of fa_fwd_ext / fa_bwd_ext
(local window, ALiBi, seqused) against the fp64 oracle, element by element.

Cases span several query tiles and key blocks with ragged tails, both head
dims, both dtypes, GQA, Sq != Sk, varlen, deterministic mode, and bands that
leave some query rows and some key blocks with nothing visible."""
import numpy as np
import pytest
import torch

from attention_backward_preprocess_gb300.workloads import Workload
from gpu_util import check_bar, small_case, to64

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


def W(name, B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=False, **kw):
    return Workload(name, B, Sq, Sk, Hq, Hkv, D, dtype, causal, **kw)


# (workload, extension options); alibi: "h" = slopes [Hq], "bh" = [B, Hq]
CASES = [
    (W("win_d128", 1, 300, 300, 2, 1, 128), dict(window=(100, 30))),
    (W("win_causal_d64", 1, 600, 600, 2, 2, 64, causal=True), dict(window=(150, -1))),
    (W("win_sq_lt_sk_d128", 1, 200, 450, 2, 2, 128), dict(window=(60, 20))),
    (W("win_sq_gt_sk_d64_fp16", 1, 400, 150, 2, 1, 64, "fp16"), dict(window=(40, 0))),
    (W("win_zero_d64", 2, 130, 130, 2, 2, 64), dict(window=(0, 0))),
    (W("win_right_only_d128", 1, 260, 260, 2, 2, 128), dict(window=(-1, 5))),
    (W("alibi_causal_d128_gqa", 1, 384, 384, 4, 2, 128, causal=True), dict(alibi="h")),
    (W("alibi_d64_fp16", 2, 200, 260, 2, 2, 64, "fp16"), dict(alibi="bh")),
    (W("alibi_win_causal_d128", 1, 300, 300, 2, 1, 128, causal=True),
     dict(alibi="h", window=(90, -1))),
    # ALiBi at D = 128 with keys right of the diagonal (the |.| form), and
    # causal with Sq < Sk (the linear form with diag > 0)
    (W("alibi_noncausal_d128", 1, 260, 300, 2, 2, 128), dict(alibi="bh")),
    (W("alibi_win_right_d128", 1, 300, 300, 2, 1, 128), dict(alibi="h", window=(50, 40))),
    (W("alibi_causal_sq_lt_sk_d128", 1, 200, 450, 2, 2, 128, causal=True), dict(alibi="h")),
    (W("seqused_causal_d128", 2, 300, 300, 2, 1, 128, causal=True),
     dict(seqused_q=[300, 170], seqused_k=[257, 300])),
    (W("seqused_win_d64", 2, 256, 256, 2, 2, 64), dict(seqused_q=[100, 256], seqused_k=[256, 31],
                                                        window=(40, 40))),
]


def _options(w, opt, seed=5):
    """(oracle keywords, GPU keywords) of an option dict."""
    ok, gk = {}, {}
    if "window" in opt:
        ok["window"] = gk["window"] = opt["window"]
    if "alibi" in opt:
        rng = np.random.default_rng(seed)
        shape = (w.Hq,) if opt["alibi"] == "h" else (w.B, w.Hq)
        sl = rng.uniform(0.02, 0.5, size=shape).astype(np.float32)
        ok["alibi"] = sl.astype(np.float64)
        gk["alibi_slopes"] = torch.from_numpy(sl).cuda()
    for name in ("seqused_q", "seqused_k"):
        if name in opt:
            a = np.asarray(opt[name], dtype=np.int32)
            ok[name] = a
            gk[name] = torch.from_numpy(a).cuda()
    if "bias" in opt:
        # "full" [B, Hq, ...], "b1" [1, Hq, ...], "h1" [B, 1, ...]; rows padded
        # past Sk (a row stride above Sk)
        g = torch.Generator().manual_seed(seed + 1)
        nb = 1 if opt["bias"] == "b1" else w.B
        nh = 1 if opt["bias"] == "h1" else w.Hq
        pad = (w.Sk + 7) // 8 * 8 + 8
        full = torch.randn((nb, nh, w.Sq, pad), generator=g).to(w.torch_dtype)
        view = full.cuda()[..., :w.Sk]
        ok["bias"] = to64(full[..., :w.Sk].contiguous())
        gk["bias"] = view
    if "dropout" in opt:
        # the library quantises p to t / 256, t = round(256 p) in fp32 (at most 255)
        pr, seed, off = opt["dropout"]
        t = min(255, int(np.float32(pr) * np.float32(256) + np.float32(0.5)))
        ok["dropout"] = (t, seed, off)
        gk["dropout"] = (pr, seed, off)
    return ok, gk


def _case(oracle_mod, w, opt, lengths=None):
    x = small_case(oracle_mod, w, lengths=lengths)
    ok, gk = _options(w, opt)
    cu = x.get("cu_q")
    cu_np = None if cu is None else cu.numpy()
    o64, lse64 = oracle_mod.forward(to64(x["q"]), to64(x["k"]), to64(x["v"]), w.softmax_scale,
                                    w.causal, cu_q=cu_np, cu_k=cu_np, **ok)
    x["o64"], x["lse64"] = o64, lse64
    x["o"] = torch.from_numpy(o64).to(w.torch_dtype)
    x["lse"] = torch.from_numpy(lse64).float()
    return x, ok, gk


def _used_rows(w, x, ok, side):
    """Boolean mask over the packed / dense rows a side uses: [B, S] or [total]."""
    cu = x.get("cu_q")
    used = ok.get("seqused_q" if side == "q" else "seqused_k")
    if cu is None:
        S = w.Sq if side == "q" else w.Sk
        n = np.full(w.B, S) if used is None else used
        return np.arange(S)[None, :] < np.asarray(n)[:, None]
    cu = cu.numpy()
    total = int(cu[-1])
    mask = np.zeros(total, dtype=bool)
    for b in range(len(cu) - 1):
        n = cu[b + 1] - cu[b] if used is None else used[b]
        mask[cu[b]:cu[b] + n] = True
    return mask


def _kw(w, x):
    if x.get("cu_q") is None:
        return {}
    cu = x["cu_q"].cuda()
    return dict(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=x["max_len"],
                max_seqlen_k=x["max_len"])


@pytest.mark.parametrize("w,opt", CASES, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_ext_forward_matches_oracle(fa, oracle_mod, cuda_device, w, opt):
    x, ok, gk = _case(oracle_mod, w, opt)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale, **_kw(w, x), **gk)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    mq = _used_rows(w, x, ok, "q")
    g, r = to64(o)[mq], x["o64"][mq]
    check_bar(g, r, "o")
    # LSE [B, Hq, Sq]: used rows only
    lg, lr = to64(lse).transpose(0, 2, 1)[mq], x["lse64"].transpose(0, 2, 1)[mq]
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert np.max(np.abs(lg[fin] - lr[fin])) < 1e-4


def _run_bwd(fa, w, x, gk, deterministic=False):
    dev = torch.device("cuda")
    outs = [torch.full_like(x[n], SENTINEL, device=dev) for n in ("q", "k", "v")]
    fa.fa_bwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), x["o"].to(dev),
              x["dout"].to(dev), x["lse"].to(dev), causal=w.causal,
              softmax_scale=w.softmax_scale, deterministic=deterministic, dq=outs[0],
              dk=outs[1], dv=outs[2], **_kw(w, x), **gk)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return outs


def _check_bwd(oracle_mod, w, x, ok, outs):
    cu = x.get("cu_q")
    cu_np = None if cu is None else cu.numpy()
    ref = oracle_mod.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["dout"]),
                              w.softmax_scale, w.causal, o=to64(x["o"]), lse=to64(x["lse"]),
                              cu_q=cu_np, cu_k=cu_np, **ok)
    mq, mk = _used_rows(w, x, ok, "q"), _used_rows(w, x, ok, "k")
    # When the exact gradient is 0 (a band of width 0: P = 1 on the diagonal,
    # so dS = P (dP - Dv) = 0), the GPU's dS is rounding only: dP and Dv are
    # fp32 sums of the same D products in different orders, each within
    # D * 2^-24 * sum|dO_d v_d|; dQ / dK multiply that by scale * |K| (|Q|).
    amax = lambda t: float(np.max(np.abs(to64(t)))) if t.numel() else 0.0
    zero_bound = (w.D * 2.0 ** -24 * w.D * amax(x["dout"]) * amax(x["v"]) * w.softmax_scale *
                  max(amax(x["q"]), amax(x["k"])) * 4)
    for t, rt, m, n in zip(outs, ref, (mq, mk, mk), ("dq", "dk", "dv")):
        g = to64(t)
        if rt[m].size and np.max(np.abs(rt[m])) == 0.0:
            assert np.max(np.abs(g[m])) <= zero_bound, (n, np.max(np.abs(g[m])), zero_bound)
        else:
            check_bar(g[m], rt[m], n)
        assert np.all(g[~m] == SENTINEL), n + ": rows past seqused were written"


@pytest.mark.parametrize("w,opt", CASES, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_ext_backward_matches_oracle(fa, oracle_mod, cuda_device, w, opt):
    x, ok, gk = _case(oracle_mod, w, opt)
    _check_bwd(oracle_mod, w, x, ok, _run_bwd(fa, w, x, gk))


BIAS_CASES = [
    (W("bias_d128_gqa", 2, 200, 200, 4, 2, 128), dict(bias="full")),
    (W("bias_causal_d64", 1, 330, 330, 2, 2, 64, causal=True), dict(bias="b1")),
    (W("bias_sq_lt_sk_d128_fp16", 2, 150, 270, 2, 1, 128, "fp16", causal=True), dict(bias="h1")),
    (W("bias_alibi_win_d64", 1, 260, 260, 2, 1, 64), dict(bias="full", alibi="h", window=(70, 20))),
    (W("bias_seqused_d128", 2, 256, 256, 2, 2, 128, causal=True),
     dict(bias="full", seqused_q=[256, 100], seqused_k=[200, 256])),
    # Sk a multiple of 8 (dBias rows by 16-byte stores) with used key lengths
    # that are not: the last 8-key group of a row is written element by element
    (W("bias_seqused_ragged_d128", 2, 256, 256, 2, 1, 128, causal=True),
     dict(bias="full", seqused_q=[250, 77], seqused_k=[203, 131])),
    (W("bias_seqused_ragged_d64_fp16", 1, 192, 320, 2, 2, 64, "fp16"),
     dict(bias="h1", seqused_k=[77])),
]


def _oracle_dbias(oracle_mod, w, x, ok):
    """dS of every (sequence, query head), [B, Hq, Sq, Sk], zero outside the used rows."""
    ref = np.zeros((w.B, w.Hq, w.Sq, w.Sk))
    for b in range(w.B):
        for h in range(w.Hq):
            _, dS = oracle_mod.head_matrices(to64(x["q"]), to64(x["k"]), to64(x["v"]),
                                             to64(x["dout"]), w.softmax_scale, w.causal,
                                             o=to64(x["o"]), lse=to64(x["lse"]), b=b, h=h, **ok)
            ref[b, h, :dS.shape[0], :dS.shape[1]] = dS
    return ref


@pytest.mark.parametrize("w,opt", BIAS_CASES, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_bias_forward_backward_dbias(fa, oracle_mod, cuda_device, w, opt):
    x, ok, gk = _case(oracle_mod, w, opt)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale, **gk)
    torch.cuda.synchronize()
    mq = _used_rows(w, x, ok, "q")
    check_bar(to64(o)[mq], x["o64"][mq], "o")
    lg, lr = to64(lse).transpose(0, 2, 1)[mq], x["lse64"].transpose(0, 2, 1)[mq]
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert np.max(np.abs(lg[fin] - lr[fin])) < 1e-4
    dbias = torch.full((w.B, w.Hq, w.Sq, w.Sk), SENTINEL, dtype=w.torch_dtype, device="cuda")
    outs = _run_bwd(fa, w, x, dict(gk, dbias=dbias))
    _check_bwd(oracle_mod, w, x, ok, outs)
    check_bar(dbias, _oracle_dbias(oracle_mod, w, x, ok), "dbias")


DROP_CASES = [
    (W("drop_causal_d128_gqa", 2, 300, 300, 4, 2, 128, causal=True),
     dict(dropout=(0.1, 0x0123456789ABCDEF, 0))),
    (W("drop_d64_fp16_sq_lt_sk", 1, 190, 333, 2, 2, 64, "fp16"),
     dict(dropout=(0.3, 42, 7))),
    (W("drop_alibi_win_d128", 1, 260, 260, 2, 1, 128, causal=True),
     dict(dropout=(0.2, 99, 1), alibi="h", window=(100, -1))),
    (W("drop_bias_d96", 2, 200, 200, 2, 2, 96), dict(dropout=(0.15, 5, 3), bias="b1")),
]


@pytest.mark.parametrize("w,opt", DROP_CASES, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_dropout_forward_backward(fa, oracle_mod, cuda_device, w, opt):
    x, ok, gk = _case(oracle_mod, w, opt)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale, **gk)
    torch.cuda.synchronize()
    check_bar(o, x["o64"], "o")
    fin = np.isfinite(x["lse64"])
    assert np.max(np.abs(to64(lse)[fin] - x["lse64"][fin])) < 1e-4
    extra = {}
    if "bias" in gk:
        extra["dbias"] = torch.full((w.B, w.Hq, w.Sq, w.Sk), SENTINEL, dtype=w.torch_dtype,
                                    device="cuda")
    outs = _run_bwd(fa, w, x, dict(gk, **extra))
    _check_bwd(oracle_mod, w, x, ok, outs)
    if extra:
        check_bar(extra["dbias"], _oracle_dbias(oracle_mod, w, x, ok), "dbias")


def test_dropout_varlen_and_deterministic(fa, oracle_mod, cuda_device):
    w = W("drop_vl_d128", 3, 0, 0, 2, 1, 128, "bf16", True, varlen=(3, 1, 300),
          deterministic=True)
    opt = dict(dropout=(0.25, 1234567, 11))
    x, ok, gk = _case(oracle_mod, w, opt, lengths=[300, 129, 40])
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale, **_kw(w, x), **gk)
    torch.cuda.synchronize()
    check_bar(o, x["o64"], "o")
    a = _run_bwd(fa, w, x, gk, deterministic=True)
    b = _run_bwd(fa, w, x, gk, deterministic=True)
    for t, u in zip(a, b):
        assert torch.equal(t.view(torch.int16), u.view(torch.int16))
    _check_bwd(oracle_mod, w, x, ok, a)


# The keep-flag buffer: fa_fwd writes the flags, fa_bwd reads them instead of
# running Philox again (workload, options, varlen lengths).
MASK_CASES = [
    (W("drop_mask_causal_d128_gqa", 2, 300, 300, 4, 2, 128, causal=True),
     dict(dropout=(0.1, 77, 5)), None),
    (W("drop_mask_d64_fp16_sq_lt_sk", 1, 190, 333, 2, 2, 64, "fp16"),
     dict(dropout=(0.3, 42, 7)), None),
    (W("drop_mask_bias_alibi_d128", 1, 260, 260, 2, 1, 128, causal=True),
     dict(dropout=(0.2, 9, 1), bias="b1", alibi="h"), None),
    (W("drop_mask_vl_d128", 3, 0, 0, 2, 1, 128, "bf16", True, varlen=(3, 1, 300)),
     dict(dropout=(0.25, 1234567, 11)), [300, 129, 40]),
]


@pytest.mark.parametrize("w,opt,lengths", MASK_CASES,
                         ids=lambda v: v.name if hasattr(v, "name") else "")
def test_dropout_mask_buffer(fa, oracle_mod, cuda_device, w, opt, lengths):
    x, ok, gk = _case(oracle_mod, w, opt, lengths=lengths)
    kw = _kw(w, x)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    shape = fa.dropout_mask_shape(q, k, kw.get("cu_seqlens_q"), kw.get("max_seqlen_k"))
    mask = torch.full(shape, -1, dtype=torch.int32, device="cuda")
    gk_m = dict(gk, dropout=tuple(gk["dropout"]) + (mask,))
    o, lse = fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale, **kw, **gk_m)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    check_bar(o, x["o64"], "o")
    # reading the flags gives the gradients drawing them gives, bit for bit in
    # deterministic mode (otherwise the dQ sums' order varies from run to run)
    drawn = _run_bwd(fa, w, x, gk, deterministic=True)
    read = _run_bwd(fa, w, x, gk_m, deterministic=True)
    for a, b, n in zip(drawn, read, ("dq", "dk", "dv")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), n
    _check_bwd(oracle_mod, w, x, ok, read)
    # the stored flags against the oracle's mask on every visible entry
    words = mask.cpu().numpy().view(np.uint32)
    cu = x.get("cu_q")
    cu_np = None if cu is None else cu.numpy()
    for b in sorted({0, x["q"].shape[0] - 1 if cu is None else len(lengths) - 1}):
        for h in sorted({0, w.Hq - 1}):
            S_o = (w.Sq, w.Sk) if cu is None else (x["max_len"], x["max_len"])
            F = oracle_mod.dropout_factors(w.B, S_o[0], S_o[1], w.Hq, w.Hkv, w.D, b, h,
                                           cu_q=cu_np, cu_k=cu_np, **ok)
            lq, lk = F.shape
            if cu is None:
                rows = words[b, h, :lq]
            else:
                rows = words[h, int(cu_np[b]):int(cu_np[b]) + lq]
            j = np.arange(lk)
            bits = (rows[:, j // 32] >> (j % 32).astype(np.uint32)) & 1
            vis = np.ones((lq, lk), dtype=bool)
            if w.causal:
                vis = j[None, :] <= np.arange(lq)[:, None] + (lk - lq)
            assert np.array_equal(bits[vis].astype(bool), (F > 0)[vis]), (b, h)


def test_dbias_without_bias(fa, oracle_mod, cuda_device):
    w = W("dbias_only", 1, 190, 190, 2, 2, 128, causal=True)
    x, ok, gk = _case(oracle_mod, w, {})
    dbias = torch.full((w.B, w.Hq, w.Sq, w.Sk), SENTINEL, dtype=w.torch_dtype, device="cuda")
    outs = _run_bwd(fa, w, x, dict(dbias=dbias))
    _check_bwd(oracle_mod, w, x, ok, outs)
    check_bar(dbias, _oracle_dbias(oracle_mod, w, x, ok), "dbias")


VARLEN = [
    (W("vl_win_causal_d64", 3, 0, 0, 2, 2, 64, "bf16", True, varlen=(3, 1, 300)),
     [300, 77, 129], dict(window=(50, -1), seqused_q=[300, 60, 129], seqused_k=[280, 77, 0])),
    (W("vl_alibi_d128_gqa", 2, 0, 0, 4, 2, 128, "bf16", False, varlen=(2, 1, 260)),
     [260, 140], dict(alibi="bh", window=(-1, 70))),
]


@pytest.mark.parametrize("w,lengths,opt", VARLEN, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_ext_varlen(fa, oracle_mod, cuda_device, w, lengths, opt):
    x, ok, gk = _case(oracle_mod, w, opt, lengths=lengths)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale, **_kw(w, x), **gk)
    torch.cuda.synchronize()
    mq = _used_rows(w, x, ok, "q")
    check_bar(to64(o)[mq], x["o64"][mq], "o")
    lg, lr = to64(lse)[:, mq], x["lse64"][:, mq]
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert np.max(np.abs(lg[fin] - lr[fin])) < 1e-4
    _check_bwd(oracle_mod, w, x, ok, _run_bwd(fa, w, x, gk))


@pytest.mark.parametrize("D", [64, 128])
def test_ext_deterministic_window(fa, oracle_mod, cuda_device, D):
    """Deterministic order with a left window: a row block's contributions
    start at the first key block it sees, not at block 0."""
    w = W("det_win", 2, 520, 520, 4, 2, D, causal=True, deterministic=True)
    opt = dict(window=(200, -1), alibi="h")
    x, ok, gk = _case(oracle_mod, w, opt)
    a = _run_bwd(fa, w, x, gk, deterministic=True)
    b = _run_bwd(fa, w, x, gk, deterministic=True)
    for t, u in zip(a, b):
        assert torch.equal(t.view(torch.int16), u.view(torch.int16))
    _check_bwd(oracle_mod, w, x, ok, a)


def test_ext_rejects_bad_options(fa, cuda_device):
    q = torch.zeros((1, 64, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError):
        fa.fa_fwd(q, q, q, window=(-2, 0))
    with pytest.raises(fa.FaError):
        fa.fa_fwd(q, q, q, window=(0, -5))
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, alibi_slopes=torch.zeros(2, dtype=torch.float64, device="cuda"))
    bias = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError):   # a row stride that is not a multiple of 8
        fa.fa_fwd(q, q, q, bias=torch.zeros((1, 2, 64, 70), dtype=torch.bfloat16,
                                            device="cuda")[..., :64])
    qv = torch.zeros((64, 2, 64), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    with pytest.raises(fa.FaError) as e:   # bias with varlen: unsupported
        fa.fa_fwd(qv, qv, qv, cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=64,
                  max_seqlen_k=64, bias=bias)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
