"""GPU backward (and forward, and preprocess) against the fp64 oracle, element
by element, on seeded inputs small enough for the oracle to run in full, but
spanning several tiles with ragged tails, GQA, varlen, causal with Sq != Sk,
fp16 and deterministic mode."""
import numpy as np
import pytest
import torch

from attention_backward_preprocess_gb300.workloads import WORKLOADS, Workload
from gpu_util import check_bar, oracle_grads, run_gpu_bwd, small_case, to64

pytestmark = pytest.mark.gpu


def W(name, B, Sq, Sk, Hq, Hkv, D, dtype="bf16", causal=False, **kw):
    return Workload(name, B, Sq, Sk, Hq, Hkv, D, dtype, causal, **kw)


CASES = [
    WORKLOADS["b1_h1_s128_d64"],
    W("d128_causal_ragged", 2, 200, 200, 2, 2, 128, causal=True),
    W("d128_fp16_s130", 1, 130, 130, 3, 3, 128, "fp16"),
    W("d64_causal_s257", 1, 257, 257, 2, 2, 64, causal=True),
    W("d128_gqa_causal", 1, 192, 192, 4, 2, 128, causal=True),
    W("d64_gqa3", 2, 100, 100, 6, 2, 64),
    W("d64_causal_sq_lt_sk", 1, 100, 300, 2, 2, 64, causal=True),
    W("d128_causal_sq_gt_sk", 1, 300, 100, 2, 1, 128, causal=True),
    W("s1_d64", 1, 1, 1, 1, 1, 64),
    W("s17_d128_causal", 2, 17, 17, 1, 1, 128, causal=True),
    W("d128_scale", 1, 256, 256, 2, 2, 128, scale=0.37, qk_dist=("normal", 2.0)),
    W("d64_uniform", 1, 384, 384, 2, 2, 64, vdo_dist=("uniform", 1.0)),
    # head dims between 64 and 128 run at the 128 tile width, zero-padded
    W("d96_causal_gqa", 2, 300, 300, 4, 2, 96, causal=True),
    W("d80_fp16_sq_lt_sk", 1, 200, 260, 2, 2, 80, "fp16"),
    W("d72_causal", 1, 257, 257, 2, 1, 72, causal=True),
    W("d120", 1, 130, 130, 2, 2, 120),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_oracle(fa, oracle_mod, cuda_device, w):
    x = small_case(oracle_mod, w)
    dq, dk, dv = run_gpu_bwd(fa, w, x)
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")


VARLEN = [
    (W("varlen_d64_fp16_causal", 4, 0, 0, 2, 2, 64, "fp16", True, varlen=(4, 1, 300)),
     [130, 1, 300, 64]),
    (W("varlen_d128_bf16", 2, 0, 0, 4, 2, 128, varlen=(2, 1, 200)), [200, 77]),
    (W("varlen_empty_seq", 3, 0, 0, 2, 2, 64, "bf16", True, varlen=(3, 0, 129)), [50, 0, 129]),
    (W("varlen_d128_causal_gqa", 3, 0, 0, 4, 1, 128, "bf16", True, varlen=(3, 1, 260)),
     [260, 128, 33]),
    (W("varlen_d96_causal", 2, 0, 0, 2, 2, 96, "bf16", True, varlen=(2, 1, 300)), [300, 111]),
]


@pytest.mark.parametrize("w,lengths", VARLEN, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_varlen_backward_matches_oracle(fa, oracle_mod, cuda_device, w, lengths):
    x = small_case(oracle_mod, w, lengths=lengths)
    dq, dk, dv = run_gpu_bwd(fa, w, x)
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")


@pytest.mark.parametrize("D", [64, 96, 128])
def test_deterministic_is_bit_identical_and_correct(fa, oracle_mod, cuda_device, D):
    w = W("det", 2, 300, 300, 4, 2, D, causal=True, deterministic=True)
    x = small_case(oracle_mod, w)
    a = run_gpu_bwd(fa, w, x)
    b = run_gpu_bwd(fa, w, x)
    for t, u in zip(a, b):
        assert torch.equal(t.view(torch.int16), u.view(torch.int16))
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(a[0], rq, "dq")
    check_bar(a[1], rk, "dk")
    check_bar(a[2], rv, "dv")


# D = 64 with at least 4096 keys (dense) runs in the 128-wide tile, its upper
# columns zero
LONG_D64 = [
    W("d64_s4096_causal_gqa", 1, 4096, 4096, 4, 2, 64, causal=True),
    W("d64_s4096_fp16", 1, 4096, 4096, 2, 2, 64, "fp16"),
    W("d64_s4100_det", 1, 4100, 4100, 2, 1, 64, causal=True, deterministic=True),
]


@pytest.mark.parametrize("w", LONG_D64, ids=lambda w: w.name)
def test_long_d64_matches_oracle(fa, oracle_mod, cuda_device, w):
    x = small_case(oracle_mod, w)
    dq, dk, dv = run_gpu_bwd(fa, w, x)
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(dq, rq, "dq")
    check_bar(dk, rk, "dk")
    check_bar(dv, rv, "dv")
    if w.deterministic:
        again = run_gpu_bwd(fa, w, x)
        for t, u in zip((dq, dk, dv), again):
            assert torch.equal(t.view(torch.int16), u.view(torch.int16))


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "fp16"), (96, "bf16")])
def test_dk_dv_tensor_store_and_plain_tails(fa, oracle_mod, cuda_device, D, dtype):
    """dK / dV of whole 128-key blocks leave by tensor stores, the blocks that
    end past a sequence's last key by plain stores: packed sequences of 384,
    130, 128 and 1 keys mix both, next to each other in the same rows, with
    canaries around the outputs."""
    lengths = [384, 130, 128, 1]
    w = W("store_paths", 4, 0, 0, 4, 2, D, dtype, True, varlen=(4, 1, 384))
    x = small_case(oracle_mod, w, lengths=lengths)
    pad = 4096
    outs, bufs = [], []
    for t in (x["q"], x["k"], x["v"]):
        n = t.numel()
        buf = torch.full((n + 2 * pad,), -7.0, dtype=t.dtype, device="cuda")
        bufs.append(buf)
        outs.append(buf[pad:pad + n].view(t.shape))
    run_gpu_bwd(fa, w, x, outs=outs)
    for buf in bufs:
        assert bool((buf[:pad] == -7.0).all()) and bool((buf[-pad:] == -7.0).all())
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(outs[0], rq, "dq")
    check_bar(outs[1], rk, "dk")
    check_bar(outs[2], rv, "dv")


@pytest.mark.parametrize("D", [128, 96])
def test_outputs_written_in_bounds_only(fa, oracle_mod, cuda_device, D):
    """Canary regions around dq/dk/dv stay untouched; ragged tails included
    (with D = 96, a write of the padded columns would run past the end)."""
    w = W("canary", 1, 150, 150, 2, 2, D, causal=True)
    x = small_case(oracle_mod, w)
    pad = 4096
    outs, bufs = [], []
    for t in (x["q"], x["k"], x["v"]):
        n = t.numel()
        buf = torch.full((n + 2 * pad,), -7.0, dtype=t.dtype, device="cuda")
        bufs.append(buf)
        outs.append(buf[pad:pad + n].view(t.shape))
    run_gpu_bwd(fa, w, x, outs=outs)
    for buf in bufs:
        assert bool((buf[:pad] == -7.0).all()) and bool((buf[-pad:] == -7.0).all())
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(outs[0], rq, "dq")
    check_bar(outs[1], rk, "dk")
    check_bar(outs[2], rv, "dv")


def test_caller_workspace_matches_library_workspace(fa, oracle_mod, cuda_device):
    w = W("ws", 1, 256, 256, 2, 2, 64, causal=True, deterministic=True)
    x = small_case(oracle_mod, w)
    n = fa.workspace_bytes(1, 256, 256, 2, 2, 64, deterministic=True)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    a = run_gpu_bwd(fa, w, x)
    b = run_gpu_bwd(fa, w, x, workspace=ws)
    for t, u in zip(a, b):
        assert torch.equal(t, u)


def _check_forward(o, lse, x):
    check_bar(o, to64(x["o"]), "o")
    l_gpu, l_ref = to64(lse), to64(x["lse"])
    assert np.array_equal(np.isneginf(l_gpu), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.max(np.abs(l_gpu[fin] - l_ref[fin])) < 1e-4


FWD_CASES = [
    WORKLOADS["b1_h1_s128_d64"],
    W("fwd_gqa_causal", 2, 200, 200, 4, 2, 128, causal=True),
    W("fwd_sq_gt_sk", 1, 200, 70, 2, 2, 64, "fp16", True),
    # several key blocks with a ragged last one, no mask
    W("fwd_d128_sk520", 1, 300, 520, 2, 1, 128),
    # several query tiles and key blocks under the causal mask
    W("fwd_d64_causal_s600", 1, 600, 600, 2, 2, 64, causal=True),
    # wide score range: the running maximum moves by more than 2^8 between
    # key blocks, so O and the row sum are rescaled
    W("fwd_rescale", 1, 384, 384, 2, 2, 128, scale=0.37, qk_dist=("normal", 2.0)),
    W("fwd_rescale_causal_fp16", 1, 384, 384, 2, 1, 64, "fp16", True, scale=0.5,
      qk_dist=("normal", 2.0)),
    W("fwd_s1", 1, 1, 1, 1, 1, 128),
    W("fwd_d96_causal_gqa", 2, 300, 300, 4, 2, 96, causal=True),
    W("fwd_d80_fp16", 1, 200, 260, 2, 2, 80, "fp16"),
]


@pytest.mark.parametrize("w", FWD_CASES, ids=lambda w: w.name)
def test_forward_matches_oracle(fa, oracle_mod, cuda_device, w):
    x = small_case(oracle_mod, w)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    _check_forward(o, lse, x)
    assert fa.device_status() == 0


@pytest.mark.parametrize("w,lengths", VARLEN, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_varlen_forward_matches_oracle(fa, oracle_mod, cuda_device, w, lengths):
    x = small_case(oracle_mod, w, lengths=lengths)
    cu_q, cu_k = x["cu_q"].cuda(), x["cu_k"].cuda()
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=w.causal,
                       softmax_scale=w.softmax_scale, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                       max_seqlen_q=x["max_len"], max_seqlen_k=x["max_len"])
    torch.cuda.synchronize()
    _check_forward(o, lse, x)


@pytest.mark.parametrize("w", [W("pre_d128", 2, 200, 200, 2, 2, 128, causal=True),
                               W("pre_d64_fp16", 1, 130, 130, 3, 3, 64, "fp16")],
                         ids=lambda w: w.name)
def test_preprocess_matches_oracle(fa, oracle_mod, cuda_device, w):
    """Dv = rowsum(dO o O) and LSE2 = guarded LSE * log2(e), read from the workspace."""
    x = small_case(oracle_mod, w)
    n = fa.workspace_bytes(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    lay = fa.workspace_layout(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    g = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws, causal=w.causal,
                     softmax_scale=w.softmax_scale, stages=("pre",))
    torch.cuda.synchronize()
    f = ws.view(torch.float32)
    sq_round = (w.Sq + 127) // 128 * 128
    dvec = f[lay["dvec"]:lay["dvec"] + lay["rows"]].view(w.B, w.Hq, sq_round)
    lse2 = f[lay["lse2"]:lay["lse2"] + lay["rows"]].view(w.B, w.Hq, sq_round)
    rd, rl = oracle_mod.preprocess(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["dout"]),
                                   w.softmax_scale, w.causal, o=to64(x["o"]), lse=to64(x["lse"]))
    check_bar(dvec[:, :, :w.Sq], rd, "Dv")
    assert np.max(np.abs(to64(lse2[:, :, :w.Sq]) - rl * np.log2(np.e))) < 1e-4
    assert bool(torch.isinf(lse2[:, :, w.Sq:]).all()) and bool((dvec[:, :, w.Sq:] == 0).all())
    dqacc = f[lay["dqacc"]:lay["dqacc"] + lay["rows"] * w.D]
    assert bool((dqacc == 0).all())


def test_stages_match_single_call_and_persistent_units(fa, oracle_mod, cuda_device):
    """The three stage entry points reproduce fa_bwd_with_workspace bit for bit,
    on a problem with more work units (256) than SMs, so persistent CTAs each
    process several units."""
    w = W("stages", 4, 1024, 1024, 8, 8, 128, causal=True)
    x = small_case(oracle_mod, w)
    n = fa.workspace_bytes(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    g = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    a = fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws,
                         causal=w.causal, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    b = run_gpu_bwd(fa, w, x, workspace=torch.empty_like(ws), deterministic=False)
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    for t, r, name in zip(a, (rq, rk, rv), ("dq", "dk", "dv")):
        check_bar(t, r, name)
    # dK / dV have a fixed summation order; dQ accumulates with atomics
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_main_stage_can_be_repeated(fa, oracle_mod, cuda_device):
    """The main stage hands out work units from a counter in the workspace; a
    second main stage after one preprocess must redo the same work (dK / dV
    are overwritten, dQ accumulates twice)."""
    w = W("repeat", 2, 300, 300, 4, 2, 128, causal=True)
    x = small_case(oracle_mod, w)
    n = fa.workspace_bytes(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    g = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    kw = dict(causal=w.causal, softmax_scale=w.softmax_scale)
    dq, dk, dv = fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws,
                                  stages=("pre", "main"), **kw)
    dk1, dv1 = dk.clone(), dv.clone()
    fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws, dq=dq, dk=dk,
                     dv=dv, stages=("main", "post"), **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    assert torch.equal(dk, dk1) and torch.equal(dv, dv1)
    rq, rk, rv = oracle_grads(oracle_mod, w, x)
    check_bar(dq.double() / 2, rq, "dq accumulated twice")
    check_bar(dk, rk, "dk")
