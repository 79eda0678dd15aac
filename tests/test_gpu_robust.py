"""Failure paths and host behaviour of the real kernels on the GPU.

* A deterministic-order semaphore that can never reach its target (set from
  the host after the preprocess stage) makes the main kernel's bounded wait
  run out: the call reports FA_ERR_TIMEOUT within the short budget, the
  context stays usable, and the next call is correct.  No GPU is faulted or
  hung: the wait is bounded and the kernel winds down on its own.
* Varlen lengths that break the planned layout (a sequence longer than the
  maximum given, or packed totals above B times it) are refused; the
  sequences that fit are still computed correctly.
* Varlen calls given their packed totals return to the host without waiting
  for the stream.
"""
import time

import pytest
import torch

from attention_backward_preprocess_gb300.workloads import Workload
from gpu_util import check_bar, oracle_grads, small_case, to64

pytestmark = pytest.mark.gpu


def _gpu(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def test_main_kernel_semaphore_timeout_reports_and_recovers(fa, oracle_mod, cuda_device):
    w = Workload("timeout", 1, 256, 256, 2, 2, 128, "bf16", False, deterministic=True)
    x = small_case(oracle_mod, w)
    g = _gpu(x)
    shape = (w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D)
    ws = torch.empty(fa.workspace_bytes(*shape, deterministic=True), dtype=torch.uint8,
                     device="cuda")
    sync = fa.workspace_sync_layout(*shape, deterministic=True)
    kw = dict(causal=w.causal, softmax_scale=w.softmax_scale, deterministic=True)
    fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws, stages=("pre",),
                     **kw)
    # row block 0 of (sequence 0, head 0): its semaphore counts key blocks
    # upwards from 0, so a large negative value is never reached
    sem = ws[sync["sem"]:sync["sem"] + 4 * sync["n_sem"]].view(torch.int32)
    sem[0] = -(1 << 30)
    old = fa.set_wait_timeout_ns(50_000_000)
    try:
        t0 = time.time()
        fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws,
                         stages=("main",), **kw)
        st = fa.device_status(ws)
        dt = time.time() - t0
    finally:
        fa.set_wait_timeout_ns(old)
    assert st == fa.FA_ERR_TIMEOUT, fa.status_string(st)
    assert dt < 10.0
    # the error word was cleared by the read; the context still works
    assert fa.device_status(ws) == fa.FA_OK
    y = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float(y.sum().item()) == 28.0
    # the next calls on the same workspace are correct and bit-identical
    a = fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], workspace=ws, **kw)
    b = fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], workspace=ws, **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    for t, u in zip(a, b):
        assert torch.equal(t, u)
    for t, r, name in zip(a, oracle_grads(oracle_mod, w, x), ("dq", "dk", "dv")):
        check_bar(t, r, name)


def _varlen_case(oracle_mod, lengths, D=64, dtype="bf16", causal=True):
    w = Workload("varlen_bad", len(lengths), 0, 0, 2, 2, D, dtype, causal,
                 varlen=(len(lengths), 1, max(lengths)))
    return w, small_case(oracle_mod, w, lengths=lengths)


@pytest.mark.parametrize("det", [False, True])
def test_varlen_sequence_longer_than_max_is_refused(fa, oracle_mod, cuda_device, det):
    """max_seqlen 200 while sequence 1 has 300 rows (totals 400 <= 2 * 200
    pass the host check): the device refuses sequence 1, computes sequence 0
    correctly, and the call reports FA_ERR_INVALID_ARG."""
    w, x = _varlen_case(oracle_mod, [100, 300])
    g = _gpu(x)
    vl = dict(cu_seqlens_q=g["cu_q"], cu_seqlens_k=g["cu_k"], max_seqlen_q=200, max_seqlen_k=200)
    ws = torch.empty(fa.workspace_bytes(2, 200, 200, 2, 2, 64, varlen=True, deterministic=det),
                     dtype=torch.uint8, device="cuda")
    dq = torch.zeros_like(g["q"])
    dk = torch.zeros_like(g["k"])
    dv = torch.zeros_like(g["v"])
    kw = dict(causal=w.causal, softmax_scale=w.softmax_scale, dq=dq, dk=dk, dv=dv, workspace=ws,
              deterministic=det, **vl)
    if det:
        # deterministic calls read the error word before returning
        with pytest.raises(fa.FaError) as e:
            fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], **kw)
        assert e.value.status == fa.FA_ERR_INVALID_ARG
    else:
        fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], **kw)
    assert fa.device_status(ws) == fa.FA_ERR_INVALID_ARG
    assert fa.device_status(ws) == fa.FA_OK
    # sequence 0 is computed as if alone: one key block, so each dQ row gets a
    # single contribution and the results are bit-identical to a call on it
    ok = fa.fa_bwd(g["q"][:100], g["k"][:100], g["v"][:100], g["o"][:100], g["dout"][:100],
                   g["lse"][:, :100].contiguous(), causal=w.causal,
                   softmax_scale=w.softmax_scale, cu_seqlens_q=g["cu_q"][:2].contiguous(),
                   cu_seqlens_k=g["cu_k"][:2].contiguous(), max_seqlen_q=100, max_seqlen_k=100)
    torch.cuda.synchronize()
    assert torch.equal(dq[:100], ok[0])
    assert torch.equal(dk[:100], ok[1]) and torch.equal(dv[:100], ok[2])
    # the forward refuses the same lengths through its own error word
    fa.fa_fwd(g["q"], g["k"], g["v"], causal=w.causal, softmax_scale=w.softmax_scale, **vl)
    assert fa.device_status() == fa.FA_ERR_INVALID_ARG
    assert fa.device_status() == fa.FA_OK


def test_varlen_totals_above_the_maximum_are_refused_on_the_host(fa, oracle_mod, cuda_device):
    w, x = _varlen_case(oracle_mod, [100, 300])
    g = _gpu(x)
    vl = dict(cu_seqlens_q=g["cu_q"], cu_seqlens_k=g["cu_k"], max_seqlen_q=150,
              max_seqlen_k=150)   # totals 400 > 2 * 150
    for call in (lambda: fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"],
                                   causal=True, **vl),
                 lambda: fa.fa_fwd(g["q"], g["k"], g["v"], causal=True, **vl),
                 lambda: fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"],
                                   causal=True, totals=(400, 400), **vl)):
        with pytest.raises(fa.FaError) as e:
            call()
        assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_varlen_totals_mismatch_is_refused_on_the_device(fa, oracle_mod, cuda_device):
    """Totals given that differ from cu_seqlens[B]: nothing is touched, the
    error word says FA_ERR_INVALID_ARG."""
    w, x = _varlen_case(oracle_mod, [100, 60])
    g = _gpu(x)
    vl = dict(cu_seqlens_q=g["cu_q"], cu_seqlens_k=g["cu_k"], max_seqlen_q=100, max_seqlen_k=100)
    ws = torch.empty(fa.workspace_bytes(2, 100, 100, 2, 2, 64, varlen=True), dtype=torch.uint8,
                     device="cuda")
    dq = torch.full_like(g["q"], 3.0)
    fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], causal=True, workspace=ws,
              dq=dq, totals=(150, 160), **vl)
    assert fa.device_status(ws) == fa.FA_ERR_INVALID_ARG
    assert bool((dq == 3.0).all())


@pytest.mark.parametrize("which", ["bwd", "fwd", "stages"])
def test_varlen_call_with_totals_does_not_wait_for_the_stream(fa, oracle_mod, cuda_device, which):
    lengths = [130, 1, 300, 64]
    w, x = _varlen_case(oracle_mod, lengths, dtype="fp16")
    g = _gpu(x)
    T = sum(lengths)
    vl = dict(cu_seqlens_q=g["cu_q"], cu_seqlens_k=g["cu_k"], max_seqlen_q=300,
              max_seqlen_k=300, totals=(T, T))
    ws = torch.empty(fa.workspace_bytes(4, 300, 300, 2, 2, 64, varlen=True), dtype=torch.uint8,
                     device="cuda")
    kw = dict(causal=w.causal, softmax_scale=w.softmax_scale)

    def call():
        if which == "bwd":
            return fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], workspace=ws,
                             **kw, **vl)
        if which == "stages":
            # the three stages as separate calls (fa_bwd_stages_ext)
            out = None
            for st in ("pre", "main", "post"):
                out = fa.fa_bwd_stages(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], ws,
                                       stages=(st,), dq=out[0] if out else None,
                                       dk=out[1] if out else None, dv=out[2] if out else None,
                                       **kw, **vl)
            return out
        return fa.fa_fwd(g["q"], g["k"], g["v"], **kw, **vl)

    call()                      # first use of the kernels (module loading) outside the timing
    torch.cuda.synchronize()
    torch.cuda._sleep(1_000_000_000)   # keeps the stream busy for about half a second
    t0 = time.perf_counter()
    out = call()
    t_call = time.perf_counter() - t0
    torch.cuda.synchronize()
    t_all = time.perf_counter() - t0
    assert t_all > 0.2, "the sleep kernel did not hold the stream"
    assert t_call < 0.25 * t_all, (t_call, t_all)
    if which in ("bwd", "stages"):
        assert fa.device_status(ws) == fa.FA_OK
        for t, r, name in zip(out, oracle_grads(oracle_mod, w, x), ("dq", "dk", "dv")):
            check_bar(t, r, name)
    else:
        assert fa.device_status() == fa.FA_OK
        check_bar(out[0], to64(x["o"]), "o")
