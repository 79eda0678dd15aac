"""The allocation-free backward entry point, fa_bwd_noalloc.

Some callers cannot allocate device memory when they call the library (an
inference-engine plugin whose enqueue step must not allocate, a framework that
owns every byte of device memory through its own pool, a latency-critical loop
that must not enter the driver's allocator).  fa_bwd_noalloc serves them by
working in a fixed scratch array compiled into the library.  These tests call
it through the C ABI twice in a row and check each result against the regular
fa_bwd entry point within the parity tolerance (bit for bit in deterministic
mode, where both run the same ordered reduction) and against the fp64
oracle; they read the array's own error word through fa_bwd_noalloc_status,
and check that a problem too large for the fixed array is refused before
anything runs.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from attention_backward_preprocess_gb300.workloads import Workload
from gpu_util import check_bar, oracle_grads, small_case


def test_scratch_limit_is_refused_before_any_work(fa):
    L = fa.lib()
    assert fa.noalloc_scratch_bytes() == 64 * 1024 * 1024
    need = fa.workspace_bytes(2, 8192, 8192, 32, 8, 128)
    assert need > fa.noalloc_scratch_bytes()
    vp = ctypes.c_void_p
    ptrs = [vp(0x1000 * (i + 1)) for i in range(9)]
    st = L.fa_bwd_noalloc(*ptrs, 2, 8192, 8192, 32, 8, 128, 0.088, 1, None, None, 0, 0, None)
    assert st == fa.FA_ERR_SCRATCH_LIMIT
    assert "scratch" in fa.status_string(st)


CASES = [
    (Workload("noalloc_d128_gqa_causal", 2, 300, 300, 4, 2, 128, "bf16", True), None),
    (Workload("noalloc_d64_fp16", 1, 257, 257, 3, 3, 64, "fp16", False), None),
    (Workload("noalloc_d128_det", 1, 200, 200, 2, 2, 128, "bf16", True, deterministic=True), None),
    (Workload("noalloc_varlen_d64_fp16", 3, 0, 0, 2, 2, 64, "fp16", True, varlen=(3, 1, 300)),
     [130, 1, 300]),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w,lengths", CASES, ids=lambda v: v.name if hasattr(v, "name") else "")
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(fa, oracle_mod, cuda_device, w, lengths):
    x = small_case(oracle_mod, w, lengths=lengths, seed=11)
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    q, k, v, o, do, lse = (g[n] for n in ("q", "k", "v", "o", "dout", "lse"))
    vl = {}
    if lengths is not None:
        vl = dict(cu_seqlens_q=g["cu_q"], cu_seqlens_k=g["cu_k"], max_seqlen_q=g["max_len"],
                  max_seqlen_k=g["max_len"])
    kw = dict(causal=w.causal, softmax_scale=w.softmax_scale, deterministic=w.deterministic, **vl)
    ref = fa.fa_bwd(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    want = oracle_grads(oracle_mod, w, x)
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        st = fa.fa_bwd_noalloc(q, k, v, o, do, lse, *outs, **kw)
        assert st == fa.FA_OK, fa.status_string(st)
        # the fixed array's own error word (fa_device_status reads another)
        assert fa.noalloc_status() == fa.FA_OK
        for got, same, exact, name in zip(outs, ref, want, ("dq", "dk", "dv")):
            check_bar(got, same.double().cpu().numpy(), "call %d %s against fa_bwd" % (call, name))
            check_bar(got, exact, "call %d %s against the oracle" % (call, name))
            if w.deterministic:
                assert torch.equal(got, same), "call %d %s: not bit-identical" % (call, name)
