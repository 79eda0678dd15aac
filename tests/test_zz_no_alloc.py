"""The allocation-free backward entry point, fa_bwd_noalloc.

Some callers cannot allocate device memory when they call the library (an
inference-engine plugin whose enqueue step must not allocate, a framework that
owns every byte of device memory through its own pool, a latency-critical loop
that must not enter the driver's allocator).  fa_bwd_noalloc serves them by
working in a fixed scratch array compiled into the library.  These tests call
it through the C ABI twice in a row and check each result against the regular
fa_bwd entry point within the parity tolerance, and check that a problem too
large for the fixed array is refused before anything runs.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from attention_backward_preprocess_gb300.workloads import Workload, generate
from gpu_util import check_bar


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
    Workload("noalloc_d128_gqa_causal", 2, 300, 300, 4, 2, 128, "bf16", True),
    Workload("noalloc_d64_fp16", 1, 257, 257, 3, 3, 64, "fp16", False),
    Workload("noalloc_d128_det", 1, 200, 200, 2, 2, 128, "bf16", True, deterministic=True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(fa, cuda_device, w):
    x = generate(w, "cpu", seed=11)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, causal=w.causal, softmax_scale=w.softmax_scale)
    ref = fa.fa_bwd(q, k, v, o, do, lse, causal=w.causal, softmax_scale=w.softmax_scale,
                    deterministic=w.deterministic)
    torch.cuda.synchronize()
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        st = fa.fa_bwd_noalloc(q, k, v, o, do, lse, *outs, causal=w.causal,
                               softmax_scale=w.softmax_scale, deterministic=w.deterministic)
        torch.cuda.synchronize()
        assert st == fa.FA_OK, fa.status_string(st)
        assert fa.device_status() == fa.FA_OK
        for got, want, name in zip(outs, ref, ("dq", "dk", "dv")):
            check_bar(got, want.double().cpu().numpy(), "call %d %s" % (call, name))
