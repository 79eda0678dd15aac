"""Shared helpers of the GPU parity tests.

Inputs come from the seeded generators in ``workloads``; O and LSE for the
small cases come from the ORACLE's fp64 forward (rounded to the input dtype /
fp32 as a forward kernel would store them), so the GPU backward and the
oracle backward see exactly the same tensors.  The bar is the one stated for
the method: relative L2 error <= 5e-3 and max-abs error <= 2e-2 * max|ref|
per tensor.
"""
from __future__ import annotations

import numpy as np
import torch

from attention_backward_preprocess_gb300.workloads import Workload, generate

REL_L2 = 5e-3
MAX_ABS_FRAC = 2e-2


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def check_bar(gpu, ref, what: str):
    """relative-L2 <= 5e-3 and max-abs <= 2e-2 * max|ref|; all-zero refs need exact zeros."""
    g = to64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), what + ": non-finite values"
    rmax = float(np.max(np.abs(r))) if r.size else 0.0
    if rmax == 0.0:
        assert float(np.max(np.abs(g))) == 0.0 if g.size else True, what + ": expected zeros"
        return
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    mab = float(np.max(np.abs(g - r)))
    assert rel <= REL_L2, "%s: relative L2 %.3e > %.1e" % (what, rel, REL_L2)
    assert mab <= MAX_ABS_FRAC * rmax, "%s: max abs %.3e > %.3e" % (what, mab, MAX_ABS_FRAC * rmax)


def small_case(oracle_mod, w: Workload, lengths=None, seed=0):
    """Seeded inputs + oracle-forward O / LSE, as CPU tensors.

    ``lengths`` overrides the varlen lengths (``w.varlen`` must be set)."""
    x = generate(w, "cpu", seed=seed)
    if lengths is not None:
        cu = [0]
        for L in lengths:
            cu.append(cu[-1] + L)
        total = cu[-1]
        g = torch.Generator().manual_seed(seed + 1)
        dt = w.torch_dtype
        x = dict(
            q=torch.randn((total, w.Hq, w.D), generator=g).to(dt),
            k=torch.randn((total, w.Hkv, w.D), generator=g).to(dt),
            v=torch.randn((total, w.Hkv, w.D), generator=g).to(dt),
            dout=torch.randn((total, w.Hq, w.D), generator=g).to(dt),
            cu_q=torch.tensor(cu, dtype=torch.int32), lengths=list(lengths),
            max_len=max(max(lengths), 1))
        x["cu_k"] = x["cu_q"].clone()
    cu = x.get("cu_q")
    cu_np = None if cu is None else cu.numpy()
    o64, lse64 = oracle_mod.forward(to64(x["q"]), to64(x["k"]), to64(x["v"]), w.softmax_scale,
                                    w.causal, cu_q=cu_np, cu_k=cu_np)
    x["o"] = torch.from_numpy(o64).to(w.torch_dtype)
    x["lse"] = torch.from_numpy(lse64).float()
    return x


def oracle_grads(oracle_mod, w: Workload, x):
    cu = x.get("cu_q")
    cu_np = None if cu is None else cu.numpy()
    return oracle_mod.backward(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["dout"]),
                               w.softmax_scale, w.causal, o=to64(x["o"]), lse=to64(x["lse"]),
                               cu_q=cu_np, cu_k=cu_np)


def run_gpu_bwd(fa, w: Workload, x, deterministic=None, workspace=None, outs=None):
    dev = torch.device("cuda")
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    det = w.deterministic if deterministic is None else deterministic
    kw = {}
    if "cu_q" in g:
        kw = dict(cu_seqlens_q=g["cu_q"], cu_seqlens_k=g["cu_k"], max_seqlen_q=g["max_len"],
                  max_seqlen_k=g["max_len"])
    if outs is not None:
        kw.update(dq=outs[0], dk=outs[1], dv=outs[2])
    dq, dk, dv = fa.fa_bwd(g["q"], g["k"], g["v"], g["o"], g["dout"], g["lse"], causal=w.causal,
                           softmax_scale=w.softmax_scale, deterministic=det,
                           workspace=workspace, **kw)
    torch.cuda.synchronize()
    return dq, dk, dv
