"""The backward inside a CUDA graph: dense calls, varlen calls given their
packed totals, and the deterministic order through the stage calls issue only
launches and memsets on the stream, so they can be captured once and replayed
on new inputs written into the captured buffers.  Each replay is checked
against the fp64 oracle on that replay's inputs."""
import numpy as np
import pytest
import torch

from attention_backward_preprocess_gb300.workloads import Workload
from gpu_util import check_bar, oracle_grads, small_case

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "o", "dout", "lse")


def _capture(fn):
    fn()                         # kernels loaded, attributes set: outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def _replay_and_check(fa, oracle_mod, w, graph, bufs, outs, cases, ws):
    results = []
    for x in cases:
        for n in NAMES:
            bufs[n].copy_(x[n])
        graph.replay()
        torch.cuda.synchronize()
        assert fa.device_status(ws) == fa.FA_OK
        for t, r, name in zip(outs, oracle_grads(oracle_mod, w, x), ("dq", "dk", "dv")):
            check_bar(t, r, name)
        results.append([t.clone() for t in outs])
    return results


@pytest.mark.parametrize("D", [128, 64])
def test_dense_backward_replays_from_a_cuda_graph(fa, oracle_mod, cuda_device, D):
    w = Workload("graph_dense", 2, 300, 300, 4, 2, D, "bf16", True)
    cases = [small_case(oracle_mod, w, seed=s) for s in (0, 1)]
    bufs = {n: cases[0][n].cuda() for n in NAMES}
    outs = [torch.empty_like(bufs[n]) for n in ("q", "k", "v")]
    ws = torch.empty(fa.workspace_bytes(2, 300, 300, 4, 2, D), dtype=torch.uint8, device="cuda")
    graph = _capture(lambda: fa.fa_bwd(*(bufs[n] for n in NAMES), causal=True,
                                       softmax_scale=w.softmax_scale, workspace=ws,
                                       dq=outs[0], dk=outs[1], dv=outs[2]))
    _replay_and_check(fa, oracle_mod, w, graph, bufs, outs, cases, ws)


def test_varlen_backward_with_totals_replays_from_a_cuda_graph(fa, oracle_mod, cuda_device):
    lengths = [200, 77, 1, 130]
    w = Workload("graph_varlen", 4, 0, 0, 2, 2, 64, "fp16", True, varlen=(4, 1, 200))
    cases = [small_case(oracle_mod, w, lengths=lengths, seed=s) for s in (0, 1)]
    bufs = {n: cases[0][n].cuda() for n in NAMES}
    cu = cases[0]["cu_q"].cuda()
    T = sum(lengths)
    outs = [torch.empty_like(bufs[n]) for n in ("q", "k", "v")]
    ws = torch.empty(fa.workspace_bytes(4, 200, 200, 2, 2, 64, varlen=True), dtype=torch.uint8,
                     device="cuda")
    graph = _capture(lambda: fa.fa_bwd(*(bufs[n] for n in NAMES), causal=True,
                                       softmax_scale=w.softmax_scale, cu_seqlens_q=cu,
                                       cu_seqlens_k=cu, max_seqlen_q=200, max_seqlen_k=200,
                                       totals=(T, T), workspace=ws, dq=outs[0], dk=outs[1],
                                       dv=outs[2]))
    _replay_and_check(fa, oracle_mod, w, graph, bufs, outs, cases, ws)


def test_deterministic_stages_replay_bit_identical(fa, oracle_mod, cuda_device):
    """fa_bwd reads a deterministic call's device status back (a host wait);
    the stage calls do not, so they capture, and the status is read after the
    replay.  Two replays on the same inputs are bit-identical."""
    w = Workload("graph_det", 1, 260, 260, 4, 2, 128, "bf16", True, deterministic=True)
    cases = [small_case(oracle_mod, w, seed=s) for s in (0, 1, 0)]
    bufs = {n: cases[0][n].cuda() for n in NAMES}
    outs = [torch.empty_like(bufs[n]) for n in ("q", "k", "v")]
    ws = torch.empty(fa.workspace_bytes(1, 260, 260, 4, 2, 128, deterministic=True),
                     dtype=torch.uint8, device="cuda")
    graph = _capture(lambda: fa.fa_bwd_stages(*(bufs[n] for n in NAMES), ws, causal=True,
                                              softmax_scale=w.softmax_scale, deterministic=True,
                                              dq=outs[0], dk=outs[1], dv=outs[2]))
    res = _replay_and_check(fa, oracle_mod, w, graph, bufs, outs, cases, ws)
    for a, b in zip(res[0], res[2]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
