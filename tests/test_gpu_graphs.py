"""GPU: the entry points inside captured CUDA graphs.

A serving engine captures the attention calls of a decode or prefill step
once and replays the graph with new values in the same buffers (the pages'
graph runners bake the device pointers in).  Each case calls the entry point
once on the capture stream (first-call setup: function attributes, the
decode's per-stream workspace), captures one call into a graph, writes new
inputs into the same tensors, replays, and compares the replayed outputs
with the fp64 oracle on the new inputs; a second replay with other inputs
checks that nothing of the first one is carried over.
"""
import pytest
import torch

import varlen_flashattention_forward_gb300 as fa
from test_gpu_decode import compare as compare_decode
from test_gpu_decode import small_inputs
from test_gpu_varlen import compare, make

pytestmark = pytest.mark.gpu


def _varlen_graph_case(lens_q, lens_k, H, Hk, dqk, dv, causal, want_split):
    _, split, _ = fa.fa_varlen_fwd_plan(len(lens_q), sum(lens_q), sum(lens_k), H, Hk, dqk, dv,
                                        0, 0, causal)
    assert (split > 1) == want_split, split
    dev = torch.device("cuda:0")
    q0, k0, v0, cq, ck = make(lens_q, lens_k, H, Hk, dqk, dv, seed=80)
    qd, kd, vd = q0.to(dev), k0.to(dev), v0.to(dev)
    cqd, ckd = cq.to(dev), ck.to(dev)
    out = torch.empty((qd.shape[0], H, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, qd.shape[0]), dtype=torch.float32, device=dev)
    scale = dqk ** -0.5
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        fa.fa_varlen_fwd(qd, kd, vd, cqd, ckd, 0, 0, scale, causal, out=out, lse=lse)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fa.fa_varlen_fwd(qd, kd, vd, cqd, ckd, 0, 0, scale, causal, out=out, lse=lse)
    for seed in (81, 82):
        q, k, v, _, _ = make(lens_q, lens_k, H, Hk, dqk, dv, seed=seed)
        qd.copy_(q)
        kd.copy_(k)
        vd.copy_(v)
        g.replay()
        torch.cuda.synchronize()
        compare(q, k, v, cq, ck, scale, causal, out=out.cpu(), lse=lse.cpu())
    assert fa.fa_get_device_status() == fa.FA_OK


def test_varlen_in_graph(cuda_device):
    _varlen_graph_case([300, 129, 64, 1], [300, 400, 64, 77], 4, 2, 128, 128, True, False)


def test_varlen_split_kv_in_graph(cuda_device):
    # One cluster of CTAs per work item, combined in distributed shared memory.
    _varlen_graph_case([200], [20000], 2, 2, 128, 128, False, True)


def test_varlen_d64_and_mla_in_graph(cuda_device):
    _varlen_graph_case([513, 40], [513, 300], 2, 2, 64, 64, True, False)
    _varlen_graph_case([256, 33], [600, 33], 2, 2, 192, 128, True, False)


def test_decode_split_schedule_in_graph(cuda_device):
    # Few tokens: the equal-tile split over all SMs, partials in the
    # per-stream workspace (allocated by the first call), merge kernel.
    T, H, topk, context = 3, 64, 2048, 8192
    assert fa.fa_sparse_mla_decode_plan(T, H, topk)[0] == 2  # decode + merge launches
    dev = torch.device("cuda:0")
    q0, cache0, pt, ti, scale = small_inputs(T, H, topk, context, seed=83)
    qd, cached = q0.to(dev), cache0.to(dev)
    ptd, tid = pt.to(dev), ti.to(dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        fa.fa_sparse_mla_decode(qd, cached, ptd, tid, scale, out=out, lse=lse)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fa.fa_sparse_mla_decode(qd, cached, ptd, tid, scale, out=out, lse=lse)
    for seed in (84, 85):
        q, cache, _, _, _ = small_inputs(T, H, topk, context, seed=seed)
        qd.copy_(q)
        cached.copy_(cache)
        g.replay()
        torch.cuda.synchronize()
        compare_decode(q, cache, pt, ti, scale, out=out.cpu(), lse=lse.cpu())
    assert fa.fa_get_device_status() == fa.FA_OK
