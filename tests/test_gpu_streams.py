"""GPU: calls on several streams at once.

The decode's split schedule keeps its partial results in a workspace owned by
the stream the call runs on, so that calls on different streams never share
one.  Here two split decodes, and two varlen calls (one of them a split-KV
cluster launch), are issued on two streams without synchronising between
them, so that their kernels can overlap; each result must match the oracle.
"""
import pytest
import torch

import varlen_flashattention_forward_gb300 as fa
from test_gpu_decode import compare as compare_decode
from test_gpu_decode import small_inputs
from test_gpu_varlen import compare, make

pytestmark = pytest.mark.gpu


def test_split_decodes_on_two_streams(cuda_device):
    T, H, topk, context = 3, 64, 2048, 8192
    assert fa.fa_sparse_mla_decode_plan(T, H, topk)[1] > 0  # uses the workspace
    dev = torch.device("cuda:0")
    cases = [small_inputs(T, H, topk, context, seed=s) for s in (90, 91)]
    streams = [torch.cuda.Stream(device=dev) for _ in cases]
    dev_in, outs = [], []
    for (q, cache, pt, ti, scale), s in zip(cases, streams):
        dev_in.append((q.to(dev), cache.to(dev), pt.to(dev), ti.to(dev), scale))
    torch.cuda.synchronize()
    for rep in range(3):  # the first round allocates each stream's workspace
        outs = []
        for (q, cache, pt, ti, scale), s in zip(dev_in, streams):
            with torch.cuda.stream(s):
                outs.append(fa.fa_sparse_mla_decode(q, cache, pt, ti, scale, return_lse=True))
        torch.cuda.synchronize()
    for (q, cache, pt, ti, scale), (out, lse) in zip(cases, outs):
        compare_decode(q, cache, pt, ti, scale, out=out.cpu(), lse=lse.cpu())
    assert fa.fa_get_device_status() == fa.FA_OK


def test_varlen_on_two_streams(cuda_device):
    dev = torch.device("cuda:0")
    shapes = [([300, 129, 64], [300, 400, 64], 4, 2, 128, 128, True),
              ([200], [20000], 2, 2, 128, 128, False)]  # the second one split-KV
    assert fa.fa_varlen_fwd_plan(1, 200, 20000, 2, 2, 128, 128)[1] > 1
    cases = [make(lq, lk, H, Hk, dqk, dv, seed=92 + i)
             for i, (lq, lk, H, Hk, dqk, dv, _) in enumerate(shapes)]
    streams = [torch.cuda.Stream(device=dev) for _ in cases]
    dev_in = [tuple(t.to(dev) for t in c) for c in cases]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        outs = []
        for (q, k, v, cq, ck), s, sh in zip(dev_in, streams, shapes):
            with torch.cuda.stream(s):
                outs.append(fa.fa_varlen_fwd(q, k, v, cq, ck, 0, 0, sh[4] ** -0.5, sh[6],
                                             return_lse=True))
        torch.cuda.synchronize()
    for (q, k, v, cq, ck), (out, lse), sh in zip(cases, outs, shapes):
        compare(q, k, v, cq, ck, sh[4] ** -0.5, sh[6], out=out.cpu(), lse=lse.cpu())
    assert fa.fa_get_device_status() == fa.FA_OK
