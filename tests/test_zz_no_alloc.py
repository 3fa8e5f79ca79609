"""fa_sparse_mla_decode_noalloc against fa_sparse_mla_decode (GPU).

The no-allocation entry point runs the same kernels with the partial-result
workspace taken from the library's fixed scratch buffer, so its results must
equal the allocating entry point's bit for bit, on two calls in a row (the
scratch is reused without being cleared).  The file is named to be collected
last and also passes on its own.
"""
import numpy as np
import pytest
import torch

import varlen_flashattention_forward_gb300 as fa
from varlen_flashattention_forward_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(T, H, topk, context, seed):
    d = workloads.small_decode(num_tokens=T, num_heads=H, topk=topk, context=context, seed=seed)
    pt, ti = d.make_indices()
    dev = torch.device("cuda:0")
    return (d.make_q().to(dev), d.make_cache().to(dev), pt.to(dev), ti.to(dev), d.softmax_scale)


@pytest.mark.parametrize("T,H,topk,context", [
    (4, 64, 2048, 4096),   # split schedule: partial results in the scratch
    (1, 128, 1024, 2048),  # split, two head groups
    (200, 16, 128, 512),   # whole-unit schedule: no scratch used
])
def test_noalloc_matches_allocating_entry(cuda_device, T, H, topk, context):
    q, cache, pt, ti, scale = _inputs(T, H, topk, context, seed=T + H)
    ref_o, ref_l = fa.fa_sparse_mla_decode(q, cache, pt, ti, scale, return_lse=True)
    outs = []
    for _ in range(2):  # two calls in a row reuse the scratch
        out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=q.device)
        lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=q.device)
        fa.fa_sparse_mla_decode_noalloc(q, cache, pt, ti, scale, out, lse)
        outs.append((out, lse))
    torch.cuda.synchronize()
    for out, lse in outs:
        assert torch.equal(out, ref_o)
        assert torch.equal(lse, ref_l)
    assert fa.fa_get_device_status() == fa.FA_OK


def test_noalloc_rejects_split_beyond_scratch(cuda_device):
    """A call whose split needs more partial-result space than the fixed
    scratch holds returns FA_ERR_SCRATCH and writes nothing.  The planned
    workspace comes from the library's own planner: 200 units of 32 tiles
    go to the split over two waves of SMs on a GB300."""
    T, H, topk, pages = 200, 64, 2048, 32
    launches, need = fa.fa_sparse_mla_decode_plan(T, H, topk)
    if need <= fa.NOALLOC_SCRATCH_BYTES:
        pytest.skip(f"this device's split needs {need} bytes, which fits the scratch")
    dev = torch.device("cuda:0")
    q = torch.zeros((T, H, 576), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros((pages, 64, 576), dtype=torch.bfloat16, device=dev)
    pt = torch.arange(pages, dtype=torch.int32, device=dev).repeat(T, 1)
    ti = torch.arange(topk, dtype=torch.int32, device=dev).repeat(T, 1)
    out = torch.full((T, H, 512), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fa_sparse_mla_decode_noalloc(q, cache, pt, ti, 576 ** -0.5, out)
    assert e.value.status == fa.FA_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    # The allocating entry point runs the same call.
    ref = fa.fa_sparse_mla_decode(q, cache, pt, ti, 576 ** -0.5)
    torch.cuda.synchronize()
    assert torch.all(ref == 0)
