"""The bounded-wait failure path on the GPU, without any fault.

Every pipeline wait inside the kernels has a time limit.  With the limit set
to a few microseconds (fa_set_wait_limit_ns, a test hook) a long call's waits
run out: the kernel must record FA_ERR_DEVICE_TIMEOUT in the device status
word, unwind (abort flag, bounded drain of its own copies and tensor-core
operations, tensor-memory release) and return, leaving the context usable,
so that the same calls with the default limit afterwards pass parity.
"""
import pytest
import torch

import varlen_flashattention_forward_gb300 as fa
from test_gpu_decode import compare as compare_decode
from test_gpu_decode import small_inputs
from test_gpu_varlen import compare, make

pytestmark = pytest.mark.gpu

SHORT_NS = 1000  # shorter than a load from HBM plus an MMA group


def _varlen_case():
    # Long enough that waits on loads from HBM and on the softmax take more
    # than the short limit: one 4096-token causal sequence and a short one.
    return make([4096, 300], [4096, 300], 4, 4, 128, 128, seed=70)


def _run_varlen(q, k, v, cq, ck, split_hint=None):
    dev = torch.device("cuda:0")
    out, lse = fa.fa_varlen_fwd(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), 0,
                                0 if split_hint is None else split_hint, 128 ** -0.5, True,
                                return_lse=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def test_wait_limit_runs_out_then_recovers(cuda_device):
    assert fa.fa_get_device_status() == fa.FA_OK
    q, k, v, cq, ck = _varlen_case()
    dq, dcache, dpt, dti, dscale = small_inputs(8, 64, 2048, 4096, seed=71)
    dev = torch.device("cuda:0")
    try:
        fa.fa_set_wait_limit_ns(SHORT_NS)
        _run_varlen(q, k, v, cq, ck)
        assert fa.fa_get_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
        # The split-KV launch (clusters, combine through distributed shared
        # memory) unwinds the same way.
        sq, sk, sv, scq, sck = make([200], [30000], 2, 2, 128, 128, seed=72)
        _, split, _ = fa.fa_varlen_fwd_plan(1, 200, 30000, 2, 2, 128, 128)
        assert split > 1
        _run_varlen(sq, sk, sv, scq, sck)
        assert fa.fa_get_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
        # Sparse-MLA decode (gather warps, split schedule and merge kernel).
        fa.fa_sparse_mla_decode(dq.to(dev), dcache.to(dev), dpt.to(dev), dti.to(dev), dscale,
                                return_lse=True)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    finally:
        fa.fa_set_wait_limit_ns(0)
    # The status word was cleared by the read; the context still works and
    # the same calls with the default limit are correct.
    assert fa.fa_get_device_status() == fa.FA_OK
    out, lse = _run_varlen(q, k, v, cq, ck)
    compare(q, k, v, cq, ck, 128 ** -0.5, True, out=out, lse=lse)
    sout, slse = _run_varlen(sq, sk, sv, scq, sck)
    compare(sq, sk, sv, scq, sck, 128 ** -0.5, True, out=sout, lse=slse)
    compare_decode(dq, dcache, dpt, dti, dscale)
    assert fa.fa_get_device_status() == fa.FA_OK
