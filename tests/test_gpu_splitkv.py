"""GPU parity of split-KV fa_varlen_fwd (few query tiles against long keys)
against the fp64 oracle, through the C ABI.

When the work items cannot fill the SMs, each item's key tiles are split
over a cluster of CTAs whose partial results are merged by their LSE in
distributed shared memory.  Every case first checks, through
fa_varlen_fwd_plan, that the launch really is split, then compares O and the
LSE element by element (max |dO| <= 2e-2, max |dLSE| <= 1e-3), and checks
that two runs are bitwise identical.
"""
import pytest
import torch

import varlen_flashattention_forward_gb300 as fa
from test_gpu_varlen import compare, make, run_gpu

pytestmark = pytest.mark.gpu


def plan(lens_q, lens_k, H, Hk, dqk, dv, causal=False, wl=-1, wr=-1):
    grid, split, _ = fa.fa_varlen_fwd_plan(len(lens_q), sum(lens_q), sum(lens_k), H, Hk, dqk,
                                           dv, 0, 0, causal, wl, wr)
    return grid, split


def check(lens_q, lens_k, H, Hk, dqk, dv, seed, causal=False, wl=-1, wr=-1, want_split=True):
    grid, split = plan(lens_q, lens_k, H, Hk, dqk, dv, causal, wl, wr)
    if want_split:
        assert split > 1, f"expected a split-KV launch, got grid {grid} split {split}"
    q, k, v, cq, ck = make(lens_q, lens_k, H, Hk, dqk, dv, seed=seed)
    out, lse = run_gpu(q, k, v, cq, ck, dqk ** -0.5, causal, wl, wr)
    compare(q, k, v, cq, ck, dqk ** -0.5, causal, wl, wr, out=out, lse=lse)
    out2, lse2 = run_gpu(q, k, v, cq, ck, dqk ** -0.5, causal, wl, wr)
    assert torch.equal(out, out2) and torch.equal(lse, lse2), "split-KV not bitwise deterministic"
    assert fa.fa_get_device_status() == fa.FA_OK
    return split


@pytest.mark.parametrize("dqk,dv", [(64, 64), (72, 72), (80, 80), (96, 96), (128, 128),
                                    (192, 128)])
def test_head_dims_long_keys(cuda_device, dqk, dv):
    # Two heads of one 200-row chunk against 20000 keys: two work items.
    check([200], [20000], 2, 2, dqk, dv, seed=dqk + dv, causal=True)


def test_chunk_against_64k_keys(cuda_device):
    # One 256-row chunk against 65536 keys at 16 heads (a context chunk of
    # chunked prefill: non-causal, LSE returned).
    check([256], [65536], 16, 16, 128, 128, seed=21)


def test_one_row_per_sequence_mla(cuda_device):
    # Decode-like: one query row per sequence, MLA head dims, bottom-right
    # causal, few heads so that the items leave most SMs idle.
    check([1] * 8, [32768] * 8, 8, 8, 192, 128, seed=22, causal=True)


def test_one_row_per_sequence_mla_128_heads(cuda_device):
    # The same with 128 heads: 1024 work items fill the SMs without a split.
    check([1] * 8, [32768] * 8, 128, 128, 192, 128, seed=23, causal=True, want_split=False)


def test_ragged_gqa_windows(cuda_device):
    lens_q, lens_k = [100, 3, 256, 0, 17], [20000, 5000, 9000, 10, 3000]
    check(lens_q, lens_k, 2, 1, 128, 128, seed=24, causal=True)
    check(lens_q, lens_k, 2, 1, 128, 128, seed=25, causal=True, wl=3000, wr=0)
    check(lens_q, lens_k, 2, 1, 128, 128, seed=26, wl=2000, wr=700)


def test_rows_without_keys(cuda_device):
    # q longer than k under bottom-right causal masking: the first 1000 rows
    # see no key in any part (O = 0, LSE = -inf).
    check([3000], [2000], 4, 4, 64, 64, seed=27, causal=True)


def test_split_matches_unsplit_within_rounding(cuda_device):
    # The same rows computed with and without a split (the second call has
    # enough heads to fill the SMs, so it runs unsplit) agree to rounding.
    lens_q, lens_k = [256], [30000]
    _, split = plan(lens_q, lens_k, 4, 4, 128, 128)
    _, split_many = plan(lens_q, lens_k, 128, 128, 128, 128)
    assert split > 1 and split_many == 1
    q, k, v, cq, ck = make(lens_q, lens_k, 128, 128, 128, 128, seed=28)
    o_all, l_all = run_gpu(q, k, v, cq, ck, 128 ** -0.5)
    o_4, l_4 = run_gpu(q[:, :4].contiguous(), k[:, :4].contiguous(), v[:, :4].contiguous(), cq,
                       ck, 128 ** -0.5)
    assert (o_all[:, :4].float() - o_4.float()).abs().max() <= 2e-2
    assert (l_all[:4] - l_4).abs().max() <= 1e-3
