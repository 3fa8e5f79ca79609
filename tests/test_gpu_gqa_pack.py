"""GPU parity of GQA head-group packing in fa_varlen_fwd against the fp64
oracle, through the C ABI.

With short query sequences, P query heads that share a key/value head fill
one 128-row query tile together (row r = token r / P, head r % P).  Every
case checks through fa_varlen_fwd_plan that the launch packs the expected
number of heads, then compares O and the LSE element by element (max |dO| <=
2e-2, max |dLSE| <= 1e-3), checks that two runs are bitwise identical, and
compares against the same call run unpacked (a large max_seqlen_q hint).
"""
import pytest
import torch

import varlen_flashattention_forward_gb300 as fa
from test_gpu_varlen import compare, make

pytestmark = pytest.mark.gpu


def run(q, k, v, cq, ck, scale, causal, wl, wr, q_hint):
    dev = torch.device("cuda:0")
    out, lse = fa.fa_varlen_fwd(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), q_hint,
                                0, scale, causal, wl, wr, return_lse=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def check(lens_q, lens_k, H, Hk, dqk, dv, seed, want_pack, causal=False, wl=-1, wr=-1,
          want_split=None):
    _, split, pack = fa.fa_varlen_fwd_plan(len(lens_q), sum(lens_q), sum(lens_k), H, Hk, dqk,
                                           dv, 0, 0, causal, wl, wr)
    assert pack == want_pack, f"expected {want_pack} heads per tile, got {pack}"
    if want_split is not None:
        assert (split > 1) == want_split, f"split {split}"
    _, _, pack_big = fa.fa_varlen_fwd_plan(len(lens_q), sum(lens_q), sum(lens_k), H, Hk, dqk,
                                           dv, 1 << 20, 0, causal, wl, wr)
    assert pack_big == 1
    q, k, v, cq, ck = make(lens_q, lens_k, H, Hk, dqk, dv, seed=seed)
    scale = dqk ** -0.5
    out, lse = run(q, k, v, cq, ck, scale, causal, wl, wr, 0)
    compare(q, k, v, cq, ck, scale, causal, wl, wr, out=out, lse=lse)
    out2, lse2 = run(q, k, v, cq, ck, scale, causal, wl, wr, 0)
    assert torch.equal(out, out2) and torch.equal(lse, lse2), "packed run not deterministic"
    # Unpacked: one head per tile.  Same rows, same key order; only the
    # lazy-rescale votes (taken per warp of rows) may differ, so the two agree
    # to rounding.
    out_u, lse_u = run(q, k, v, cq, ck, scale, causal, wl, wr, 1 << 20)
    assert (out.float() - out_u.float()).abs().max() <= 2e-2
    fin = torch.isfinite(lse_u)
    assert torch.equal(torch.isfinite(lse), fin)
    assert (lse[fin] - lse_u[fin]).abs().max() <= 1e-3 if fin.any() else True
    assert fa.fa_get_device_status() == fa.FA_OK


LQ = [1, 5, 17, 40, 3, 0, 9]
LK = [300, 129, 1000, 64, 2000, 7, 9]


@pytest.mark.parametrize("group", [2, 4, 8, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_group_sizes(cuda_device, group, causal):
    check(LQ, LK, 2 * group, 2, 128, 128, seed=40 + group + causal, want_pack=group,
          causal=causal)


@pytest.mark.parametrize("dqk,dv", [(64, 64), (72, 72), (80, 80), (96, 96), (192, 128)])
def test_head_dims(cuda_device, dqk, dv):
    check(LQ, LK, 8, 2, dqk, dv, seed=50 + dqk, want_pack=4, causal=True)


def test_windows(cuda_device):
    check(LQ, LK, 8, 2, 128, 128, seed=60, want_pack=4, causal=True, wl=100, wr=0)
    check(LQ, LK, 8, 2, 128, 128, seed=61, want_pack=4, wl=50, wr=20)


def test_group_wider_than_16(cuda_device):
    # 32 query heads per key/value head (MQA-like): 16 per tile, two tiles'
    # worth of heads per token.
    check(LQ, LK, 32, 1, 64, 64, seed=62, want_pack=16, causal=True)


def test_one_row_per_sequence(cuda_device):
    # Decode-like GQA: one query row per sequence, 8 heads per group.
    check([1] * 16, [4096] * 16, 32, 4, 128, 128, seed=63, want_pack=8, causal=True)


def test_tokens_spanning_two_tiles(cuda_device):
    # 60-token sequences with 4 heads per tile: 240 rows, two query tiles of
    # 32 tokens each, the second one partly beyond the sequence.
    check([60, 61, 33], [500, 61, 900], 8, 2, 128, 128, seed=64, want_pack=4, causal=True)


def test_packed_and_split(cuda_device):
    # Three query rows against 20000 keys, 8 heads per group: two packed work
    # items, split over clusters.
    check([3], [20000], 16, 2, 128, 128, seed=65, want_pack=8, causal=True, want_split=True)
