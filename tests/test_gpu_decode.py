"""GPU parity of fa_sparse_mla_decode (through the C ABI) against the fp64
oracle: max |O| error <= 2e-2 (bf16 output), max |LSE| error <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import varlen_flashattention_forward_gb300 as fa
from varlen_flashattention_forward_gb300 import workloads

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3


def run_gpu(q, cache, pt, ti, scale):
    dev = torch.device("cuda:0")
    out, lse = fa.fa_sparse_mla_decode(q.to(dev), cache.to(dev), pt.to(dev), ti.to(dev), scale,
                                       return_lse=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def compare(q, cache, pt, ti, scale, rows=None, out=None, lse=None):
    if out is None:
        out, lse = run_gpu(q, cache, pt, ti, scale)
    ref_o, ref_l = oracle.sparse_mla_decode(q, cache, pt, ti, scale, rows=rows)
    T, H, _ = out.shape
    go = out.float().numpy().reshape(T * H, 512)
    gl = lse.numpy().T.reshape(T * H)
    if rows is not None:
        go, gl = go[rows], gl[rows]
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(gl), fin)
    err_o = float(np.abs(go - ref_o).max())
    err_l = float(np.abs(gl[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert err_o <= O_TOL, f"max|dO| = {err_o}"
    assert err_l <= LSE_TOL, f"max|dLSE| = {err_l}"
    return err_o, err_l


def small_inputs(T, H, topk, context, seed, num_pages=None):
    d = workloads.small_decode(num_tokens=T, num_heads=H, topk=topk, context=context,
                               num_pages=num_pages, seed=seed)
    pt, ti = d.make_indices()
    return d.make_q(), d.make_cache(), pt, ti, d.softmax_scale


@pytest.mark.parametrize("H", [8, 16, 32, 64, 128])
def test_head_counts_elementwise(cuda_device, H):
    q, cache, pt, ti, scale = small_inputs(3, H, 256, 1024, seed=H)
    compare(q, cache, pt, ti, scale)


@pytest.mark.parametrize("topk", [128, 384, 2048])
def test_topk_sizes_elementwise(cuda_device, topk):
    q, cache, pt, ti, scale = small_inputs(2, 64, topk, 4096, seed=topk)
    compare(q, cache, pt, ti, scale)


def test_invalid_slots_are_skipped(cuda_device):
    q, cache, pt, ti, scale = small_inputs(4, 64, 256, 1024, seed=7)
    ti = ti.clone()
    ti[0, ::7] = -1                    # negative position
    ti[1, 5:40] = 1024 + 3             # past the context
    pt = pt.clone()
    pt[2, :] = -5                      # every page of token 2 out of range
    pt[3, ::3] = cache.shape[0] + 7    # some pages of token 3 past the cache
    compare(q, cache, pt, ti, scale)
    out, lse = run_gpu(q, cache, pt, ti, scale)
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[:, 2]))


def test_large_score_range_rescales(cuda_device):
    q, cache, pt, ti, scale = small_inputs(2, 64, 512, 2048, seed=9)
    q = (q.float() * 4).bfloat16()
    compare(q, cache, pt, ti, scale)


def test_bitwise_deterministic(cuda_device):
    q, cache, pt, ti, scale = small_inputs(4, 64, 512, 2048, seed=11)
    a = run_gpu(q, cache, pt, ti, scale)
    b = run_gpu(q, cache, pt, ti, scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_full_size_sampled_rows(cuda_device):
    """128 tokens, 64 heads, top-k 2048 of 32768 positions, 65536 pages."""
    d = workloads.DecodeWorkload()
    pt, ti = d.make_indices()
    q = d.make_q()
    cache = d.make_cache()
    out, lse = run_gpu(q, cache, pt, ti, d.softmax_scale)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([
        rng.integers(0, d.num_tokens * d.num_heads, size=384),
        np.arange(d.num_heads), (d.num_tokens - 1) * d.num_heads + np.arange(d.num_heads)]))
    compare(q, cache, pt, ti, d.softmax_scale, rows=rows, out=out, lse=lse)
    assert fa.fa_get_device_status() == fa.FA_OK


# Work-split schedules.  The host cuts the (token, head group) units' 64-key
# tiles into per-CTA ranges either on unit boundaries (many units) or into
# equal tile counts whose cut units are merged by their LSE (few units).
@pytest.mark.parametrize("T,H,topk,context", [
    (1, 64, 2048, 4096),    # one unit cut into 16 parts (2 tiles per CTA)
    (1, 128, 512, 1024),    # two head groups, each cut into parts
    (5, 32, 1024, 2048),    # parts of 2-3 CTAs, 32-head group
    (7, 8, 384, 1024),      # 8 heads (16-wide group), odd tile counts
])
def test_split_schedules_elementwise(cuda_device, T, H, topk, context):
    q, cache, pt, ti, scale = small_inputs(T, H, topk, context, seed=T * 1000 + H)
    compare(q, cache, pt, ti, scale)


def test_whole_unit_ranges_many_segments(cuda_device):
    """300 tokens at top-k 128: about two whole units per CTA, so every CTA
    reloads Q and hands its O accumulator over between segments."""
    q, cache, pt, ti, scale = small_inputs(300, 64, 128, 512, seed=5)
    rows = np.arange(300 * 64)
    compare(q, cache, pt, ti, scale, rows=rows[::7])


def test_split_with_invalid_part(cuda_device):
    """One part of a cut unit has no valid key (LSE -inf): its weight is 0."""
    q, cache, pt, ti, scale = small_inputs(1, 64, 2048, 4096, seed=21)
    ti = ti.clone()
    ti[0, 128:256] = -1   # tiles 2-3 (one CTA's whole range) invalid
    compare(q, cache, pt, ti, scale)


@pytest.mark.parametrize("T,H,topk,context", [(2, 64, 4096, 8192), (3, 128, 8192, 16384),
                                              (1, 16, 2176, 4096)])
def test_topk_above_one_cta_range(cuda_device, T, H, topk, context):
    # A CTA holds at most 2048 key slots: a larger top-k is always cut
    # between CTAs and merged (many parts per token).
    launches, ws = fa.fa_sparse_mla_decode_plan(T, H, topk)
    assert launches == 2 and ws > 0
    q, cache, pt, ti, scale = small_inputs(T, H, topk, context, seed=topk + T)
    compare(q, cache, pt, ti, scale)
    a = run_gpu(q, cache, pt, ti, scale)
    b = run_gpu(q, cache, pt, ti, scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_zero_tokens(cuda_device):
    dev = torch.device("cuda:0")
    q = torch.zeros((0, 64, 576), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros((4, 64, 576), dtype=torch.bfloat16, device=dev)
    pt = torch.zeros((0, 4), dtype=torch.int32, device=dev)
    ti = torch.zeros((0, 128), dtype=torch.int32, device=dev)
    out, lse = fa.fa_sparse_mla_decode(q, cache, pt, ti, 576 ** -0.5, return_lse=True)
    torch.cuda.synchronize()
    assert out.shape == (0, 64, 512)
    assert fa.fa_sparse_mla_decode_plan(0, 64, 128) == (0, 0)
    assert fa.fa_get_device_status() == fa.FA_OK
