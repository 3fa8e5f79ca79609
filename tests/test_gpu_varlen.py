"""GPU parity of fa_varlen_fwd (through the C ABI) against the fp64 oracle.

Tolerances: max |O_gpu - O_oracle| <= 2e-2 on the bf16 output and
max |LSE_gpu - LSE_oracle| <= 1e-3 on the fp32 LSE, element by element on
small cases that still span several tiles and a ragged tail, and on sampled
rows at the full workload sizes.  Results must be bitwise identical run to
run.
"""
import numpy as np
import pytest
import torch

import oracle
import varlen_flashattention_forward_gb300 as fa
from varlen_flashattention_forward_gb300 import workloads

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3


def cu(lens):
    c = [0]
    for L in lens:
        c.append(c[-1] + L)
    return torch.tensor(c, dtype=torch.int32)


def make(lens_q, lens_k, H, Hk, dqk, dv, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(sum(lens_q), H, dqk, generator=g) * std).bfloat16()
    k = (torch.randn(sum(lens_k), Hk, dqk, generator=g) * std).bfloat16()
    v = torch.randn(sum(lens_k), Hk, dv, generator=g).bfloat16()
    return q, k, v, cu(lens_q), cu(lens_k)


def run_gpu(q, k, v, cq, ck, scale, causal=False, wl=-1, wr=-1):
    dev = torch.device("cuda:0")
    out, lse = fa.fa_varlen_fwd(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev),
                                0, 0, scale, causal, wl, wr, return_lse=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def compare(q, k, v, cq, ck, scale, causal=False, wl=-1, wr=-1, rows=None, out=None, lse=None):
    if out is None:
        out, lse = run_gpu(q, k, v, cq, ck, scale, causal, wl, wr)
    ref_o, ref_l = oracle.varlen_attention(q, k, v, cq, ck, scale, causal, wl, wr, rows=rows)
    T, H, dv = out.shape
    go = out.float().numpy().reshape(T * H, dv)
    gl = lse.numpy().T.reshape(T * H)
    if rows is not None:
        go, gl = go[rows], gl[rows]
    err_o = np.abs(go - ref_o).max() if go.size else 0.0
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(gl), fin), "LSE -inf pattern differs"
    assert np.all(gl[~fin] == -np.inf)
    err_l = np.abs(gl[fin] - ref_l[fin]).max() if fin.any() else 0.0
    assert err_o <= O_TOL, f"max|dO| = {err_o}"
    assert err_l <= LSE_TOL, f"max|dLSE| = {err_l}"
    return err_o, err_l


RAGGED = [1, 63, 64, 127, 128, 129, 255, 257, 300, 513]


def test_status_word_starts_clear(cuda_device):
    assert fa.fa_get_device_status() == fa.FA_OK


def test_tiny_workload_elementwise(cuda_device):
    w = workloads.tiny()
    q, k, v, cq, ck = w.make_inputs()
    compare(q, k, v, cq, ck, w.softmax_scale)


@pytest.mark.parametrize("dqk,dv", [(64, 64), (72, 72), (80, 80), (96, 96), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims_ragged_elementwise(cuda_device, dqk, dv, causal):
    q, k, v, cq, ck = make(RAGGED, RAGGED, 2, 2, dqk, dv, seed=dqk + dv + causal)
    compare(q, k, v, cq, ck, dqk ** -0.5, causal)


def test_chunked_prefill_bottom_right(cuda_device):
    lens_q, lens_k = [5, 130, 256, 1, 200], [300, 400, 1000, 129, 200]
    q, k, v, cq, ck = make(lens_q, lens_k, 3, 3, 192, 128, seed=7)
    compare(q, k, v, cq, ck, 192 ** -0.5, causal=True)


def test_q_longer_than_k_has_empty_rows(cuda_device):
    lens_q, lens_k = [300, 40, 128], [100, 0, 1]
    q, k, v, cq, ck = make(lens_q, lens_k, 2, 2, 64, 64, seed=8)
    compare(q, k, v, cq, ck, 0.125, causal=True)
    compare(q, k, v, cq, ck, 0.125, causal=False)


def test_zero_length_sequences(cuda_device):
    lens_q, lens_k = [0, 17, 0, 140, 0], [0, 17, 5, 140, 0]
    q, k, v, cq, ck = make(lens_q, lens_k, 2, 2, 80, 80, seed=9)
    compare(q, k, v, cq, ck, 80 ** -0.5)


@pytest.mark.parametrize("wl,wr,causal", [(1024, 0, True), (100, 0, True), (127, 0, True),
                                          (128, 0, True), (50, 70, False), (0, 0, False),
                                          (-1, 5, False), (300, -1, False)])
def test_sliding_windows(cuda_device, wl, wr, causal):
    lens = [1500, 257, 64, 700]
    q, k, v, cq, ck = make(lens, lens, 2, 2, 128, 128, seed=10 + wl + wr)
    compare(q, k, v, cq, ck, 128 ** -0.5, causal, wl, wr)


@pytest.mark.parametrize("d", [64, 80])
@pytest.mark.parametrize("wl,wr,causal", [(100, 0, True), (50, 70, False), (0, 0, False)])
def test_sliding_windows_small_head_dims(cuda_device, d, wl, wr, causal):
    # d64 (P in columns of its own, S issued during the softmax) and d80 (P V
    # in two halves): window masks on boundary tiles, rows with one key.
    lens = [700, 257, 64]
    q, k, v, cq, ck = make(lens, lens, 2, 2, d, d, seed=40 + d + wl + wr)
    compare(q, k, v, cq, ck, d ** -0.5, causal, wl, wr)


def test_gqa(cuda_device):
    lens = [300, 77]
    q, k, v, cq, ck = make(lens, lens, 8, 2, 128, 128, seed=11)
    compare(q, k, v, cq, ck, 128 ** -0.5, causal=True)


@pytest.mark.parametrize("dqk,dv", [(64, 64), (80, 80), (128, 128), (192, 128)])
def test_large_scores_need_rescale(cuda_device, dqk, dv):
    """Score ranges far beyond the lazy-rescale threshold, growing along the
    key axis so the running max moves many times (d64 rescales O after the
    first half of its exponentials, the other head dims before them)."""
    lens = [1000, 600]
    q, k, v, cq, ck = make(lens, lens, 2, 2, dqk, dv, seed=12, std=3.0)
    ramp = torch.linspace(0.2, 3.0, k.shape[0])[:, None, None]
    k = (k.float() * ramp).bfloat16()
    compare(q, k, v, cq, ck, 0.5)
    compare(q, k, v, cq, ck, 0.5, causal=True)


def test_single_key_returns_v_exactly(cuda_device):
    lens = [1, 1, 1, 1]
    q, k, v, cq, ck = make(lens, lens, 4, 4, 64, 64, seed=13)
    out, lse = run_gpu(q, k, v, cq, ck, 0.125)
    assert torch.equal(out, v)


@pytest.mark.parametrize("d", [80, 128])
def test_output_only_16_byte_aligned(cuda_device, d):
    # O rows are written by bulk copies (d80), 32-byte stores when the output
    # is 32-byte aligned, and 16-byte stores otherwise: an output buffer that
    # starts 16 bytes into an allocation takes the last path (d128) and the
    # bulk-copy path with a 16-byte aligned destination (d80).
    lens = [300, 129, 64]
    q, k, v, cq, ck = make(lens, lens, 2, 2, d, d, seed=16)
    dev = torch.device("cuda:0")
    T, H = q.shape[0], q.shape[1]
    big = torch.full((T * H * d + 8,), float("nan"), dtype=torch.bfloat16, device=dev)
    out = big[8:].view(T, H, d)  # 16 bytes past a 256-byte aligned start
    assert out.data_ptr() % 32 == 16
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    fa.fa_varlen_fwd(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), 0, 0, d ** -0.5,
                     True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(big[:8].float()).all()  # nothing written before the output
    compare(q, k, v, cq, ck, d ** -0.5, causal=True, out=out.cpu(), lse=lse.cpu())


@pytest.mark.parametrize("dqk,dv,H,Hk", [(128, 128, 4, 4), (192, 128, 4, 4), (80, 80, 4, 2)])
def test_strided_views(cuda_device, dqk, dv, H, Hk):
    # V (and K) read straight out of a combined [tokens, heads, nope + v]
    # buffer, Q out of a wider buffer: row and head strides differ from the
    # dense ones, and the result must not change.
    lens_q, lens_k = [300, 129, 64], [300, 400, 64]
    g = torch.Generator().manual_seed(17)
    Tq, Tk = sum(lens_q), sum(lens_k)
    qbuf = torch.randn(Tq, H, dqk + 64, generator=g).bfloat16()
    kvbuf = torch.randn(Tk, Hk, dqk + dv, generator=g).bfloat16()
    q, k, v = qbuf[:, :, :dqk], kvbuf[:, :, :dqk], kvbuf[:, :, dqk:]
    cq, ck = cu(lens_q), cu(lens_k)
    dev = torch.device("cuda:0")
    qd, kvd = qbuf.to(dev), kvbuf.to(dev)
    out, lse = fa.fa_varlen_fwd(qd[:, :, :dqk], kvd[:, :, :dqk], kvd[:, :, dqk:], cq.to(dev),
                                ck.to(dev), 0, 0, dqk ** -0.5, True, return_lse=True)
    torch.cuda.synchronize()
    compare(q.contiguous(), k.contiguous(), v.contiguous(), cq, ck, dqk ** -0.5, causal=True,
            out=out.cpu(), lse=lse.cpu())
    # Bitwise the same as the dense call on copies.
    out2, lse2 = fa.fa_varlen_fwd(qd[:, :, :dqk].contiguous(), kvd[:, :, :dqk].contiguous(),
                                  kvd[:, :, dqk:].contiguous(), cq.to(dev), ck.to(dev), 0, 0,
                                  dqk ** -0.5, True, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out2.cpu()) and torch.equal(lse.cpu(), lse2.cpu())


@pytest.mark.parametrize("dqk,dv,H,Hk,lens_q,lens_k,want", [
    # head-group packing: 4 query heads of a K/V head share a tile, the Q
    # maps' boxes spanning heads at the strided (non-dense) head stride
    (128, 128, 8, 2, [3, 5, 1, 17], [300, 129, 64, 500], "pack"),
    (64, 64, 16, 1, [2, 9], [1000, 77], "pack"),
    # split-KV over a cluster, K and V out of the combined buffer
    (128, 128, 2, 2, [200], [20000], "split"),
    (192, 128, 2, 2, [1, 1], [9000, 12000], "split"),
])
def test_strided_views_packed_and_split(cuda_device, dqk, dv, H, Hk, lens_q, lens_k, want):
    _, split, pack = fa.fa_varlen_fwd_plan(len(lens_q), sum(lens_q), sum(lens_k), H, Hk, dqk, dv,
                                           0, 0, True)
    assert (pack > 1) if want == "pack" else (split > 1), (split, pack)
    g = torch.Generator().manual_seed(18 + dqk + H)
    Tq, Tk = sum(lens_q), sum(lens_k)
    qbuf = torch.randn(Tq, H, dqk + 32, generator=g).bfloat16()
    kvbuf = torch.randn(Tk, Hk, dqk + dv, generator=g).bfloat16()
    q, k, v = qbuf[:, :, :dqk], kvbuf[:, :, :dqk], kvbuf[:, :, dqk:]
    cq, ck = cu(lens_q), cu(lens_k)
    dev = torch.device("cuda:0")
    qd, kvd = qbuf.to(dev), kvbuf.to(dev)
    out, lse = fa.fa_varlen_fwd(qd[:, :, :dqk], kvd[:, :, :dqk], kvd[:, :, dqk:], cq.to(dev),
                                ck.to(dev), 0, 0, dqk ** -0.5, True, return_lse=True)
    torch.cuda.synchronize()
    compare(q.contiguous(), k.contiguous(), v.contiguous(), cq, ck, dqk ** -0.5, causal=True,
            out=out.cpu(), lse=lse.cpu())
    out2, lse2 = fa.fa_varlen_fwd(qd[:, :, :dqk].contiguous(), kvd[:, :, :dqk].contiguous(),
                                  kvd[:, :, dqk:].contiguous(), cq.to(dev), ck.to(dev), 0, 0,
                                  dqk ** -0.5, True, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out2.cpu()) and torch.equal(lse.cpu(), lse2.cpu())
    assert fa.fa_get_device_status() == fa.FA_OK


def test_short_segments_packed(cuda_device):
    # Runs of short segments (<= 64 rows, same token offsets in q and k) share
    # work units under a block-diagonal mask; the mix also has a long segment
    # between two runs and a zero-length one inside a run.
    lens = [64] * 9 + [5, 1, 0, 33, 64, 17] + [700] + [40] * 7 + [63, 64, 2]
    q, k, v, cq, ck = make(lens, lens, 4, 2, 80, 80, seed=18)
    compare(q, k, v, cq, ck, 80 ** -0.5)
    compare(q, k, v, cq, ck, 80 ** -0.5, causal=True)
    compare(q, k, v, cq, ck, 80 ** -0.5, wl=16, wr=8)


def test_short_segments_not_packed_when_k_differs(cuda_device):
    # Short q segments against longer k segments (chunked prefill) are not
    # packed: their rows see keys past their own q rows.
    lq, lk = [30, 50, 20], [100, 50, 64]
    q, k, v, cq, ck = make(lq, lk, 4, 4, 64, 64, seed=19)
    compare(q, k, v, cq, ck, 0.125, causal=True)
    compare(q, k, v, cq, ck, 0.125)


def test_bitwise_deterministic(cuda_device):
    w = workloads.tiny()
    lens = [3000, 50, 1200]
    q, k, v, cq, ck = make(lens, lens, 4, 4, 80, 80, seed=14)
    a = run_gpu(q, k, v, cq, ck, 80 ** -0.5, causal=True)
    b = run_gpu(q, k, v, cq, ck, 80 ** -0.5, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_max_batch_one_launch(cuda_device):
    # 2048 sequences: the largest batch one launch sorts in shared memory.
    lens = [(i * 37) % 130 for i in range(2048)]
    q, k, v, cq, ck = make(lens, lens, 1, 1, 64, 64, seed=15)
    compare(q, k, v, cq, ck, 0.125)


def test_batch_beyond_one_launch(cuda_device):
    # 5000 sequences (zero-length ones among them) run as three launches of
    # at most 2048 sequences; q shorter than k in some, so that causal rows
    # see keys from the bottom-right.
    rng = torch.Generator().manual_seed(29)
    lens_q = torch.randint(0, 40, (5000,), generator=rng).tolist()
    lens_k = [lq + int(x) for lq, x in zip(lens_q, torch.randint(0, 3, (5000,), generator=rng))]
    q, k, v, cq, ck = make(lens_q, lens_k, 2, 1, 64, 64, seed=30)
    compare(q, k, v, cq, ck, 0.125, causal=True)
    a = run_gpu(q, k, v, cq, ck, 0.125, causal=True)
    b = run_gpu(q, k, v, cq, ck, 0.125, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_many_windows_and_long_images(cuda_device):
    # Two 4K-image layers' worth of 64-token windows (2 x 700 segments, the
    # windowed layers of the sglang FA4 PR, "Speed Tests and Profiling") next
    # to two full images: 1402 segments in one launch, windows packed.
    lens = [64] * 700 + [4096] + [64] * 700 + [2000]
    q, k, v, cq, ck = make(lens, lens, 4, 4, 80, 80, seed=31, std=0.5)
    rows = sample_rows(lens, 4, 3000, seed=31)
    out, lse = run_gpu(q, k, v, cq, ck, 80 ** -0.5)
    compare(q, k, v, cq, ck, 80 ** -0.5, rows=rows, out=out, lse=lse)
    out2, lse2 = run_gpu(q, k, v, cq, ck, 80 ** -0.5)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


# ------------------------------------------------------------ full sizes
def sample_rows(lens_q, H, n, seed):
    """Boundary rows of every sequence plus random rows, all as token*H+head."""
    rng = np.random.default_rng(seed)
    toks = []
    s = 0
    for L in lens_q:
        if L:
            toks += [s, s + L - 1, s + min(L - 1, 127), s + min(L - 1, 128)]
        s += L
    toks = np.array(toks + list(rng.integers(0, s, size=n)), dtype=np.int64)
    heads = rng.integers(0, H, size=toks.shape[0])
    return np.unique(toks * H + heads)


FULL = ["vit_full_d80", "vit_full_d64", "vit_full_d72", "vit_full_d128", "vit_window_d64",
        "vit_window_d72", "vit_window_d80", "vit_window_d128", "long_16384", "long_36864",
        "long_65536", "mla_causal", "mla_chunked", "mla_swa"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(cuda_device, name):
    w = workloads.VARLEN_BENCH[name]()
    q, k, v, cq, ck = w.make_inputs()
    out, lse = run_gpu(q, k, v, cq, ck, w.softmax_scale, w.causal, *w.window)
    rows = sample_rows(w.lens_q, w.num_heads, 160, seed=len(name))
    compare(q, k, v, cq, ck, w.softmax_scale, w.causal, *w.window, rows=rows, out=out, lse=lse)
    assert fa.fa_get_device_status() == fa.FA_OK


def test_no_keys_at_all(cuda_device):
    # total_k = 0: every row has no visible key (O = 0, LSE = -inf), with and
    # without the causal mask.
    lens_q, lens_k = [5, 130, 1], [0, 0, 0]
    q, k, v, cq, ck = make(lens_q, lens_k, 2, 2, 64, 64, seed=32)
    assert k.shape[0] == 0
    for causal in (False, True):
        out, lse = run_gpu(q, k, v, cq, ck, 0.125, causal=causal)
        assert torch.all(out == 0)
        assert torch.all(lse == -float("inf"))


def test_all_sequences_empty(cuda_device):
    # total_q = 0: nothing to compute, nothing written, no error.
    q = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda:0")
    k = torch.randn((10, 2, 64), device="cuda:0").bfloat16()
    v = torch.randn((10, 2, 64), device="cuda:0").bfloat16()
    cq = torch.zeros(3, dtype=torch.int32, device="cuda:0")
    ck = torch.tensor([0, 4, 10], dtype=torch.int32, device="cuda:0")
    out, lse = fa.fa_varlen_fwd(q, k, v, cq, ck, 0, 0, 0.125, return_lse=True)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 64) and lse.shape == (2, 0)
    assert fa.fa_get_device_status() == fa.FA_OK


def _guarded(T, H, d, guard_rows, dev):
    """out [T, H, d] and lse [H, T] as views at the start of NaN-filled
    buffers with guard_rows more rows (resp. guard_rows * H more values)."""
    ob = torch.full(((T + guard_rows) * H * d,), float("nan"), dtype=torch.bfloat16, device=dev)
    lb = torch.full((H * (T + guard_rows),), float("nan"), dtype=torch.float32, device=dev)
    return ob, lb, ob[:T * H * d].view(T, H, d), lb[:H * T].view(H, T)


def test_cu_seqlens_past_the_tensors_are_clamped(cuda_device):
    # The last entries point 100 tokens past total_q / total_k: the call
    # behaves as if they ended at the tensors' ends, and writes nothing past
    # out or lse.
    T, H, d = 200, 2, 64
    q, k, v, cq, ck = make([100, 100], [100, 100], H, H, d, d, seed=33)
    bad = torch.tensor([0, 100, 300], dtype=torch.int32)
    dev = torch.device("cuda:0")
    ob, lb, out, lse = _guarded(T, H, d, 64, dev)
    fa.fa_varlen_fwd(q.to(dev), k.to(dev), v.to(dev), bad.to(dev), bad.to(dev), 0, 0, 0.125,
                     True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(ob[T * H * d:].float()).all() and torch.isnan(lb[H * T:]).all()
    compare(q, k, v, cq, ck, 0.125, causal=True, out=out.cpu(), lse=lse.cpu())
    assert fa.fa_get_device_status() == fa.FA_OK


def test_decreasing_cu_seqlens_give_empty_sequences(cuda_device):
    # cu = [0, 100, 60, 200]: sequence 1 would end before it starts (empty),
    # sequence 2 covers tokens [60, 200) and overlaps sequence 0's last 40
    # rows, whose values are then undefined.  The rows only one sequence
    # writes must match that sequence alone, and nothing is written past out.
    T, H, d = 200, 2, 64
    g = torch.Generator().manual_seed(34)
    q = torch.randn(T, H, d, generator=g).bfloat16()
    k = torch.randn(T, H, d, generator=g).bfloat16()
    v = torch.randn(T, H, d, generator=g).bfloat16()
    bad = torch.tensor([0, 100, 60, 200], dtype=torch.int32)
    dev = torch.device("cuda:0")
    ob, lb, out, lse = _guarded(T, H, d, 64, dev)
    fa.fa_varlen_fwd(q.to(dev), k.to(dev), v.to(dev), bad.to(dev), bad.to(dev), 0, 0, 0.125,
                     False, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(ob[T * H * d:].float()).all() and torch.isnan(lb[H * T:]).all()
    assert fa.fa_get_device_status() == fa.FA_OK
    out, lse = out.cpu(), lse.cpu()
    # Sequence 0 alone owns rows [0, 60), sequence 2 alone rows [100, 200).
    rows0 = np.arange(60 * H)
    compare(q[:100].contiguous(), k[:100].contiguous(), v[:100].contiguous(), cu([100]),
            cu([100]), 0.125, rows=rows0, out=out[:100], lse=lse[:, :100])
    rows2 = np.arange(40 * H, 140 * H)
    compare(q[60:].contiguous(), k[60:].contiguous(), v[60:].contiguous(), cu([140]), cu([140]),
            0.125, rows=rows2, out=out[60:], lse=lse[:, 60:].contiguous())
