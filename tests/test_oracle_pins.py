"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties the oracle to a library routine, a closed form, an invariant
or a hand-enumerated golden case, chosen so that a plausible slip in the
oracle (a dropped scale, a wrong sign or offset in a mask, transposed
operands, a wrong head mapping, a wrong LSE base, a wrong gather) fails at
least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return x.to(torch.bfloat16)


def randn_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return bf16(torch.randn(shape, generator=g) * std)


def cu(lens):
    c = [0]
    for L in lens:
        c.append(c[-1] + L)
    return torch.tensor(c, dtype=torch.int32)


def run(q, k, v, lens_q, lens_k, scale, causal=False, wl=-1, wr=-1):
    out, lse = oracle.varlen_attention(q, k, v, cu(lens_q), cu(lens_k), scale,
                                       causal, wl, wr)
    T, H = q.shape[0], q.shape[1]
    return out.reshape(T, H, -1), lse.reshape(T, H)


def seq_slices(lens):
    s = 0
    for L in lens:
        yield slice(s, s + L)
        s += L


# ------------------------------------------------------------ library pins
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_square(causal):
    """Lq == Lk: fp64 SDPA (full or top-left causal, identical when square)."""
    lens = [3, 7, 12]
    H, d = 2, 8
    q = randn_bf16((sum(lens), H, d), 1)
    k = randn_bf16((sum(lens), H, d), 2)
    v = randn_bf16((sum(lens), H, d), 3)
    scale = 0.37
    out, lse = run(q, k, v, lens, lens, scale, causal)
    for sl in seq_slices(lens):
        qs, ks, vs = (t[sl].double().transpose(0, 1) for t in (q, k, v))
        ref = F.scaled_dot_product_attention(qs, ks, vs, is_causal=causal, scale=scale)
        np.testing.assert_allclose(out[sl], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        scores = scale * qs @ ks.transpose(-1, -2)
        if causal:
            L = scores.shape[-1]
            scores = scores.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), -math.inf)
        ref_lse = torch.logsumexp(scores, dim=-1).transpose(0, 1)
        np.testing.assert_allclose(lse[sl], ref_lse.numpy(), rtol=0, atol=1e-12)


def test_bottom_right_causal_matches_torch_causal_lower_right():
    """Lq < Lk: torch's lower-right causal bias is the bottom-right diagonal."""
    from torch.nn.attention.bias import causal_lower_right
    lens_q, lens_k = [2, 5, 9], [6, 5, 20]
    H, d = 3, 16
    q = randn_bf16((sum(lens_q), H, d), 4)
    k = randn_bf16((sum(lens_k), H, d), 5)
    v = randn_bf16((sum(lens_k), H, d), 6)
    scale = d ** -0.5
    out, _ = run(q, k, v, lens_q, lens_k, scale, causal=True)
    for sq, sk, lq, lk in zip(seq_slices(lens_q), seq_slices(lens_k), lens_q, lens_k):
        qs = q[sq].double().transpose(0, 1)
        ks, vs = (t[sk].double().transpose(0, 1) for t in (k, v))
        ref = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=causal_lower_right(lq, lk),
                                             scale=scale)
        np.testing.assert_allclose(out[sq], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def test_gqa_head_mapping_matches_repeated_heads():
    """H_k < H: query head h reads kv head h // (H / H_k) (library repeat)."""
    lens = [5, 11]
    H, Hk, d = 6, 2, 8
    q = randn_bf16((sum(lens), H, d), 7)
    k = randn_bf16((sum(lens), Hk, d), 8)
    v = randn_bf16((sum(lens), Hk, 12), 9)
    out, _ = run(q, k, v, lens, lens, 0.5)
    for sl in seq_slices(lens):
        qs = q[sl].double().transpose(0, 1)
        ks = k[sl].double().transpose(0, 1).repeat_interleave(H // Hk, dim=0)
        vs = v[sl].double().transpose(0, 1).repeat_interleave(H // Hk, dim=0)
        ref = F.scaled_dot_product_attention(qs, ks, vs, scale=0.5)
        np.testing.assert_allclose(out[sl], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def test_different_qk_and_v_dims_match_sdpa():
    """d_qk = 192, d_v = 128 (the MLA shapes): SDPA with different head dims."""
    lens = [9, 4]
    H = 2
    q = randn_bf16((sum(lens), H, 192), 10)
    k = randn_bf16((sum(lens), H, 192), 11)
    v = randn_bf16((sum(lens), H, 128), 12)
    scale = 192 ** -0.5
    out, _ = run(q, k, v, lens, lens, scale, causal=True)
    for sl in seq_slices(lens):
        qs, ks, vs = (t[sl].double().transpose(0, 1) for t in (q, k, v))
        ref = F.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=scale)
        np.testing.assert_allclose(out[sl], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------------ golden masks
def load_mask_cases():
    with open(os.path.join(GOLDEN, "masks.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", load_mask_cases(), ids=lambda c: f"{c['lq']}x{c['lk']}"
                         f"{'c' if c['causal'] else ''}w{c['window'][0]}_{c['window'][1]}")
def test_golden_visible_key_sets(case):
    """Q = 0 makes every visible score equal, so with V = one-hot(key index)
    O[i] is the uniform distribution over the visible set and exp(LSE) is its
    size.  This pins the whole mask row by row against hand enumeration."""
    lq, lk = case["lq"], case["lk"]
    wl, wr = case["window"]
    q = torch.zeros((lq, 1, 8), dtype=torch.bfloat16)
    k = randn_bf16((lk, 1, 8), 13)
    v = bf16(torch.eye(max(lk, 1))[:lk].reshape(lk, 1, max(lk, 1)))
    out, lse = run(q, k, v, [lq], [lk], 1.0, case["causal"], wl, wr)
    for i, visible in enumerate(case["rows"]):
        expect = np.zeros(max(lk, 1))
        if visible:
            expect[visible] = 1.0 / len(visible)
            assert math.isclose(math.exp(lse[i, 0]), len(visible), rel_tol=1e-12)
        else:
            assert lse[i, 0] == -math.inf
        np.testing.assert_allclose(out[i, 0], expect, rtol=0, atol=1e-15)


def test_metrics_visible_key_counts_match_golden():
    """The FLOP counter's closed-form counts agree with the golden sets."""
    from varlen_flashattention_forward_gb300.metrics import visible_keys_per_row
    for case in load_mask_cases():
        got = visible_keys_per_row(case["lq"], case["lk"], case["causal"], *case["window"])
        assert list(got) == [len(r) for r in case["rows"]]


# ------------------------------------------------------------ closed forms
def test_single_key_returns_v_exactly():
    lens = [1, 1, 1]
    H, d = 4, 64
    q = randn_bf16((3, H, d), 14)
    k = randn_bf16((3, H, d), 15)
    v = randn_bf16((3, H, d), 16)
    out, lse = run(q, k, v, lens, lens, 0.125)
    np.testing.assert_array_equal(out, v.double().numpy())
    score = 0.125 * (q.double() * k.double()).sum(-1)
    np.testing.assert_allclose(lse, score.numpy(), rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_values():
    lens = [6, 17]
    H, d = 2, 16
    q = torch.zeros((sum(lens), H, d), dtype=torch.bfloat16)
    k = randn_bf16((sum(lens), H, d), 17)
    v = randn_bf16((sum(lens), H, 24), 18)
    out, lse = run(q, k, v, lens, lens, 0.3)
    for sl, L in zip(seq_slices(lens), lens):
        mean = v[sl].double().mean(0).numpy()
        np.testing.assert_allclose(out[sl], np.broadcast_to(mean, out[sl].shape), atol=1e-13)
        np.testing.assert_allclose(np.exp(lse[sl]), L, rtol=1e-13)


def test_all_ones_values_give_ones():
    lens = [5, 33]
    q = randn_bf16((sum(lens), 2, 8), 19, 3.0)
    k = randn_bf16((sum(lens), 2, 8), 20, 3.0)
    v = torch.ones((sum(lens), 2, 8), dtype=torch.bfloat16)
    for causal, wl, wr in [(False, -1, -1), (True, -1, -1), (True, 3, 0), (False, 2, 2)]:
        out, _ = run(q, k, v, lens, lens, 0.9, causal, wl, wr)
        np.testing.assert_allclose(out, 1.0, atol=1e-13)


def test_causal_first_row_is_first_value():
    lens = [7, 20]
    q = randn_bf16((sum(lens), 3, 16), 21)
    k = randn_bf16((sum(lens), 3, 16), 22)
    v = randn_bf16((sum(lens), 3, 16), 23)
    out, _ = run(q, k, v, lens, lens, 0.25, causal=True)
    for sl in seq_slices(lens):
        np.testing.assert_array_equal(out[sl.start], v[sl.start].double().numpy())


def test_two_keys_closed_form():
    """Two keys: O = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1."""
    q = randn_bf16((1, 1, 4), 24)
    k = randn_bf16((2, 1, 4), 25)
    v = randn_bf16((2, 1, 4), 26)
    out, lse = run(q, k, v, [1], [2], 0.7)
    s = [0.7 * float((q[0, 0].double() * k[j, 0].double()).sum()) for j in range(2)]
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    ref = w0 * v[0, 0].double().numpy() + (1 - w0) * v[1, 0].double().numpy()
    np.testing.assert_allclose(out[0, 0], ref, atol=1e-14)
    assert math.isclose(lse[0, 0], math.log(math.exp(s[0]) + math.exp(s[1])), rel_tol=1e-13)


# ------------------------------------------------------------ invariants
def test_convex_hull_and_lse_bounds():
    lens = [40, 3]
    H, d = 2, 32
    q = randn_bf16((sum(lens), H, d), 27, 2.0)
    k = randn_bf16((sum(lens), H, d), 28, 2.0)
    v = randn_bf16((sum(lens), H, d), 29)
    scale = d ** -0.5
    out, lse = run(q, k, v, lens, lens, scale, causal=True)
    for sl in seq_slices(lens):
        for i in range(sl.stop - sl.start):
            keys = slice(sl.start, sl.start + i + 1)
            vv = v[keys].double()
            assert np.all(out[sl.start + i] >= vv.min(0).values.numpy() - 1e-12)
            assert np.all(out[sl.start + i] <= vv.max(0).values.numpy() + 1e-12)
            s = scale * (q[sl.start + i].double()[None] * k[keys].double()).sum(-1)
            smax = s.max(0).values.numpy()
            assert np.all(lse[sl.start + i] >= smax - 1e-12)
            assert np.all(lse[sl.start + i] <= smax + math.log(i + 1) + 1e-12)


def test_noncausal_invariant_to_key_permutation():
    L = 23
    q = randn_bf16((L, 2, 8), 30)
    k = randn_bf16((L, 2, 8), 31)
    v = randn_bf16((L, 2, 8), 32)
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(0))
    a, la = run(q, k, v, [L], [L], 0.5)
    b, lb = run(q, k[perm].contiguous(), v[perm].contiguous(), [L], [L], 0.5)
    np.testing.assert_allclose(a, b, atol=1e-13)
    np.testing.assert_allclose(la, lb, atol=1e-13)


def test_packed_equals_each_sequence_alone():
    lens_q, lens_k = [4, 0, 9, 13], [7, 3, 9, 20]
    q = randn_bf16((sum(lens_q), 2, 16), 33)
    k = randn_bf16((sum(lens_k), 2, 16), 34)
    v = randn_bf16((sum(lens_k), 2, 16), 35)
    packed, lp = run(q, k, v, lens_q, lens_k, 0.25, causal=True, wl=5, wr=0)
    for sq, sk, lq, lk in zip(seq_slices(lens_q), seq_slices(lens_k), lens_q, lens_k):
        if lq == 0:
            continue
        alone, la = run(q[sq].contiguous(), k[sk].contiguous(), v[sk].contiguous(), [lq], [lk],
                        0.25, causal=True, wl=5, wr=0)
        np.testing.assert_array_equal(packed[sq], alone)
        np.testing.assert_array_equal(lp[sq], la)


def test_window_equivalences():
    lens = [19, 31]
    q = randn_bf16((sum(lens), 2, 8), 36)
    k = randn_bf16((sum(lens), 2, 8), 37)
    v = randn_bf16((sum(lens), 2, 8), 38)
    full, lf = run(q, k, v, lens, lens, 0.4)
    wide, lw = run(q, k, v, lens, lens, 0.4, wl=100, wr=100)
    np.testing.assert_array_equal(full, wide)
    np.testing.assert_array_equal(lf, lw)
    causal, lc = run(q, k, v, lens, lens, 0.4, causal=True)
    right0, lr = run(q, k, v, lens, lens, 0.4, wl=-1, wr=0)
    np.testing.assert_array_equal(causal, right0)
    np.testing.assert_array_equal(lc, lr)


def test_rows_without_visible_keys_are_zero_with_minus_inf_lse():
    lens_q, lens_k = [5, 3], [2, 0]
    q = randn_bf16((8, 1, 8), 39)
    k = randn_bf16((2, 1, 8), 40)
    v = randn_bf16((2, 1, 8), 41)
    out, lse = run(q, k, v, lens_q, lens_k, 1.0, causal=True)
    # sequence 0: off = -3, rows 0..2 see nothing; sequence 1: no keys at all
    for t in [0, 1, 2, 5, 6, 7]:
        assert lse[t, 0] == -math.inf
        np.testing.assert_array_equal(out[t, 0], 0.0)
    assert np.isfinite(lse[3, 0]) and np.isfinite(lse[4, 0])


def test_row_subset_matches_full_run():
    lens = [30, 50]
    q = randn_bf16((80, 4, 16), 42)
    k = randn_bf16((80, 4, 16), 43)
    v = randn_bf16((80, 4, 16), 44)
    full, lf = oracle.varlen_attention(q, k, v, cu(lens), cu(lens), 0.25, True)
    rows = np.array([0, 5, 77, 200, 319], dtype=np.int64)
    sub, ls = oracle.varlen_attention(q, k, v, cu(lens), cu(lens), 0.25, True, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(ls, lf[rows])


# ------------------------------------------------------------ decode
def _identity_decode(T, H, ctx, seed):
    q = randn_bf16((T, H, 576), seed)
    pages = ctx // 64
    cache = randn_bf16((T * pages, 64, 576), seed + 1)
    page_table = torch.arange(T * pages, dtype=torch.int32).view(T, pages)
    return q, cache, page_table


def test_decode_equals_dense_mqa_over_whole_context():
    """topk = every position, identity pages: dense non-causal attention with
    one shared kv head, d_qk = 576 and d_v = 512."""
    T, H, ctx = 3, 4, 128
    q, cache, page_table = _identity_decode(T, H, ctx, 50)
    topk = torch.arange(ctx, dtype=torch.int32).repeat(T, 1)
    out, lse = oracle.sparse_mla_decode(q, cache, page_table, topk, 1 / 24)
    rows = cache.view(T, ctx, 576)
    for t in range(T):
        ks = rows[t].double()
        qs = q[t].double()
        ref = F.scaled_dot_product_attention(qs[None], ks[None], ks[None, :, :512], scale=1 / 24)[0]
        np.testing.assert_allclose(out.reshape(T, H, 512)[t], ref.numpy(), atol=1e-12)
        ref_lse = torch.logsumexp(qs @ ks.T / 24, dim=-1)
        np.testing.assert_allclose(lse.reshape(T, H)[t], ref_lse.numpy(), atol=1e-12)


def test_decode_page_translation_and_slot_order():
    """Scrambled physical pages with a matching page table give the same
    result as the identity layout; the slot order does not matter."""
    T, H, ctx = 2, 8, 256
    q, cache, page_table = _identity_decode(T, H, ctx, 60)
    g = torch.Generator().manual_seed(1)
    topk = torch.stack([torch.randperm(ctx, generator=g)[:128] for _ in range(T)]).int()
    a, la = oracle.sparse_mla_decode(q, cache, page_table, topk, 0.05)
    perm = torch.randperm(cache.shape[0], generator=g)        # new physical position of page p
    cache2 = torch.empty_like(cache)
    cache2[perm] = cache
    page_table2 = perm[page_table.long()].int()
    b, lb = oracle.sparse_mla_decode(q, cache2, page_table2, topk, 0.05)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    shuffled = topk[:, torch.randperm(128, generator=g)].contiguous()
    c, lc = oracle.sparse_mla_decode(q, cache, page_table, shuffled, 0.05)
    np.testing.assert_allclose(a, c, atol=1e-13)
    np.testing.assert_allclose(la, lc, atol=1e-13)


def test_decode_skips_out_of_range_slots():
    T, H, ctx = 2, 2, 128
    q, cache, page_table = _identity_decode(T, H, ctx, 70)
    topk = torch.arange(128, dtype=torch.int32).repeat(T, 1)
    ref, lref = oracle.sparse_mla_decode(q, cache, page_table, topk[:, :100].contiguous(), 0.1)
    bad = topk.clone()
    bad[:, 100:] = torch.tensor([-1, ctx, ctx + 5, -7] * 7)[:28].int()
    got, lgot = oracle.sparse_mla_decode(q, cache, page_table, bad, 0.1)
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(lgot, lref)


# ------------------------------------------------------------ merge
def test_merge_of_context_and_new_tokens_equals_full_chunked_prefill():
    """Chunked prefill split: non-causal attention over the context keys,
    causal attention over the new tokens' own keys, merged by LSE, equals
    bottom-right causal attention over context + new keys (a decomposition
    identity; the oracle's full run is itself pinned to SDPA above)."""
    Lc, Ln, H, d = 37, 21, 3, 16
    q = randn_bf16((Ln, H, d), 80)
    kc, vc = randn_bf16((Lc, H, d), 81), randn_bf16((Lc, H, d), 82)
    kn, vn = randn_bf16((Ln, H, d), 83), randn_bf16((Ln, H, d), 84)
    scale = 0.3
    o_ctx, l_ctx = oracle.varlen_attention(q, kc, vc, cu([Ln]), cu([Lc]), scale, causal=False)
    o_new, l_new = oracle.varlen_attention(q, kn, vn, cu([Ln]), cu([Ln]), scale, causal=True)
    merged, lm = oracle.merge_states(o_ctx, l_ctx, o_new, l_new)
    k_all, v_all = torch.cat([kc, kn]), torch.cat([vc, vn])
    full, lf = oracle.varlen_attention(q, k_all, v_all, cu([Ln]), cu([Lc + Ln]), scale,
                                       causal=True)
    np.testing.assert_allclose(merged, full, atol=1e-13)
    np.testing.assert_allclose(lm, lf, atol=1e-13)


def test_merge_with_empty_parts():
    rng = np.random.default_rng(0)
    o = rng.normal(size=(4, 8))
    lse = np.array([0.3, -1.0, 2.0, 5.0])
    empty_o, empty_l = np.zeros((4, 8)), np.full(4, -np.inf)
    a, la = oracle.merge_states(o, lse, empty_o, empty_l)
    np.testing.assert_array_equal(a, o)
    np.testing.assert_array_equal(la, lse)
    b, lb = oracle.merge_states(empty_o, empty_l, empty_o, empty_l)
    np.testing.assert_array_equal(b, 0.0)
    assert np.all(np.isneginf(lb))
    c, lc = oracle.merge_states(o, lse, o, lse)     # equal halves: same O, LSE + ln 2
    np.testing.assert_allclose(c, o, atol=1e-15)
    np.testing.assert_allclose(lc, lse + math.log(2.0), atol=1e-15)
