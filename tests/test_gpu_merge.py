"""GPU parity of fa_merge_attn_states (through the C ABI) against the oracle
merge, and the chunked-prefill use: context partial (non-causal) + new-token
partial (causal), both from fa_varlen_fwd, merged, against the fp64 oracle of
bottom-right causal attention over context + new keys."""
import numpy as np
import pytest
import torch

import oracle
import varlen_flashattention_forward_gb300 as fa

pytestmark = pytest.mark.gpu


def cu(lens):
    c = [0]
    for L in lens:
        c.append(c[-1] + L)
    return torch.tensor(c, dtype=torch.int32)


def test_merge_matches_oracle_elementwise(cuda_device):
    g = torch.Generator().manual_seed(0)
    T, H, d = 1000, 8, 128
    oa = torch.randn(T, H, d, generator=g).bfloat16()
    ob = torch.randn(T, H, d, generator=g).bfloat16()
    la = torch.randn(H, T, generator=g) * 4
    lb = torch.randn(H, T, generator=g) * 4
    la[0, :10] = -float("inf")
    lb[1, :10] = -float("inf")
    la[2, :5] = -float("inf")
    lb[2, :5] = -float("inf")
    dev = torch.device("cuda:0")
    out, lse = fa.fa_merge_attn_states(oa.to(dev), la.to(dev), ob.to(dev), lb.to(dev))
    torch.cuda.synchronize()
    ro, rl = oracle.merge_states(oa.reshape(T * H, d), la.T.reshape(-1),
                                 ob.reshape(T * H, d), lb.T.reshape(-1))
    go = out.float().cpu().numpy().reshape(T * H, d)
    gl = lse.cpu().numpy().T.reshape(-1)
    assert np.abs(go - ro).max() <= 2e-2
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.abs(gl[fin] - rl[fin]).max() <= 1e-3


def test_chunked_prefill_context_plus_new_tokens(cuda_device):
    g = torch.Generator().manual_seed(1)
    H, dqk, dv = 16, 192, 128
    lens_new, lens_ctx = [300, 129, 1000], [1000, 64, 2500]
    tn, tc = sum(lens_new), sum(lens_ctx)
    q = torch.randn(tn, H, dqk, generator=g).bfloat16()
    kn = torch.randn(tn, H, dqk, generator=g).bfloat16()
    vn = torch.randn(tn, H, dv, generator=g).bfloat16()
    kc = torch.randn(tc, H, dqk, generator=g).bfloat16()
    vc = torch.randn(tc, H, dv, generator=g).bfloat16()
    dev = torch.device("cuda:0")
    scale = dqk ** -0.5
    o_ctx, l_ctx = fa.fa_varlen_fwd(q.to(dev), kc.to(dev), vc.to(dev), cu(lens_new).to(dev),
                                    cu(lens_ctx).to(dev), 0, 0, scale, False, return_lse=True)
    o_new, l_new = fa.fa_varlen_fwd(q.to(dev), kn.to(dev), vn.to(dev), cu(lens_new).to(dev),
                                    cu(lens_new).to(dev), 0, 0, scale, True, return_lse=True)
    out, lse = fa.fa_merge_attn_states(o_ctx, l_ctx, o_new, l_new)
    torch.cuda.synchronize()
    # Full keys per sequence: its context followed by its new tokens.
    ks, vs, lk = [], [], []
    sc = sn = 0
    for lc, ln in zip(lens_ctx, lens_new):
        ks += [kc[sc:sc + lc], kn[sn:sn + ln]]
        vs += [vc[sc:sc + lc], vn[sn:sn + ln]]
        lk.append(lc + ln)
        sc += lc
        sn += ln
    rng = np.random.default_rng(0)
    rows = np.unique(rng.integers(0, tn * H, size=600))
    ro, rl = oracle.varlen_attention(q, torch.cat(ks), torch.cat(vs), cu(lens_new), cu(lk),
                                     scale, causal=True, rows=rows)
    go = out.float().cpu().numpy().reshape(tn * H, dv)[rows]
    gl = lse.cpu().numpy().T.reshape(-1)[rows]
    assert np.abs(go - ro).max() <= 2e-2
    assert np.abs(gl - rl).max() <= 1e-3
