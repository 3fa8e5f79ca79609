"""Seeded synthetic workloads: shapes and input generators, nothing else.

This module holds no attention arithmetic.  It only states the shapes of the
benchmark/parity workloads and draws their inputs from seeded CPU
``torch.Generator`` streams, so the same host bytes feed both the CUDA path
and the fp64 oracle.

Workload shapes (taken from the pages' workloads; synthetic data stands in
for the images, models and caches named there):
  tiny          3 sequences [17, 64, 100], 4 heads, d=64, N(0,1), scale 1/8.
  vit_full      ViT encoder, packed images [576, 1024, 2304, 4096, 256, 9216],
                16 heads, d in {64, 72, 80, 128}, non-causal, Q and K scaled by
                0.5, V ~ N(0,1) (sglang PR #41344, "Speed Tests and Profiling":
                ViT shapes with head dims 64/72/80/128, 16 heads).
  vit_window    the same tensors split into consecutive 256-token windows,
                each window its own cu_seqlens segment (576 -> 256+256+64).
  long_L        one image of L in {16384, 36864, 65536} tokens, 16 heads,
                d=128, N(0,1), returning LSE.
  mla_causal    MLA prefill, 4 x 4096 tokens, 128 heads, d_qk=192 (128 nope +
                64 rope), d_v=128, causal (vLLM flash_attn page,
                FlashAttnPrefillBackend.run_prefill_new_tokens).
  mla_chunked   q lengths [2048, 2048] against k lengths [8192, 8192],
                bottom-right causal (chunked prefill, q shorter than k).
  mla_swa       mla_causal with a sliding window (1024, 0).
  decode        sparse-MLA decode: 128 tokens, each with its own context of
                32768 positions = 512 pages of 64 (physical pages: a seeded
                permutation of 0..65535), 64 heads, 576-wide rows, top-k 2048
                distinct positions per token, scale 1/sqrt(576).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Tuple

import torch

VIT_LENGTHS = [576, 1024, 2304, 4096, 256, 9216]


@dataclass
class VarlenWorkload:
    name: str
    lens_q: List[int]
    lens_k: List[int]
    num_heads: int
    num_heads_k: int
    d_qk: int
    d_v: int
    softmax_scale: float
    causal: bool = False
    window: Tuple[int, int] = (-1, -1)
    qk_std: float = 1.0
    v_std: float = 1.0
    seed: int = 0
    return_lse: bool = True

    @property
    def total_q(self) -> int:
        return sum(self.lens_q)

    @property
    def total_k(self) -> int:
        return sum(self.lens_k)

    def cu_seqlens(self) -> Tuple[torch.Tensor, torch.Tensor]:
        cq = torch.zeros(len(self.lens_q) + 1, dtype=torch.int32)
        ck = torch.zeros(len(self.lens_k) + 1, dtype=torch.int32)
        cq[1:] = torch.cumsum(torch.tensor(self.lens_q, dtype=torch.int64), 0).to(torch.int32)
        ck[1:] = torch.cumsum(torch.tensor(self.lens_k, dtype=torch.int64), 0).to(torch.int32)
        return cq, ck

    def make_inputs(self):
        """(q, k, v, cu_q, cu_k) on the CPU; q,k,v bf16."""
        g = torch.Generator(device="cpu").manual_seed(self.seed)
        q = _randn((self.total_q, self.num_heads, self.d_qk), g, self.qk_std)
        k = _randn((self.total_k, self.num_heads_k, self.d_qk), g, self.qk_std)
        v = _randn((self.total_k, self.num_heads_k, self.d_v), g, self.v_std)
        cq, ck = self.cu_seqlens()
        return q, k, v, cq, ck

    def make_inputs_on(self, device):
        """The same shapes and distributions drawn by a seeded generator on
        `device` (a different stream of numbers than make_inputs; for timing
        runs, where drawing gigabytes on the CPU would dominate)."""
        g = torch.Generator(device=device).manual_seed(self.seed)

        def draw(shape, std):
            x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            if std != 1.0:
                x.mul_(std)
            return x.to(torch.bfloat16)

        q = draw((self.total_q, self.num_heads, self.d_qk), self.qk_std)
        k = draw((self.total_k, self.num_heads_k, self.d_qk), self.qk_std)
        v = draw((self.total_k, self.num_heads_k, self.d_v), self.v_std)
        cq, ck = self.cu_seqlens()
        return q, k, v, cq.to(device), ck.to(device)


def _randn(shape, g, std):
    """N(0, std^2) drawn in fp32 chunks, rounded to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    n = flat.numel()
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e] = x.to(torch.bfloat16)
    return out


def window_lengths(lengths: List[int], w: int = 256) -> List[int]:
    """Splits each sequence into consecutive w-token windows (last may be short)."""
    out = []
    for L in lengths:
        full, rem = divmod(L, w)
        out += [w] * full + ([rem] if rem else [])
    return out


def tiny() -> VarlenWorkload:
    return VarlenWorkload("tiny", [17, 64, 100], [17, 64, 100], 4, 4, 64, 64,
                          1.0 / 8.0, seed=0)


def vit_full(d: int = 80) -> VarlenWorkload:
    return VarlenWorkload(f"vit_full_d{d}", list(VIT_LENGTHS), list(VIT_LENGTHS),
                          16, 16, d, d, d ** -0.5, qk_std=0.5, seed=1,
                          return_lse=False)


def vit_window(d: int = 80) -> VarlenWorkload:
    lens = window_lengths(VIT_LENGTHS)
    return VarlenWorkload(f"vit_window_d{d}", lens, list(lens), 16, 16, d, d,
                          d ** -0.5, qk_std=0.5, seed=1, return_lse=False)


def vit_window64(d: int = 80) -> VarlenWorkload:
    """The same tensors in 64-token windows (the Qwen2.5-VL windowed layers of
    the sglang FA4 PR, "Speed Tests and Profiling": windows of 64 patches,
    16 heads, d=80): 273 segments, the short-segment path."""
    lens = window_lengths(VIT_LENGTHS, 64)
    return VarlenWorkload(f"vit_window64_d{d}", lens, list(lens), 16, 16, d, d,
                          d ** -0.5, qk_std=0.5, seed=1, return_lse=False)


def long_seq(L: int) -> VarlenWorkload:
    return VarlenWorkload(f"long_{L}", [L], [L], 16, 16, 128, 128, 128 ** -0.5,
                          seed=2)


def mla_causal() -> VarlenWorkload:
    return VarlenWorkload("mla_causal", [4096] * 4, [4096] * 4, 128, 128, 192,
                          128, 192 ** -0.5, causal=True, seed=3)


def mla_chunked() -> VarlenWorkload:
    return VarlenWorkload("mla_chunked", [2048, 2048], [8192, 8192], 128, 128,
                          192, 128, 192 ** -0.5, causal=True, seed=3)


def mla_swa() -> VarlenWorkload:
    return VarlenWorkload("mla_swa", [4096] * 4, [4096] * 4, 128, 128, 192, 128,
                          192 ** -0.5, causal=True, window=(1024, 0), seed=3)


@dataclass
class DecodeWorkload:
    name: str = "decode"
    num_tokens: int = 128
    num_heads: int = 64
    topk: int = 2048
    context: int = 32768          # positions per token
    page_size: int = 64
    num_pages: int = 65536        # physical pages in the cache
    softmax_scale: float = 576 ** -0.5
    seed: int = 4

    @property
    def pages_per_token(self) -> int:
        return self.context // self.page_size

    def make_indices(self):
        """(page_table [T, P] int32, topk_idx [T, topk] int32)."""
        g = torch.Generator(device="cpu").manual_seed(self.seed)
        P = self.pages_per_token
        assert self.num_tokens * P <= self.num_pages
        perm = torch.randperm(self.num_pages, generator=g)
        page_table = perm[: self.num_tokens * P].view(self.num_tokens, P).to(torch.int32)
        topk = torch.stack([
            torch.randperm(self.context, generator=g)[: self.topk]
            for _ in range(self.num_tokens)
        ]).to(torch.int32)
        return page_table.contiguous(), topk.contiguous()

    def make_q(self):
        g = torch.Generator(device="cpu").manual_seed(self.seed + 1000)
        return _randn((self.num_tokens, self.num_heads, 576), g, 1.0)

    def make_cache(self, device="cpu"):
        """[num_pages, 64, 576] bf16 N(0,1), drawn in page blocks on the CPU."""
        g = torch.Generator(device="cpu").manual_seed(self.seed + 2000)
        cache = torch.empty((self.num_pages, self.page_size, 576), dtype=torch.bfloat16,
                            device=device)
        block = 1024
        for p0 in range(0, self.num_pages, block):
            p1 = min(self.num_pages, p0 + block)
            x = _randn((p1 - p0, self.page_size, 576), g, 1.0)
            cache[p0:p1].copy_(x)
        return cache


def small_decode(num_tokens=4, num_heads=64, topk=256, context=1024,
                 num_pages=None, seed=5) -> DecodeWorkload:
    P = context // 64
    return DecodeWorkload(name="decode_small", num_tokens=num_tokens,
                          num_heads=num_heads, topk=topk, context=context,
                          num_pages=num_pages or num_tokens * P + 3, seed=seed)


VARLEN_BENCH = {
    "tiny": tiny,
    "vit_full_d80": lambda: vit_full(80),
    "vit_full_d64": lambda: vit_full(64),
    "vit_full_d72": lambda: vit_full(72),
    "vit_full_d128": lambda: vit_full(128),
    "vit_window_d64": lambda: vit_window(64),
    "vit_window_d72": lambda: vit_window(72),
    "vit_window_d80": lambda: vit_window(80),
    "vit_window_d128": lambda: vit_window(128),
    "vit_window64_d80": lambda: vit_window64(80),
    "long_16384": lambda: long_seq(16384),
    "long_36864": lambda: long_seq(36864),
    "long_65536": lambda: long_seq(65536),
    "mla_causal": mla_causal,
    "mla_chunked": mla_chunked,
    "mla_swa": mla_swa,
}


def splitkv_long_k() -> VarlenWorkload:
    """Few query rows against a long key sequence: one 256-row chunk against
    65536 keys, 16 heads, d=128 (chunked prefill's context pass, which the
    vLLM flash_attn page runs non-causal and with the LSE returned:
    FlashAttnPrefillBackend.run_prefill_context_chunk).  Only 16 query
    tiles exist for the SMs: the split-KV case."""
    return VarlenWorkload("splitkv_q256_k65536", [256], [65536], 16, 16, 128, 128,
                          128 ** -0.5, seed=6)


def splitkv_decode_like() -> VarlenWorkload:
    """One query row per sequence against 32768 keys, 8 sequences, 128 heads,
    MLA dims (192, 128), bottom-right causal."""
    return VarlenWorkload("splitkv_q1x8_k32768_mla", [1] * 8, [32768] * 8, 128, 128, 192, 128,
                          192 ** -0.5, causal=True, seed=7)


def gqa_prefill(group: int = 4) -> VarlenWorkload:
    """Grouped-query attention: 32 query heads over 32/group key/value heads,
    d=128, 4 x 4096 causal (sglang FA4 PR, "Accuracy Tests": GQA and
    pack_gqa)."""
    return VarlenWorkload(f"gqa{group}_causal_4x4096", [4096] * 4, [4096] * 4, 32, 32 // group,
                          128, 128, 128 ** -0.5, causal=True, seed=8)


def gqa_decode_like(group: int = 8) -> VarlenWorkload:
    """Grouped-query attention with one query row per sequence: 64 sequences
    against 8192 keys each, 32 query heads over 32/group key/value heads,
    d=128, bottom-right causal."""
    return VarlenWorkload(f"gqa{group}_q1x64_k8192", [1] * 64, [8192] * 64, 32, 32 // group,
                          128, 128, 128 ** -0.5, causal=True, seed=9)


def vit_many_windows(d: int = 80) -> VarlenWorkload:
    """Two 4K-image windowed layers' worth of 64-token windows (700 each, the
    Qwen2.5-VL windowed layers of the sglang FA4 PR, "Speed Tests and
    Profiling") next to two full images of 4096 and 2000 tokens: 1402
    segments in one call, 16 heads."""
    lens = [64] * 700 + [4096] + [64] * 700 + [2000]
    return VarlenWorkload(f"vit_many_windows_d{d}", lens, list(lens), 16, 16, d, d, d ** -0.5,
                          qk_std=0.5, seed=10, return_lse=False)


def work_list_2048() -> VarlenWorkload:
    """2048 one-token sequences, one head: almost no attention work, so the
    time is the work-list build (sort and scan of 2048 sequences in every
    CTA) plus launch overhead."""
    return VarlenWorkload("work_list_2048", [1] * 2048, [1] * 2048, 1, 1, 64, 64, 0.125,
                          seed=11, return_lse=False)


# Workloads timed only in the bench's extra block (and covered by parity
# tests at reduced sizes).
EXTRA_ONLY = {
    "vit_many_windows_d80": lambda: vit_many_windows(80),
    "work_list_2048": work_list_2048,
    "splitkv_q256_k65536": splitkv_long_k,
    "splitkv_q1x8_k32768_mla": splitkv_decode_like,
    "gqa4_causal_4x4096": lambda: gqa_prefill(4),
    "gqa8_q1x64_k8192": lambda: gqa_decode_like(8),
}
