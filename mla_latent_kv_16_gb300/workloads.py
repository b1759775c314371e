"""Seeded synthetic workloads for MLA decode over a paged latent cache.

This module only draws random numbers and lays out pages. It holds none of the
method's arithmetic (no RoPE, no absorption, no attention, no quantisation), so
that the CUDA path and the CPU oracle can both consume the very same input
bytes without sharing any compute code.

Recipe (every workload):
  * activations q_nope [B,Lq,H,128], q_rope [B,Lq,H,64] ~ N(0,1);
  * weights W_UK, W_UV [H,128,512] ~ N(0,1) * (1/sqrt(512));
  * cached rows: c_KV [N,512] and pre-rotation k_R [N,64] ~ N(0,1) for every
    context token of every sequence, positions 0..L_b-1;
  * everything is drawn in fp32 from one seeded ``torch.Generator`` and then
    rounded (RNE, by torch's own dtype conversion) to the activation dtype;
  * pages: sequence b owns ceil(L_b / page_size) pages; the physical page ids
    are a seeded permutation of the pool; unused block-table entries are -1;
  * the optional outlier fraction multiplies the c_KV and k_R rows of a seeded
    subset of tokens by 4.0 (a power of two, exact in every dtype used here);
  * the output projection W_O [d_model, H, 128] (d_model = 7168 for the
    DeepSeek-V3 shape) ~ N(0,1) * (1/sqrt(H*128)), from a generator of its own
    so that drawing it leaves every other input unchanged;
  * the front end's hidden states h [B*Lq, d_model] ~ N(0,1) and its weights
    W_DQ [1536, d], W_UQ [H*128, 1536], W_QR [H*64, 1536], W_DKV [512, d],
    W_KR [64, d] ~ N(0,1) * (1/sqrt(fan_in)), RMSNorm gains 1 + 0.1 N(0,1),
    also from a generator of its own.

The named presets are the five decode workloads the method is measured on:
a tiny fp32 case, the DeepSeek-V3-shaped bf16 decode, a ragged bf16 batch, a
long-context split-KV case and an FP8 (E4M3) cache with two draft tokens.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

D_NOPE = 128
D_ROPE = 64
D_C = 512
D_V = 128
ROW = D_C + D_ROPE  # 576 values per cached token
D_MODEL = 7168      # hidden size of the DeepSeek-V3 shape
D_CQ = 1536         # query latent width
RMS_EPS = 2.0 ** -23  # nn.RMSNorm's default eps (float32 machine epsilon)

# dtype names shared with the C ABI (mla_dtype_t)
F32, BF16, E4M3 = "f32", "bf16", "e4m3"

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    q_len: int
    heads: int
    seq_lens: Sequence[int]
    page_size: int
    act_dtype: str          # dtype of q, weights and the rows handed to append
    cache_dtype: str        # dtype stored in the paged cache
    seed: int
    outlier_frac: float = 0.0
    num_splits: int = 0     # 0 = let the library choose
    shuffle_pages: bool = True
    rope_base: float = 10000.0

    @property
    def pages_per_seq(self):
        return [-(-int(L) // self.page_size) for L in self.seq_lens]

    @property
    def num_pages(self):
        return sum(self.pages_per_seq)

    @property
    def max_pages_per_seq(self):
        return max(self.pages_per_seq)

    @property
    def total_tokens(self):
        return int(sum(int(L) for L in self.seq_lens))

    @property
    def max_pos(self):
        return int(max(self.seq_lens))

    def row_bytes(self) -> int:
        """Bytes read per cached token: values plus, for E4M3, 5 fp32 scales."""
        if self.cache_dtype == F32:
            return ROW * 4
        if self.cache_dtype == BF16:
            return ROW * 2
        return ROW + 5 * 4


def preset(name: str, **over) -> Workload:
    """The five named decode workloads (full size). Keyword overrides give the
    reduced parity-test variants of the same recipe."""
    if name == "tiny_fp32":
        w = Workload(name, batch=2, q_len=1, heads=16, seq_lens=[256, 256], page_size=256,
                     act_dtype=F32, cache_dtype=F32, seed=0, shuffle_pages=False)
    elif name == "dsv3_bf16":
        w = Workload(name, batch=32, q_len=1, heads=128, seq_lens=[4096] * 32, page_size=64,
                     act_dtype=BF16, cache_dtype=BF16, seed=1)
    elif name == "ragged_bf16":
        g = torch.Generator().manual_seed(2)
        lens = torch.randint(1, 32768 + 1, (64,), generator=g).tolist()
        w = Workload(name, batch=64, q_len=1, heads=128, seq_lens=lens, page_size=64,
                     act_dtype=BF16, cache_dtype=BF16, seed=2)
    elif name == "long_splitkv_bf16":
        w = Workload(name, batch=4, q_len=1, heads=128, seq_lens=[131072] * 4, page_size=64,
                     act_dtype=BF16, cache_dtype=BF16, seed=3, outlier_frac=0.01, num_splits=128)
    elif name == "fp8_lq2":
        w = Workload(name, batch=128, q_len=2, heads=128, seq_lens=[8192] * 128, page_size=64,
                     act_dtype=BF16, cache_dtype=E4M3, seed=4)
    else:
        raise KeyError(name)
    for k, v in over.items():
        setattr(w, k, v)
    if "seq_lens" in over or "batch" in over:
        lens = list(w.seq_lens)
        if len(lens) != w.batch:
            lens = (lens * (w.batch // max(len(lens), 1) + 1))[: w.batch]
        w.seq_lens = lens
    return w


PRESETS = ("tiny_fp32", "dsv3_bf16", "ragged_bf16", "long_splitkv_bf16", "fp8_lq2")


def _randn(g, shape, dtype):
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def make_page_layout(w: Workload):
    """Block table [B, max_pages] int32 (-1 where unused) and, per sequence,
    the list of its physical pages. Layout only: which page holds which rows."""
    g = torch.Generator().manual_seed(w.seed * 7919 + 17)
    n = w.num_pages
    perm = torch.randperm(n, generator=g) if w.shuffle_pages else torch.arange(n)
    bt = torch.full((w.batch, w.max_pages_per_seq), -1, dtype=torch.int32)
    off = 0
    for b, np_b in enumerate(w.pages_per_seq):
        bt[b, :np_b] = perm[off: off + np_b].to(torch.int32)
        off += np_b
    return bt


def make_slots(w: Workload, block_table: torch.Tensor, positions_per_seq):
    """slot = physical_page * page_size + offset-in-page, for each listed
    (sequence, position) pair, in the same order. int64."""
    out = []
    P = w.page_size
    for b, pos in enumerate(positions_per_seq):
        pos = torch.as_tensor(pos, dtype=torch.int64)
        page = block_table[b].to(torch.int64)[pos // P]
        out.append(page * P + pos % P)
    return torch.cat(out) if out else torch.zeros(0, dtype=torch.int64)


def make_inputs(w: Workload, with_context: bool = True):
    """All CPU tensors of one decode step.

    Returns a dict with
      q_nope [B,Lq,H,128], q_rope [B,Lq,H,64] (act dtype; q_rope is taken as
      already rotated), w_uk, w_uv [H,128,512] (act dtype),
      block_table [B,maxp] int32, seq_lens [B] int32,
      ctx_c_kv [N,512], ctx_k_r [N,64] (act dtype, k_r before rotation),
      ctx_positions [N] int32, ctx_slots [N] int64 -- every cached token of every
      sequence (N = sum of seq_lens), sequence-major,
      new_index [B*Lq] int64 -- rows of the ctx_* arrays that are the step's
      Lq new tokens (the last Lq positions of each sequence).
    """
    g = torch.Generator().manual_seed(w.seed)
    dt = TORCH_DTYPE[w.act_dtype]
    B, Lq, H = w.batch, w.q_len, w.heads
    d = {}
    d["q_nope"] = _randn(g, (B, Lq, H, D_NOPE), dt)
    d["q_rope"] = _randn(g, (B, Lq, H, D_ROPE), dt)
    std = 1.0 / math.sqrt(D_C)
    d["w_uk"] = (torch.randn(H, D_NOPE, D_C, generator=g) * std).to(dt)
    d["w_uv"] = (torch.randn(H, D_V, D_C, generator=g) * std).to(dt)
    bt = make_page_layout(w)
    d["block_table"] = bt
    d["seq_lens"] = torch.tensor([int(L) for L in w.seq_lens], dtype=torch.int32)
    if with_context:
        N = w.total_tokens
        c = torch.randn(N, D_C, generator=g)
        k = torch.randn(N, D_ROPE, generator=g)
        if w.outlier_frac > 0:
            n_out = int(round(w.outlier_frac * N))
            idx = torch.randperm(N, generator=g)[:n_out]
            c[idx] *= 4.0
            k[idx] *= 4.0
        d["ctx_c_kv"] = c.to(dt)
        d["ctx_k_r"] = k.to(dt)
        pos = [torch.arange(int(L), dtype=torch.int64) for L in w.seq_lens]
        d["ctx_positions"] = torch.cat(pos).to(torch.int32)
        d["ctx_slots"] = make_slots(w, bt, pos)
        starts = torch.tensor([0] + list(w.seq_lens), dtype=torch.int64).cumsum(0)[:-1]
        new = [starts[b] + int(w.seq_lens[b]) - Lq + torch.arange(Lq) for b in range(B)]
        d["new_index"] = torch.cat(new)
    return d


def make_out_weight(w: Workload, d_model: int = D_MODEL) -> torch.Tensor:
    """W_O [d_model, H, 128] (act dtype), the output projection over the
    concatenated head outputs, seeded independently of make_inputs."""
    g = torch.Generator().manual_seed(w.seed * 1000003 + 29)
    std = 1.0 / math.sqrt(w.heads * D_V)
    return (torch.randn(d_model, w.heads, D_V, generator=g) * std).to(TORCH_DTYPE[w.act_dtype])


def make_front_inputs(w: Workload, d_model: int = D_MODEL, d_cq: int = D_CQ) -> dict:
    """Hidden states of the step's B*Lq new tokens and the front end's weights
    (nn.Linear layouts [out, in], act dtype), seeded independently of make_inputs."""
    g = torch.Generator().manual_seed(w.seed * 1000033 + 41)
    dt = TORCH_DTYPE[w.act_dtype]
    H = w.heads

    def lin(n_out, n_in):
        return (torch.randn(n_out, n_in, generator=g) / math.sqrt(n_in)).to(dt)

    d = {"h": torch.randn(w.batch * w.q_len, d_model, generator=g).to(dt),
         "w_dq": lin(d_cq, d_model), "w_uq": lin(H * D_NOPE, d_cq), "w_qr": lin(H * D_ROPE, d_cq),
         "w_dkv": lin(D_C, d_model), "w_kr": lin(D_ROPE, d_model)}
    d["g_q"] = (1.0 + 0.1 * torch.randn(d_cq, generator=g)).to(dt)
    d["g_kv"] = (1.0 + 0.1 * torch.randn(D_C, generator=g)).to(dt)
    return d


def make_prefill_inputs(n_tokens: int, n_queries: int, heads: int = 128, seed: int = 5,
                        act_dtype: str = BF16) -> dict:
    """One sequence for prefill in the MHA form: its n_tokens cached rows
    [T, 576] (c_KV and the k_R part, both drawn N(0,1); the k_R part stands for
    already-rotated keys, as a cache row holds them), the queries of its last
    n_queries positions q_nope [Tq, H, 128] and q_rope [Tq, H, 64] (rotated)
    ~ N(0,1), and W_UK, W_UV [H, 128, 512] ~ N(0,1) / sqrt(512)."""
    g = torch.Generator().manual_seed(seed * 7919 + 3)
    dt = TORCH_DTYPE[act_dtype]
    return {"rows": torch.randn(n_tokens, ROW, generator=g).to(dt),
            "q_nope": torch.randn(n_queries, heads, D_NOPE, generator=g).to(dt),
            "q_rope": torch.randn(n_queries, heads, D_ROPE, generator=g).to(dt),
            "w_uk": (torch.randn(heads, D_NOPE, D_C, generator=g) / math.sqrt(D_C)).to(dt),
            "w_uv": (torch.randn(heads, D_V, D_C, generator=g) / math.sqrt(D_C)).to(dt)}


def sample_sequences(w: Workload, k: int, seed: int = 12345):
    """A seeded subset of sequence indices (for checks at full size)."""
    g = torch.Generator().manual_seed(seed)
    k = min(k, w.batch)
    return sorted(torch.randperm(w.batch, generator=g)[:k].tolist())
