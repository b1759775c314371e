"""Feeds workload inputs (CPU torch tensors from the seeded generator) to the
oracle. TEST INFRASTRUCTURE ONLY, like the rest of this package."""
from __future__ import annotations

import numpy as np
import torch

from . import mla_oracle as O


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a tensor as numpy (bf16 -> uint16, fp32, uint8)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.uint8):
        return t.numpy()
    raise TypeError(t.dtype)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def seq_token_mask(w, seqs):
    """Boolean mask over the generator's context tokens of the listed sequences."""
    starts = np.concatenate([[0], np.cumsum(np.asarray(w.seq_lens, np.int64))])
    m = np.zeros(int(starts[-1]), dtype=bool)
    for b in seqs:
        m[starts[b]:starts[b + 1]] = True
    return m


def oracle_pool(w, d, token_mask=None):
    """The oracle's paged cache for workload w built from inputs d (optionally
    only the tokens where token_mask is True)."""
    cos_t, sin_t = O.rope_tables(w.max_pos, 64, w.rope_base)
    pool, sc = O.new_pool(w.num_pages, w.page_size, w.cache_dtype)
    c, k = bits(d["ctx_c_kv"]), bits(d["ctx_k_r"])
    pos, sl = d["ctx_positions"].numpy(), d["ctx_slots"].numpy()
    if token_mask is not None:
        c, k, pos, sl = c[token_mask], k[token_mask], pos[token_mask], sl[token_mask]
    O.append(pool, sc, c, k, pos.astype(np.int64), sl, cos_t, sin_t, w.act_dtype, w.cache_dtype)
    return pool, sc
