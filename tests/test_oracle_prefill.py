"""Pins for the oracle's prefill in the MHA form (K and V expanded from the
latent, causal attention): the per-query non-absorbed form, torch's causal
scaled_dot_product_attention in float64, and the absorbed decode of the last
query. CPU only."""
import math

import numpy as np
import torch

from oracle import mla_oracle as O


def _case(seed, H=3, T=21, Tq=None):
    rng = np.random.default_rng(seed)
    Tq = T if Tq is None else Tq
    return (rng.standard_normal((Tq, H, 128)), rng.standard_normal((Tq, H, 64)), rng.standard_normal((T, 576)),
            rng.standard_normal((H, 128, 512)) / math.sqrt(512), rng.standard_normal((H, 128, 512)) / math.sqrt(512))


def test_prefill_matches_per_query_form():
    """Every query row equals the non-absorbed attention over its visible rows."""
    q_nope, q_rope, rows, w_uk, w_uv = _case(0, Tq=7)
    sc = O.default_scale()
    o, lse = O.prefill_mha(q_nope, q_rope, rows, w_uk, w_uv, sc)
    T, Tq = rows.shape[0], q_nope.shape[0]
    for j in range(Tq):
        ro, _, rl = O.attend_nonabsorbed(q_nope[j], q_rope[j], w_uk, w_uv, rows[:T - Tq + j + 1], sc)
        assert np.max(np.abs(o[j] - ro)) <= 1e-12 * np.max(np.abs(ro))
        assert np.max(np.abs(lse[j] - rl)) <= 1e-12 * np.max(np.abs(rl))


def test_prefill_matches_torch_causal_sdpa():
    """A whole prompt (Tq = T) against torch's causal attention on the expanded K, V."""
    q_nope, q_rope, rows, w_uk, w_uv = _case(1, H=4, T=33)
    k, v = O.expand_kv(rows, w_uk, w_uv)
    q = np.concatenate([q_nope, q_rope], -1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k).permute(1, 0, 2),
        torch.from_numpy(v).permute(1, 0, 2), is_causal=True, scale=O.default_scale()).permute(1, 0, 2)
    o, _ = O.prefill_mha(q_nope, q_rope, rows, w_uk, w_uv, O.default_scale())
    assert np.allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_prefill_last_row_equals_absorbed_decode():
    """The MHA and absorbed (MQA) forms agree: the last query's output equals
    W_UV applied to the absorbed latent sum over all rows."""
    q_nope, q_rope, rows, w_uk, w_uv = _case(2, T=40, Tq=5)
    sc = O.default_scale()
    o, lse = O.prefill_mha(q_nope, q_rope, rows, w_uk, w_uv, sc)
    u, l2 = O.attend_absorbed(O.absorb_q(q_nope[-1], w_uk), q_rope[-1], rows, sc)
    assert np.max(np.abs(o[-1] - O.out_proj(u, w_uv))) <= 1e-12 * np.max(np.abs(o[-1]))
    assert np.max(np.abs(lse[-1] - l2)) <= 1e-12 * np.max(np.abs(l2))


def test_expanded_keys_by_loops_and_causality():
    q_nope, q_rope, rows, w_uk, w_uv = _case(3, H=2, T=6)
    k, v = O.expand_kv(rows, w_uk, w_uv)
    for t, h, e in ((0, 0, 0), (5, 1, 127), (3, 1, 64)):
        assert abs(k[t, h, e] - math.fsum(w_uk[h, e, c] * rows[t, c] for c in range(512))) <= 1e-12
        assert abs(v[t, h, e] - math.fsum(w_uv[h, e, c] * rows[t, c] for c in range(512))) <= 1e-12
    assert np.array_equal(k[:, 1, 128:], rows[:, 512:])
    # the first query of a whole prompt sees only row 0: its output is V[0]
    o, _ = O.prefill_mha(q_nope, q_rope, rows, w_uk, w_uv, O.default_scale())
    assert np.allclose(o[0], v[0], rtol=0, atol=1e-14)
    # a later row's content must not reach an earlier query
    rows2 = rows.copy()
    rows2[4:] *= 7.0
    o2, _ = O.prefill_mha(q_nope, q_rope, rows2, w_uk, w_uv, O.default_scale())
    assert np.array_equal(o[:4], o2[:4]) and not np.allclose(o[4:], o2[4:])
