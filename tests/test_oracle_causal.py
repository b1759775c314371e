"""Pins for the oracle's decode at q_len > 1 (two draft tokens attending causally
within the step): query j of a q_len-token step sees rows 0 .. L - q_len + j.

The reading: the step's q_len new tokens are appended before attending ("Multi-
Head Latent Attention (MLA)" page, "PyTorch Reference Implementation": the
decode step concatenates the new latent rows to the cache first), so the last
q_len rows of a sequence are the step's own tokens and each one sees itself and
everything before it. Checked against torch's causal scaled_dot_product_attention
in float64 on the square problem (every position a query, the library's own
causal mask), against scalar loops, and against the MHA-form prefill; planted
off-by-one mistakes in the visible range must fail. CPU only."""
import math

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O


def _case(H=3, T=11, Lq=2, seed=21):
    g = np.random.default_rng(seed)
    rows = g.standard_normal((T, 576)).astype(np.float32)       # one sequence, fp32 cache
    q_lat = g.standard_normal((T, H, 512)) / 4.0                  # a query at every position
    q_rope = g.standard_normal((T, H, 64))
    return rows, q_lat, q_rope


def _decode(rows, q_lat, q_rope, Lq, page=4):
    """decode_latent for the last Lq positions, the rows spread over shuffled pages."""
    T = rows.shape[0]
    n_pages = -(-T // page)
    perm = np.random.default_rng(3).permutation(n_pages + 2)[:n_pages]
    pool = np.full(((n_pages + 2) * page, 576), np.nan, np.float32)
    for t in range(T):
        pool[perm[t // page] * page + t % page] = rows[t]
    out = O.decode_latent(q_lat[None, T - Lq:], q_rope[None, T - Lq:], pool, None, perm[None], [T], Lq, page, "f32",
                          O.default_scale())
    return out[0]


def _sdpa_square(rows, q_lat, q_rope):
    """torch's causal attention over all T positions (query i sees keys 0..i)."""
    q = torch.from_numpy(np.concatenate([q_lat, q_rope], -1)).permute(1, 0, 2)[None]    # [1,H,T,576]
    H = q.shape[1]
    k = torch.from_numpy(rows.astype(np.float64))[None, None].expand(1, H, -1, -1)        # [1,H,T,576]
    v = torch.from_numpy(rows[:, :512].astype(np.float64))[None, None].expand(1, H, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=O.default_scale())
    return o[0].permute(1, 0, 2).numpy()                                                   # [T,H,512]


@pytest.mark.parametrize("Lq", [1, 2, 3])
def test_decode_causality_matches_torch_causal_sdpa(Lq):
    rows, q_lat, q_rope = _case()
    T = rows.shape[0]
    u, lse = _decode(rows, q_lat, q_rope, Lq)
    ref = _sdpa_square(rows, q_lat, q_rope)[T - Lq:]
    assert u.shape == ref.shape
    assert np.max(np.abs(u - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_decode_causality_by_scalar_loops():
    """q_len 2: the first draft token sees T-1 rows, the second all T (fsum loops)."""
    rows, q_lat, q_rope = _case(H=2, T=6)
    T, Lq = rows.shape[0], 2
    u, lse = _decode(rows, q_lat, q_rope, Lq)
    sc = 1.0 / math.sqrt(192.0)
    r = rows.astype(np.float64)
    for j in range(Lq):
        pos = T - Lq + j
        for h in range(2):
            s = [math.fsum([q_lat[pos, h, c] * r[t, c] for c in range(512)] +
                           [q_rope[pos, h, e] * r[t, 512 + e] for e in range(64)]) * sc for t in range(pos + 1)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            assert abs(lse[j, h] - (m + math.log(z))) < 1e-12
            for c in (0, 255, 511):
                assert abs(u[j, h, c] - math.fsum(e[t] / z * r[t, c] for t in range(pos + 1))) < 1e-12


def test_decode_full_matches_prefill_last_rows():
    """The non-absorbed decode at q_len 2 equals the last two rows of the MHA-form
    prefill of the same sequence (both forms, both masks)."""
    g = np.random.default_rng(22)
    H, T, Lq, page = 4, 9, 2, 4
    rows = g.standard_normal((T, 576)).astype(np.float32)
    q_nope = g.standard_normal((Lq, H, 128))
    q_rope = g.standard_normal((Lq, H, 64))
    w_uk = g.standard_normal((H, 128, 512)) / math.sqrt(512)
    w_uv = g.standard_normal((H, 128, 512)) / math.sqrt(512)
    pool = np.full((3 * page, 576), np.nan, np.float32)
    pool[:T] = rows
    full = O.decode_full(q_nope[None], q_rope[None], w_uk, w_uv, pool, None, np.array([[0, 1, 2]]), [T], Lq, page,
                         "f32", O.default_scale())
    o, _, lse = full[0]
    o_p, lse_p = O.prefill_mha(q_nope, q_rope, rows.astype(np.float64), w_uk, w_uv, O.default_scale())
    assert np.max(np.abs(o - o_p)) <= 1e-12 * np.max(np.abs(o_p))
    assert np.max(np.abs(lse - lse_p)) <= 1e-12 * np.max(np.abs(lse_p))


@pytest.mark.parametrize("mistake", ["no_plus_one", "no_causality", "reversed"])
def test_planted_visibility_mistakes_fail(monkeypatch, mistake):
    wrong = {
        "no_plus_one": lambda L, q_len, j: L - q_len + j,
        "no_causality": lambda L, q_len, j: L,
        "reversed": lambda L, q_len, j: L - j,
    }[mistake]
    rows, q_lat, q_rope = _case()
    T, Lq = rows.shape[0], 2
    ref = _sdpa_square(rows, q_lat, q_rope)[T - Lq:]
    monkeypatch.setattr(O, "visible_tokens", wrong)
    u, _ = _decode(rows, q_lat, q_rope, Lq)
    assert np.max(np.abs(u - ref)) > 1e-6
