"""Parity of prefill in the MHA form (mla_prefill_mha, through the C ABI)
against the fp64 oracle's prefill_mha: K and V expanded from the latent rows,
causal attention of the last Tq positions over all T rows.

Small cases span several 128-query and 128-key tiles with ragged tails, fewer
queries than tokens (the causal diagonal off a tile boundary) and a one-token
sequence; the DeepSeek-V3-shaped prompt (4096 tokens, 128 heads) is checked on
sampled queries and heads, one query at a time in the non-absorbed form.
Tolerances: rel-L2 <= 5e-3 and max-abs <= 2e-2 on o; lse within the bound the
kernel's arithmetic implies (bf16 K from the expansion, bf16 P)."""
import numpy as np
import pytest
import torch

from _util import U_BF16, U_F32, assert_close, f64
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from mla_latent_kv_16_gb300 import build
    build.build()
    from mla_latent_kv_16_gb300 import capi
    capi.load()
    yield


def _inputs(T, Tq, H, seed):
    from mla_latent_kv_16_gb300 import workloads as W
    return W.make_prefill_inputs(T, Tq, H, seed)


def _run(d):
    from mla_latent_kv_16_gb300 import capi
    dev_error = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = capi.mla_prefill_mha(d["q_nope"].cuda(), d["q_rope"].cuda(), d["rows"].cuda(), d["w_uk"].cuda(),
                                  d["w_uv"].cuda(), dev_error=dev_error)
    torch.cuda.synchronize()
    assert int(dev_error.item()) == 0
    return f64(o), lse.cpu().numpy().astype(np.float64)


def _lse_bound(q_nope, q_rope, rows, w_uk, h, pos):
    """|lse_gpu - lse| <= max_t |ds_t| + 2^-21 + n 2^-24: the scores use K_nope
    rounded to bf16 by the expansion (2^-8 relative each) accumulated in fp32,
    and the row sum adds the fp32 weights (exp2 within 2^-21 relative) in fp32."""
    r = f64(rows)[:pos + 1]
    k = np.abs(r[:, :512] @ f64(w_uk)[h].T)                       # |K_nope| exact
    mag_n = k @ np.abs(f64(q_nope)[h])
    mag_r = np.abs(r[:, 512:]) @ np.abs(f64(q_rope)[h])
    d = O.default_scale() * np.max(mag_n * (U_BF16 + 600 * U_F32) + mag_r * 600 * U_F32)
    return d + 2.0 ** -21 + (pos + 64) * U_F32 + 1e-6


@pytest.mark.parametrize("T,Tq,H", [(1, 1, 4), (200, 200, 8), (333, 77, 16), (130, 130, 128), (700, 300, 3)])
def test_prefill_small(T, Tq, H):
    d = _inputs(T, Tq, H, seed=T + H)
    o, lse = _run(d)
    ro, rl = O.prefill_mha(f64(d["q_nope"]), f64(d["q_rope"]), f64(d["rows"]), f64(d["w_uk"]), f64(d["w_uv"]),
                           O.default_scale())
    assert_close(o, ro, what=f"o T={T} Tq={Tq} H={H}")
    for j in range(Tq):
        pos = T - Tq + j
        for h in range(H):
            if j % 17 == 0 or j == Tq - 1:
                b = _lse_bound(d["q_nope"][j], d["q_rope"][j], d["rows"], d["w_uk"], h, pos)
                assert abs(lse[j, h] - rl[j, h]) <= b, (j, h, lse[j, h], rl[j, h], b)


def test_prefill_full_size_sampled():
    """A DeepSeek-V3-shaped prompt: 4096 tokens, 128 heads, every position a
    query; sampled (query, head) pairs against the per-query non-absorbed form."""
    T, H = 4096, 128
    d = _inputs(T, T, H, seed=11)
    o, lse = _run(d)
    rows = f64(d["rows"])
    g = np.random.default_rng(3)
    queries = sorted(set([0, 1, 127, 128, 2047, T - 1] + g.integers(0, T, 10).tolist()))
    heads = [0, 5, 77, 127]
    wuk, wuv = f64(d["w_uk"])[heads], f64(d["w_uv"])[heads]
    for j in queries:
        ro, _, rl = O.attend_nonabsorbed(f64(d["q_nope"][j])[heads], f64(d["q_rope"][j])[heads], wuk, wuv,
                                         rows[:j + 1], O.default_scale())
        assert_close(o[j, heads], ro, what=f"o query {j}")
        for i, h in enumerate(heads):
            b = _lse_bound(d["q_nope"][j], d["q_rope"][j], d["rows"], d["w_uk"], h, j)
            assert abs(lse[j, h] - rl[i]) <= b, (j, h)
    assert np.all(np.isfinite(o))


def test_prefill_rejects_bad_arguments():
    from mla_latent_kv_16_gb300 import capi
    L = capi.load()
    D = capi.dims(8)
    assert L.mla_prefill_mha(16, 16, 16, 16, 16, 10, 11, 0.1, 16, 1 << 30, 16, None, None, D, capi.MLA_BF16,
                             None) == capi.MLA_ERR_INVALID_ARG          # more queries than tokens
    assert L.mla_prefill_mha(16, 16, 16, 16, 16, 10, 10, 0.1, 16, 1 << 30, 16, None, None, D, capi.MLA_F32,
                             None) == capi.MLA_ERR_UNSUPPORTED
    assert L.mla_prefill_mha(16, 16, 16, 16, 16, 10, 10, 0.1, 16, 16, 16, None, None, D, capi.MLA_BF16,
                             None) == capi.MLA_ERR_WORKSPACE_TOO_SMALL
