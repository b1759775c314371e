"""Parity of the fused output projection (W~ = W_O W_UV folded per head, then
y = W~ u over all heads) through the C ABI against the fp64 CPU oracle.

The fold is held to one bf16 ulp of the exact product plus the fp32 summation
bound of its 128 exact products (it rounds once, after the fp32 sum). The GEMM gets the oracle's own W~ (rounded to
the activation type) as input, never the GPU's. Tolerances for y: rel-L2 <=
5e-3 and max-abs <= 2e-2 (bf16), fp32-level for fp32.
"""
import math

import numpy as np
import pytest
import torch

from _util import assert_close, bits, f64, oracle_pool
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


def _C():
    from mla_latent_kv_16_gb300 import capi
    return capi


def _W():
    from mla_latent_kv_16_gb300 import workloads as W
    return W


def _weights(H, d_model, act, seed):
    """W_O [d, H, 128] and W_UV [H, 128, 512] from the seeded generators."""
    W = _W()
    w = W.Workload("fused", batch=1, q_len=1, heads=H, seq_lens=[1], page_size=64, act_dtype=act,
                   cache_dtype=act, seed=seed)
    return W.make_out_weight(w, d_model), W.make_inputs(w, with_context=False)["w_uv"]


def _to_act(x64, act):
    """fp64 oracle values as a tensor of the activation type (bf16: RNE via fp32)."""
    if act == "bf16":
        return torch.from_numpy(O.round_bf16(x64).astype(np.float32)).to(torch.bfloat16)
    return torch.from_numpy(np.asarray(x64, np.float32))


def _ulp_bf16(x):
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _fold_bound(w_o64, w_uv64, exact):
    """Error bound of a bf16 fold: one ulp of the result (the final rounding, with
    room for the fp32 sum pushing it across a rounding boundary) plus the fp32
    summation bound 128 * 2^-24 * sum_e |W_O W_UV|, which dominates where the 128
    products cancel."""
    mag = O.fuse_out_weights(np.abs(w_o64), np.abs(w_uv64))
    return _ulp_bf16(exact) + 128 * 2.0 ** -24 * mag


@pytest.mark.parametrize("act,H,d_model", [("bf16", 4, 200), ("bf16", 2, 128), ("f32", 3, 70)])
def test_fuse_weights(act, H, d_model):
    w_o, w_uv = _weights(H, d_model, act, seed=11)
    got = f64(_C().mla_fuse_out_weights(w_o.cuda(), w_uv.cuda()))
    torch.cuda.synchronize()
    exact = O.fuse_out_weights(f64(w_o), f64(w_uv))
    assert got.shape == exact.shape
    if act == "bf16":
        # at most one ulp from the exact value, and the oracle's own rounding almost everywhere
        assert np.all(np.abs(got - exact) <= _fold_bound(f64(w_o), f64(w_uv), exact)), "fold off by more than its bound"
        assert np.mean(got != O.round_bf16(exact)) <= 1e-3
    else:
        assert np.max(np.abs(got - exact)) <= 1e-5 * np.max(np.abs(exact))


# (act, H, d_model, n_tokens): tensor-core path with and without a K split, a
# ragged token count, two token tiles, one token; CUDA-core path for d_model %
# 128 != 0 and for fp32
GEMM_CASES = [
    ("bf16", 4, 384, 5),
    ("bf16", 128, 256, 32),
    ("bf16", 2, 128, 300),
    ("bf16", 1, 128, 1),
    ("bf16", 8, 200, 7),
    ("f32", 16, 96, 3),
]


@pytest.mark.parametrize("act,H,d_model,n", GEMM_CASES, ids=lambda v: str(v))
def test_out_proj_fused(act, H, d_model, n):
    w_o, w_uv = _weights(H, d_model, act, seed=12)
    w_f = _to_act(O.fuse_out_weights(f64(w_o), f64(w_uv)), act)
    g = torch.Generator().manual_seed(13)
    u = torch.randn(n, H, 512, generator=g).to(w_f.dtype)
    y = _C().mla_out_proj_fused(u.cuda(), w_f.cuda())
    torch.cuda.synchronize()
    ref = O.out_proj_fused(f64(u), f64(w_f))
    tol = dict(rel=1e-5, mabs=1e-4, ulp_rel=0.0) if act == "f32" else {}
    assert y.shape == (n, d_model)
    assert_close(f64(y), ref, what=f"y {act} H={H} d={d_model} n={n}", **tol)


def test_out_proj_fused_no_tokens_and_small_workspace():
    C = _C()
    w_f = torch.zeros(128, 4, 512, dtype=torch.bfloat16, device="cuda")
    u = torch.zeros(0, 4, 512, dtype=torch.bfloat16, device="cuda")
    y = C.mla_out_proj_fused(u, w_f)
    assert y.shape == (0, 128)
    need = C.mla_out_proj_fused_workspace_size(5, 384, 4)
    assert need > 0
    u5 = torch.zeros(5, 4, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(C.MlaError) as e:
        C.mla_out_proj_fused(u5, torch.zeros(384, 4, 512, dtype=torch.bfloat16, device="cuda"),
                             workspace=torch.empty(need - 256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == C.MLA_ERR_WORKSPACE_TOO_SMALL


def test_out_proj_fused_full_size():
    """DeepSeek-V3 shape (d_model 7168, 128 heads, a decode batch of 32) in the
    launch configuration the benchmark times: every output element against the
    oracle, with the oracle's own W~ as input; plus the GPU fold on sampled rows."""
    W = _W()
    w = W.preset("dsv3_bf16")
    d_model, H, n = W.D_MODEL, w.heads, w.batch
    w_o = W.make_out_weight(w, d_model)
    w_uv = W.make_inputs(w, with_context=False)["w_uv"]
    wo64, wuv64 = f64(w_o), f64(w_uv)
    w_f = torch.empty(d_model, H, 512, dtype=torch.bfloat16)
    for h in range(H):  # the oracle's fold, one head at a time (fp64, then rounded)
        w_f[:, h, :] = _to_act(O.fuse_out_weights(wo64[:, h:h + 1, :], wuv64[h:h + 1])[:, 0, :], "bf16")
    g = torch.Generator().manual_seed(14)
    u = torch.randn(n, H, 512, generator=g).to(torch.bfloat16)
    y = f64(_C().mla_out_proj_fused(u.cuda(), w_f.cuda()))
    torch.cuda.synchronize()
    u64 = f64(u)
    ref = np.zeros((n, d_model))
    for h in range(H):  # the oracle's product, summed over head slices
        ref += O.out_proj_fused(u64[:, h:h + 1, :], f64(w_f[:, h:h + 1, :]))
    assert_close(y, ref, what="y full size")
    # the GPU fold, sampled rows against the exact fold
    gf = _C().mla_fuse_out_weights(w_o.cuda(), w_uv.cuda())
    rows = torch.randperm(d_model, generator=torch.Generator().manual_seed(15))[:48].tolist()
    got = f64(gf[rows])
    exact = O.fuse_out_weights(wo64[rows], wuv64)
    assert np.all(np.abs(got - exact) <= _fold_bound(wo64[rows], wuv64, exact))


def test_decode_then_fused_projection_matches_materialised_attention():
    """The layer's output in the model dimension, GPU: decode step (append,
    absorb, paged decode) -> fold -> fused projection; oracle: K and V
    materialised per head, softmax, then W_O over the concatenated heads."""
    W = _W()
    from mla_latent_kv_16_gb300.engine import build_layer, step_inputs
    w = W.preset("dsv3_bf16", batch=3, seq_lens=[4096, 700, 129])
    d = W.make_inputs(w)
    d_model = 1024
    w_o = W.make_out_weight(w, d_model)
    layer = build_layer(w, d)
    s = step_inputs(d)
    layer.step(**s)
    w_f = _C().mla_fuse_out_weights(w_o.cuda(), layer.w_uv)
    y = f64(_C().mla_out_proj_fused(layer.u, w_f))
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    pool, sc = oracle_pool(w, d)
    full = O.decode_full(f64(d["q_nope"]), f64(d["q_rope"]), f64(d["w_uk"]), f64(d["w_uv"]), pool, sc,
                         d["block_table"].numpy(), d["seq_lens"].numpy(), w.q_len, w.page_size, w.cache_dtype,
                         O.default_scale())
    wo64 = f64(w_o)
    for b in range(w.batch):
        ref = O.out_proj_model(full[b][0], wo64)  # [Lq, d_model]
        assert_close(y[b], ref, what=f"layer output, sequence {b}")
