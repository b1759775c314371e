"""Parity of the generic linear layer and the decode-layer front end (through
the C ABI) against the fp64 CPU oracle, and of a whole decode layer: front end,
cache append, absorbed decode and the fused output projection against the
oracle's materialised attention. Tolerances: rel-L2 <= 5e-3 and max-abs <= 2e-2
for bf16 outputs, fp32-level for fp32."""
import math

import numpy as np
import pytest
import torch

from _util import assert_close, bits, f64, oracle_pool
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

F32_TOL = dict(rel=1e-5, mabs=1e-4, ulp_rel=0.0)


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


# (act, n_tokens, n_out, n_in): tensor cores with a K split and a ragged last
# row tile, the front end's first product, one token, two token tiles; many
# tokens (tokens as the MMA M dimension: ragged token and output tiles, and
# n_out % 8 != 0, which keeps rows of W as M); CUDA cores for n_in % 64 != 0
# and for fp32
LINEAR_CASES = [
    ("bf16", 5, 200, 7168),
    ("bf16", 32, 2112, 7168),
    ("bf16", 1, 64, 128),
    ("bf16", 300, 256, 256),
    ("bf16", 640, 264, 192),
    ("bf16", 1000, 512, 512),
    ("bf16", 600, 100, 64),
    # tokens as M over more units than CTAs: a ragged last token tile, a ragged
    # last tile of W rows, and a K of ten chunks
    ("bf16", 4100, 2048, 512),
    ("bf16", 3000, 2056, 384),
    ("bf16", 700, 512, 640),
    ("bf16", 7, 96, 100),
    ("f32", 3, 70, 96),
]


@pytest.mark.parametrize("act,n,n_out,n_in", LINEAR_CASES, ids=lambda v: str(v))
def test_linear(act, n, n_out, n_in):
    dt = torch.float32 if act == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(21)
    x = torch.randn(n, n_in, generator=g).to(dt)
    w = (torch.randn(n_out, n_in, generator=g) / math.sqrt(n_in)).to(dt)
    y = _C().mla_linear(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert_close(f64(y), O.linear(f64(x), f64(w)), what=f"linear {act} {n}x{n_out}x{n_in}",
                 **(F32_TOL if act == "f32" else {}))


def _front_case(act, n, d_model, d_cq, H, seed, max_pos=70000):
    W = _W()
    w = W.Workload("front", batch=n, q_len=1, heads=H, seq_lens=[1] * n, page_size=64, act_dtype=act,
                   cache_dtype=act, seed=seed)
    d = W.make_front_inputs(w, d_model, d_cq)
    g = torch.Generator().manual_seed(seed + 5)
    pos = torch.randint(0, max_pos, (n,), generator=g, dtype=torch.int32)
    pos[0] = 0
    if n > 1:
        pos[-1] = max_pos - 1
    return d, pos, max_pos


def _run_front(d, pos, max_pos, H, dev_error=None):
    C = _C()
    cos, sin = C.mla_rope_table(max_pos)
    w_dqkv = torch.cat([d["w_dq"], d["w_dkv"], d["w_kr"]], 0).cuda()
    w_uqr = torch.cat([d["w_uq"], d["w_qr"]], 0).cuda()
    out = C.mla_decode_front(d["h"].cuda(), w_dqkv, d["g_q"].cuda(), d["g_kv"].cuda(), w_uqr, pos.cuda(),
                             cos.cuda(), sin.cuda(), _W().RMS_EPS, H, dev_error=dev_error)
    torch.cuda.synchronize()
    return out


def _oracle_front(d, pos):
    return O.decode_front(f64(d["h"]), f64(d["w_dq"]), f64(d["g_q"]), f64(d["w_uq"]), f64(d["w_qr"]),
                          f64(d["w_dkv"]), f64(d["g_kv"]), f64(d["w_kr"]), pos.numpy(), _W().RMS_EPS)


@pytest.mark.parametrize("act,n,d_model,d_cq,H", [("bf16", 5, 512, 192, 4), ("bf16", 32, 7168, 1536, 128),
                                                  ("bf16", 3, 200, 96, 2), ("f32", 4, 256, 128, 3)],
                         ids=lambda v: str(v))
def test_front(act, n, d_model, d_cq, H):
    d, pos, max_pos = _front_case(act, n, d_model, d_cq, H, seed=22)
    got = _run_front(d, pos, max_pos, H)
    ref = _oracle_front(d, pos)
    tol = F32_TOL if act == "f32" else {}
    for name, g_, r_ in zip(("q_nope", "q_rope", "c_kv", "k_r"), got, ref):
        assert tuple(g_.shape) == r_.shape, name
        assert_close(f64(g_), r_, what=f"front {name} {act} n={n} d={d_model}", **tol)


def test_linear_and_front_past_grid_y_limit():
    """Token counts whose tiles exceed a grid's y extent (65,535): the CUDA-core
    linear layer at 600,000 tokens (75,000 tiles of 8) and the front end at
    70,000 tokens (its per-token finishing kernels)."""
    g = torch.Generator().manual_seed(24)
    x = torch.randn(600_000, 64, generator=g)
    w = torch.randn(8, 64, generator=g) / 8.0
    y = _C().mla_linear(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert_close(f64(y), O.linear(f64(x), f64(w)), what="linear, 600k tokens", **F32_TOL)
    d, pos, max_pos = _front_case("bf16", 70_000, 64, 64, 1, seed=25, max_pos=4096)
    got = _run_front(d, pos, max_pos, 1)
    ref = _oracle_front(d, pos)
    for name, g_, r_ in zip(("q_nope", "q_rope", "c_kv", "k_r"), got, ref):
        assert_close(f64(g_), r_, what=f"front {name}, 70k tokens")


def test_front_bad_position_flags_and_zeroes():
    d, pos, max_pos = _front_case("bf16", 3, 256, 128, 2, seed=23, max_pos=100)
    pos[1] = 100  # one past the table
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_nope, q_rope, c_kv, _ = _run_front(d, pos, max_pos, 2, dev_error=err)
    assert _C().mla_read_device_error(err) & _C().MLA_DEVERR_BAD_POSITION
    assert torch.count_nonzero(q_rope[1]).item() == 0
    ref = _oracle_front(d, pos)
    assert_close(f64(q_rope[[0, 2]]), ref[1][[0, 2]], what="q_rope of the good tokens")
    assert_close(f64(q_nope), ref[0], what="q_nope")


@pytest.mark.parametrize("fused", [True, False], ids=["fused_output", "unfused_output"])
def test_decode_layer_end_to_end(fused):
    """One decode step of a whole layer from the hidden states, through the
    layer API. GPU: front end -> append of the new tokens -> absorb -> paged
    decode -> output projection (W_UV folded into W_O, or W_UV per head then
    W_O). Oracle: its own front end, the new tokens' rows appended to its cache,
    K and V materialised per head, softmax, W_O over the concatenated heads."""
    W = _W()
    from mla_latent_kv_16_gb300.engine import build_layer
    w = W.preset("dsv3_bf16", batch=3, seq_lens=[4096, 700, 129])
    d = W.make_inputs(w)
    d_model, d_cq = 1024, 256
    fr = W.make_front_inputs(w, d_model, d_cq)
    w_o = W.make_out_weight(w, d_model)
    layer = build_layer(w, d)  # context without the step's new tokens
    layer.attach_front(fr["w_dq"], fr["w_dkv"], fr["w_kr"], fr["g_q"], fr["g_kv"], fr["w_uq"], fr["w_qr"], W.RMS_EPS)
    layer.attach_output(w_o, fused=fused)
    ni = d["new_index"]
    pos = d["ctx_positions"][ni].contiguous()
    y = f64(layer.step_from_hidden(fr["h"].cuda(), pos.cuda(), d["ctx_slots"][ni].cuda()))
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    # oracle: front end in fp64; the new rows enter its cache in the activation type
    rq_nope, rq_rope, rc_kv, rk_r = _oracle_front(fr, pos)
    d2 = dict(d)
    c_all, k_all = d["ctx_c_kv"].clone(), d["ctx_k_r"].clone()
    c_all[ni] = torch.from_numpy(O.round_bf16(rc_kv).astype(np.float32)).to(torch.bfloat16)
    k_all[ni] = torch.from_numpy(O.round_bf16(rk_r).astype(np.float32)).to(torch.bfloat16)
    d2["ctx_c_kv"], d2["ctx_k_r"] = c_all, k_all
    pool, sc = oracle_pool(w, d2)
    full = O.decode_full(rq_nope.reshape(w.batch, w.q_len, w.heads, 128),
                         rq_rope.reshape(w.batch, w.q_len, w.heads, 64), f64(d["w_uk"]), f64(d["w_uv"]), pool, sc,
                         d["block_table"].numpy(), d["seq_lens"].numpy(), w.q_len, w.page_size, w.cache_dtype,
                         O.default_scale())
    wo64 = f64(w_o)
    for b in range(w.batch):
        assert_close(y[b], O.out_proj_model(full[b][0], wo64), what=f"layer output, sequence {b}")
