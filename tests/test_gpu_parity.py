"""Parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases span several tiles and ragged page tails; the full-size workloads
are checked on all or a seeded sample of sequences in the launch configuration
the benchmark times. Tolerances: bit-exact for cache bytes and page indexing;
rel-L2 <= 5e-3 and max-abs <= 2e-2 for floating outputs.
"""
import math

import numpy as np
import pytest
import torch

from _util import (F32_TOL, assert_close, bits, check_lse, decode_full_bf16_interface, f64, oracle_pool,
                   seq_token_mask, tol_for, visible_rows)
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


def _W():
    from mla_latent_kv_16_gb300 import workloads as W
    return W


def _layer(w, d, **kw):
    from mla_latent_kv_16_gb300.engine import build_layer
    return build_layer(w, d, **kw)


def _step(layer, d):
    from mla_latent_kv_16_gb300.engine import step_inputs
    s = step_inputs(d)
    o = layer.step(**s)
    torch.cuda.synchronize()
    return o


SMALL = {
    "tiny_fp32": dict(),
    "dsv3_bf16": dict(batch=3, seq_lens=[4096, 700, 129]),
    "ragged_bf16": dict(batch=5, seq_lens=[1, 63, 64, 65, 1000]),
    "long_splitkv_bf16": dict(batch=2, seq_lens=[20000, 9000], num_splits=16),
    "fp8_lq2": dict(batch=3, seq_lens=[2, 130, 515]),
    # two draft tokens on the bf16 cache (the query positions' causal cut on the bf16 kernel)
    "dsv3_bf16_lq2": dict(batch=3, q_len=2, seq_lens=[2, 300, 1030], num_splits=2),
}


def _small(name):
    return _W().preset(name.replace("_lq2", "") if name.startswith("dsv3") else name, **SMALL[name])


# ----------------------------------------------------------------------------- append

@pytest.mark.parametrize("name", list(SMALL))
def test_append_bit_exact(name):
    w = _small(name)
    d = _W().make_inputs(w)
    layer = _layer(w, d, fill_context=False)
    from mla_latent_kv_16_gb300.engine import step_inputs
    layer.append_chunked(d["ctx_c_kv"], d["ctx_k_r"], d["ctx_positions"], d["ctx_slots"])
    torch.cuda.synchronize()
    pool, sc = oracle_pool(w, d)
    got = bits(layer.cache).reshape(pool.shape)
    assert np.array_equal(got.view(np.uint8), pool.view(np.uint8)), "cache bytes differ"
    if sc is not None:
        assert np.array_equal(bits(layer.scales).reshape(sc.shape).view(np.uint32), sc.view(np.uint32))
    assert layer.device_error() == 0


def test_rope_table_matches_oracle():
    from mla_latent_kv_16_gb300 import capi
    cos, sin = capi.mla_rope_table(5000)
    oc, os_ = O.rope_tables(5000)
    assert np.array_equal(cos.numpy().view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(sin.numpy().view(np.uint32), os_.view(np.uint32))


# ----------------------------------------------------------------------------- projections

@pytest.mark.parametrize("name", ["tiny_fp32", "dsv3_bf16", "fp8_lq2"])
@pytest.mark.parametrize("n_tok", [1, 7, 32, 33, 256])
def test_absorb_and_out_proj(name, n_tok):
    from mla_latent_kv_16_gb300 import capi
    w = _small(name)
    d = _W().make_inputs(w, with_context=False)
    H = w.heads
    g = torch.Generator().manual_seed(n_tok)
    dt = d["q_nope"].dtype
    q = torch.randn(n_tok, H, 128, generator=g).to(dt)
    u = torch.randn(n_tok, H, 512, generator=g).to(dt)
    q_lat = capi.mla_absorb_q(q.cuda(), d["w_uk"].cuda())
    o = capi.mla_out_proj(u.cuda(), d["w_uv"].cuda())
    torch.cuda.synchronize()
    ref_q = O.absorb_q(f64(q), f64(d["w_uk"]))
    ref_o = O.out_proj(f64(u), f64(d["w_uv"]))
    tol = dict(F32_TOL) if dt == torch.float32 else {}
    assert_close(f64(q_lat), ref_q, **tol, what="absorb")
    assert_close(f64(o), ref_o, **tol, what="out_proj")


# ----------------------------------------------------------------------------- decode
#
# Every decode check below takes its reference from oracle inputs alone: the
# oracle's own absorbed query (exact fp64, from q_nope and W_UK) and the cache
# read back exactly (E4M3 as decode(byte) * scale). The GPU gets the same
# q_nope (its own absorb) or the oracle's q_lat rounded to the ABI's type.


def _eps_c(w):
    """Relative error of the cache values as the kernel multiplies them: the
    E4M3 path rounds code * scale to bf16; other caches are used as stored."""
    return 2.0 ** -8 if w.cache_dtype == "e4m3" else 0.0


def _q_exact(d):
    return O.absorb_q(f64(d["q_nope"]), f64(d["w_uk"]))


def _check_latent(w, d, pool, sc, u_gpu, lse_gpu, q_gpu, seqs=None, what=""):
    """u [B,Lq,H,512] and lse [B,Lq,H] from the GPU against the oracle's decode
    from its exact absorbed query; q_gpu = the q_lat the GPU decoded with. The
    long-context workload's x4 outliers take the query as the ABI carries it
    (the exact absorbed query rounded to bf16): its rounding alone moves their
    dominant logits, and u (of magnitude 16 and more there), past 2e-2."""
    q_ex = _q_exact(d)
    if w.outlier_frac > 0:
        q_ex = O.round_bf16(q_ex)
    ref = O.decode_latent(q_ex, f64(d["q_rope"]), pool, sc, d["block_table"].numpy(), list(w.seq_lens), w.q_len,
                          w.page_size, w.cache_dtype, O.default_scale(), batch_index=seqs)
    tol = tol_for(w)
    for b, (ru, rl) in ref.items():
        assert_close(u_gpu[b], ru, **tol, what=f"{what} u seq {b}")
        if lse_gpu is not None:
            check_lse(lse_gpu[b], rl, q_gpu[b], q_ex[b], f64(d["q_rope"])[b], visible_rows(w, d, pool, sc, b),
                      O.default_scale(), _eps_c(w), what=f"{what} lse seq {b}")
    return ref


def _check_o(w, d, og, pool, sc, seqs, heads=None):
    """End-to-end output o against the exact fp64 oracle from oracle inputs.
    heads=None: all heads, through the oracle's absorbed form (pinned equal to
    the non-absorbed one to 1e-12); else the listed heads in the non-absorbed
    (materialised K/V) form. The long-context workload's x4 outliers keep the
    max-abs reading against the oracle with the ABI's bf16 roundings."""
    tol = tol_for(w)
    args = (f64(d["q_rope"]), pool, sc, d["block_table"].numpy(), list(w.seq_lens), w.q_len, w.page_size,
            w.cache_dtype, O.default_scale())
    if heads is None:
        lat = O.decode_latent(_q_exact(d), *args, batch_index=seqs)
        ref = {b: O.out_proj(u, f64(d["w_uv"])) for b, (u, _) in lat.items()}
        hs = slice(None)
    else:
        full = O.decode_full(f64(d["q_nope"]), f64(d["q_rope"]), f64(d["w_uk"]), f64(d["w_uv"]), pool, sc,
                             d["block_table"].numpy(), list(w.seq_lens), w.q_len, w.page_size, w.cache_dtype,
                             O.default_scale(), batch_index=seqs, heads=heads)
        ref = {b: v[0] for b, v in full.items()}
        hs = list(heads)
    iface = None
    if w.outlier_frac > 0:
        iface = decode_full_bf16_interface(f64(d["q_nope"]), f64(d["q_rope"]), f64(d["w_uk"]), f64(d["w_uv"]),
                                           pool, sc, d["block_table"].numpy(), list(w.seq_lens), w.q_len,
                                           w.page_size, w.cache_dtype, O.default_scale(), batch_index=seqs)
    for b, ro in ref.items():
        if iface is None:
            assert_close(og[b][:, hs], ro, **tol, what=f"o seq {b}")
        else:
            assert_close(og[b][:, hs], ro, rel=tol["rel"], mabs=float("inf"), what=f"o seq {b} vs exact")
            assert_close(og[b][:, hs], iface[b][:, hs], **tol, what=f"o seq {b} vs bf16-interface oracle")


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_and_step_small(name):
    w = _small(name)
    d = _W().make_inputs(w)
    layer = _layer(w, d)
    o = _step(layer, d)
    assert layer.device_error() == 0
    pool, sc = oracle_pool(w, d)
    # absorb + decode on the GPU against the oracle from its own absorbed query
    _check_latent(w, d, pool, sc, f64(layer.u), layer.lse.cpu().numpy(), f64(layer.q_lat), what=name)
    # whole step (absorb + decode + out_proj): all heads through the absorbed
    # form, and 16 heads in the non-absorbed fp64 form
    seqs = list(range(w.batch))
    _check_o(w, d, f64(o), pool, sc, seqs)
    _check_o(w, d, f64(o), pool, sc, seqs, heads=range(0, w.heads, max(1, w.heads // 16)))


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_from_oracle_query(name):
    """mla_decode_paged alone, fed the oracle's absorbed query rounded to the
    ABI's activation type (no GPU absorb in the loop)."""
    from mla_latent_kv_16_gb300 import capi
    w = _small(name)
    d = _W().make_inputs(w)
    layer = _layer(w, d)
    _step(layer, d)                     # appends the step's tokens: the cache is complete
    pool, sc = oracle_pool(w, d)
    q_in = torch.from_numpy(_q_exact(d)).to(layer.act)
    layer.dev_error.zero_()
    u, lse = capi.mla_decode_paged(q_in.cuda(), d["q_rope"].cuda(), layer.cache, layer.scales, layer.block_table,
                                   layer.seq_lens, w.page_size, w.cache_dtype, num_splits=w.num_splits,
                                   dev_error=layer.dev_error)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    _check_latent(w, d, pool, sc, f64(u), lse.cpu().numpy(), f64(q_in), what=f"{name} oracle q")


@pytest.mark.parametrize("cache", ["bf16", "e4m3"])
@pytest.mark.parametrize("page_size,splits", [(128, 0), (128, 2), (256, 3)])
def test_pages_larger_than_a_tile(cache, page_size, splits):
    """Pages of 128 and 256 tokens: the tensor-core kernel walks them in 64-token
    tiles that start inside a page (row offset 64, 128, 192), including the
    E4M3 converter's per-row scales and ragged last pages."""
    W = _W()
    name = "dsv3_bf16" if cache == "bf16" else "fp8_lq2"
    w = W.preset(name, batch=3, seq_lens=[1000, 129, 300], page_size=page_size, num_splits=splits)
    d = W.make_inputs(w)
    layer = _layer(w, d)
    _step(layer, d)
    assert layer.device_error() == 0
    pool, sc = oracle_pool(w, d)
    _check_latent(w, d, pool, sc, f64(layer.u), layer.lse.cpu().numpy(), f64(layer.q_lat), what=f"page {page_size}")


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7, 8, 64])
def test_split_count_invariance(splits):
    w = _W().preset("ragged_bf16", batch=4, seq_lens=[3000, 17, 640, 2049], num_splits=splits)
    d = _W().make_inputs(w)
    layer = _layer(w, d)
    _step(layer, d)
    pool, sc = oracle_pool(w, d)
    _check_latent(w, d, pool, sc, f64(layer.u), layer.lse.cpu().numpy(), f64(layer.q_lat), what=f"splits={splits}")


def test_page_permutation_bit_identical():
    W = _W()
    outs = []
    for shuffle in (False, True):
        w = W.preset("dsv3_bf16", batch=2, seq_lens=[1000, 333], shuffle_pages=shuffle, num_splits=3)
        d = W.make_inputs(w)
        layer = _layer(w, d)
        o = _step(layer, d)
        outs.append((bits(layer.u).copy(), bits(o).copy(), d["block_table"]))
    assert not torch.equal(outs[0][2], outs[1][2])
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


def test_single_token_sequence_returns_its_row():
    W = _W()
    w = W.preset("dsv3_bf16", batch=2, seq_lens=[1, 1])
    d = W.make_inputs(w)
    layer = _layer(w, d)
    _step(layer, d)
    u = bits(layer.u)
    c = bits(d["ctx_c_kv"])
    pool, sc = oracle_pool(w, d)
    for b in range(2):
        assert np.all(u[b, 0] == c[b][None, :]), "softmax over one token must return c_KV exactly"
    # lse of a single score is the score itself
    _check_latent(w, d, pool, sc, f64(layer.u), layer.lse.cpu().numpy(), f64(layer.q_lat), what="one token")


# ----------------------------------------------------------------------------- data faults

def test_bad_block_table_and_seq_len_are_flagged_not_fatal():
    W = _W()
    w = W.preset("dsv3_bf16", batch=3, seq_lens=[200, 300, 100], num_splits=2)
    d = W.make_inputs(w)
    layer = _layer(w, d)
    _step(layer, d)                     # appends the step's new tokens: every visible row is written
    from mla_latent_kv_16_gb300 import capi
    bt = layer.block_table.clone()
    bt[0, 1] = w.num_pages + 5          # outside the pool
    sl = layer.seq_lens.clone()
    sl[2] = 10 ** 6                     # beyond max_pages * page_size
    layer.dev_error.zero_()
    q_lat = layer.absorb(d["q_nope"].cuda())
    u, lse = capi.mla_decode_paged(q_lat, d["q_rope"].cuda(), layer.cache, layer.scales, bt, sl, w.page_size,
                                   w.cache_dtype, num_splits=2, dev_error=layer.dev_error)
    code = layer.device_error()
    assert code & capi.MLA_DEVERR_BAD_PAGE and code & capi.MLA_DEVERR_BAD_SEQLEN
    assert torch.isfinite(u[1]).all()   # the healthy sequence is unaffected
    assert torch.all(u[2] == 0) and torch.all(torch.isinf(lse[2]))
    # context still usable afterwards
    layer.dev_error.zero_()
    _step(layer, d)
    assert layer.device_error() == 0


def test_bad_slot_and_position_in_append_are_flagged():
    W = _W()
    w = W.preset("dsv3_bf16", batch=1, seq_lens=[64])
    d = W.make_inputs(w)
    layer = _layer(w, d, fill_context=False)
    sl = d["ctx_slots"].clone()
    sl[3] = -1
    sl[5] = w.num_pages * w.page_size
    pos = d["ctx_positions"].clone()
    pos[7] = 10 ** 6
    layer.append(d["ctx_c_kv"].cuda(), d["ctx_k_r"].cuda(), pos.cuda(), sl.cuda())
    from mla_latent_kv_16_gb300 import capi
    code = layer.device_error()
    assert code & capi.MLA_DEVERR_BAD_SLOT and code & capi.MLA_DEVERR_BAD_POSITION


def test_invalid_arguments_rejected_synchronously():
    from mla_latent_kv_16_gb300 import capi
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(4, 128, 512, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(2, 4, 512, dtype=torch.bfloat16, device="cuda")
    L = capi.load()
    bad = capi.MlaDims(4, 64, 512, 64, 128)
    assert L.mla_absorb_q(q.data_ptr(), w.data_ptr(), out.data_ptr(), 2, bad, capi.MLA_BF16, None) == \
        capi.MLA_ERR_INVALID_ARG
    assert L.mla_absorb_q(q.data_ptr() + 2, w.data_ptr(), out.data_ptr(), 2, capi.dims(4), capi.MLA_BF16, None) == \
        capi.MLA_ERR_INVALID_ARG
    assert L.mla_decode_paged(q.data_ptr(), q.data_ptr(), w.data_ptr(), None, None, None, 1, 1, 4, 4, 64, 0.1, 0,
                              None, 0, out.data_ptr(), None, None, capi.dims(4), capi.MLA_BF16, capi.MLA_E4M3,
                              None) == capi.MLA_ERR_INVALID_ARG


# ----------------------------------------------------------------------------- full size

@pytest.mark.parametrize("name,nseq", [("dsv3_bf16", 32), ("ragged_bf16", 6), ("long_splitkv_bf16", 2),
                                       ("fp8_lq2", 16), ("tiny_fp32", 2)])
def test_full_size_workloads(name, nseq):
    """The benchmark's launch configuration at full size, from oracle inputs:
    cache bytes of the sampled sequences bit-exact; u and lse of the sampled
    sequences (all sequences of the DeepSeek-V3-shaped case) against the
    oracle's decode from its exact absorbed query; o of every head (and both
    queries of the two-token case) for 4 sequences, and 3 heads of 2 sequences
    in the non-absorbed form."""
    W = _W()
    w = W.preset(name)
    d = W.make_inputs(w)
    layer = _layer(w, d)
    o = _step(layer, d)
    assert layer.device_error() == 0
    seqs = W.sample_sequences(w, nseq)
    mask = seq_token_mask(w, seqs)
    pool, sc = oracle_pool(w, d, token_mask=mask)
    # cache bytes of the sampled sequences are bit-exact
    gcache = bits(layer.cache).reshape(pool.shape[0], -1)
    slots = d["ctx_slots"].numpy()[mask]
    assert np.array_equal(gcache[slots].view(np.uint8), pool[slots].view(np.uint8))
    _check_latent(w, d, pool, sc, f64(layer.u), layer.lse.cpu().numpy(), f64(layer.q_lat), seqs=seqs, what=name)
    og = f64(o)
    _check_o(w, d, og, pool, sc, seqs[:4])
    hs = [0, 37, 127] if w.heads == 128 else [0, 15]
    _check_o(w, d, og, pool, sc, seqs[:2], heads=hs)
