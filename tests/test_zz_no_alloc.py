"""The decode entry point that allocates nothing (mla_decode_paged_static_scratch).

Its split-KV partials live in one fixed device array of the library, so it is
checked bit for bit against mla_decode_paged (caller workspace) on the same
inputs and split count, for two calls in a row (the second call reuses the array the first
one left behind), and for the rejection of a problem whose partials do not fit.
This file is collected last so that it also runs after every other GPU test.
"""
import pytest
import torch


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


CASES = {
    # tcgen05 path: bf16, 128 heads, 64-token pages, forced split-KV
    "dsv3_bf16": dict(batch=4, seq_lens=[4096, 1500, 4096, 70], num_splits=8),
    # SIMT path: fp32, 16 heads, 256-token pages
    "tiny_fp32": dict(seq_lens=[1024, 600], num_splits=3),
}


def _setup(name):
    from mla_latent_kv_16_gb300 import workloads as W
    from mla_latent_kv_16_gb300.engine import build_layer, step_inputs
    w = W.preset(name, **CASES[name])
    d = W.make_inputs(w)
    layer = build_layer(w, d)
    layer.step(**step_inputs(d))  # writes the step's new tokens, completing every sequence
    torch.cuda.synchronize()
    return w, d, layer


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_workspace_decode_twice(name):
    from mla_latent_kv_16_gb300 import capi
    w, d, layer = _setup(name)
    assert layer.splits > 1  # the scratch array is really used
    need = capi.mla_decode_workspace_size(w.batch, w.q_len, w.max_pages_per_seq, w.page_size, w.num_splits,
                                          w.heads, w.cache_dtype)
    assert 0 < need <= capi.MLA_STATIC_SCRATCH_BYTES
    g = torch.Generator().manual_seed(77)
    for call in range(2):
        # a different query each call, so stale partials from call 0 would show in call 1
        q_lat = (torch.randn(w.batch, w.q_len, w.heads, 512, generator=g) * 0.5).to(layer.act).cuda()
        q_rope = (torch.randn(w.batch, w.q_len, w.heads, 64, generator=g) * 0.5).to(layer.act).cuda()
        u_ref, lse_ref = capi.mla_decode_paged(q_lat, q_rope, layer.cache, layer.scales, layer.block_table,
                                               layer.seq_lens, w.page_size, w.cache_dtype,
                                               num_splits=w.num_splits)
        u = torch.full_like(u_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        capi.mla_decode_paged_static_scratch(q_lat, q_rope, layer.cache, layer.scales, layer.block_table,
                                             layer.seq_lens, w.page_size, w.cache_dtype, num_splits=w.num_splits,
                                             u_out=u, lse_out=lse)
        torch.cuda.synchronize()
        # the same kernels on the same inputs and split count: identical bits
        assert torch.equal(u.view(torch.int16 if u.dtype == torch.bfloat16 else torch.int32),
                           u_ref.view(torch.int16 if u.dtype == torch.bfloat16 else torch.int32)), f"u call {call}"
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), f"lse call {call}"


def test_static_scratch_rejects_oversize_problem():
    from mla_latent_kv_16_gb300 import capi
    w, d, layer = _setup("dsv3_bf16")
    splits = 64
    need = capi.mla_decode_workspace_size(w.batch, w.q_len, w.max_pages_per_seq, w.page_size, splits, w.heads,
                                          w.cache_dtype)
    assert need > capi.MLA_STATIC_SCRATCH_BYTES
    q_lat = torch.zeros(w.batch, w.q_len, w.heads, 512, dtype=layer.act, device="cuda")
    q_rope = torch.zeros(w.batch, w.q_len, w.heads, 64, dtype=layer.act, device="cuda")
    u = torch.full((w.batch, w.q_len, w.heads, 512), 7.0, dtype=layer.act, device="cuda")
    with pytest.raises(capi.MlaError) as e:
        capi.mla_decode_paged_static_scratch(q_lat, q_rope, layer.cache, layer.scales, layer.block_table,
                                             layer.seq_lens, w.page_size, w.cache_dtype, num_splits=splits,
                                             u_out=u)
    assert e.value.status == capi.MLA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((u == 7.0).all())  # nothing was enqueued
