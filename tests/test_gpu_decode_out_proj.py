"""mla_decode_out_proj: the decode and the value up-projection as one call.

With 2 to 4 KV splits on the tensor-core decode the split merge runs inside the
projection kernel; the call promises the bits of mla_decode_paged followed by
mla_out_proj (the same merge arithmetic, the same bf16 u, the same MMAs). Also
checked against the oracle end to end, and for split counts and paths where the
call simply runs the two kernels back to back.
"""
import pytest
import torch

from _util import assert_close, f64, oracle_pool, tol_for
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


def _setup(preset, **kw):
    from mla_latent_kv_16_gb300 import workloads as W
    from mla_latent_kv_16_gb300.engine import build_layer, step_inputs
    w = W.preset(preset, **kw)
    d = W.make_inputs(w)
    layer = build_layer(w, d)
    layer.step(**step_inputs(d))  # writes the step's new tokens, completing every sequence
    torch.cuda.synchronize()
    return w, d, layer


def _same_bits(x, y):
    it = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
    return torch.equal(x.view(it), y.view(it))


CASES = [
    ("dsv3_bf16", dict(batch=32, seq_lens=None, num_splits=2)),  # the DeepSeek-V3 step: 32 tokens, one tile
    ("dsv3_bf16", dict(batch=5, seq_lens=[1000, 77, 4096, 1, 2049], num_splits=3)),
    ("dsv3_bf16", dict(batch=3, seq_lens=[1000, 77, 4096], num_splits=4)),  # empty later splits
    ("dsv3_bf16", dict(batch=70, seq_lens=None, num_splits=2)),  # two token tiles, the second ragged
    ("fp8_lq2", dict(batch=40, seq_lens=None, num_splits=2)),  # E4M3 cache, 80 query rows
    ("dsv3_bf16", dict(batch=4, seq_lens=[3000, 17, 640, 2049], num_splits=1)),  # no merge
    ("dsv3_bf16", dict(batch=4, seq_lens=[3000, 17, 640, 2049], num_splits=7)),  # merge kernel
    ("tiny_fp32", dict()),  # CUDA-core path
]


@pytest.mark.parametrize("preset,kw", CASES, ids=lambda v: str(v))
def test_fused_call_matches_two_calls_bit_for_bit(preset, kw):
    from mla_latent_kv_16_gb300 import capi
    kw = {k: v for k, v in kw.items() if v is not None}
    if "seq_lens" not in kw and "batch" in kw and preset != "tiny_fp32":
        kw["seq_lens"] = [300 + 97 * i for i in range(kw["batch"])]
    w, d, layer = _setup(preset, **kw)
    g = torch.Generator().manual_seed(3)
    q_lat = (torch.randn(w.batch, w.q_len, w.heads, 512, generator=g) * 0.5).to(layer.act).cuda()
    q_rope = (torch.randn(w.batch, w.q_len, w.heads, 64, generator=g) * 0.5).to(layer.act).cuda()
    args = (q_lat, q_rope, layer.cache, layer.scales, layer.block_table, layer.seq_lens, w.page_size, w.cache_dtype)
    u_ref, lse_ref = capi.mla_decode_paged(*args, num_splits=w.num_splits)
    o_ref = capi.mla_out_proj(u_ref, layer.w_uv)
    u, lse, o = capi.mla_decode_out_proj(*args, layer.w_uv, num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert _same_bits(u, u_ref)
    assert _same_bits(lse, lse_ref)
    assert _same_bits(o, o_ref)
    assert torch.isfinite(o.float()).all()
    assert layer.device_error() == 0


def test_fused_step_against_oracle():
    """The layer's step (append, absorb, decode_out_proj) end to end against the
    oracle's exact decode and up-projection, from the oracle's own inputs."""
    w, d, layer = _setup("dsv3_bf16", batch=6, seq_lens=[4096, 1, 65, 700, 2049, 129], num_splits=2)
    assert layer.splits == 2
    pool, sc = oracle_pool(w, d)
    q_ex = O.absorb_q(f64(d["q_nope"]), f64(d["w_uk"]))
    ref = O.decode_latent(q_ex, f64(d["q_rope"]), pool, sc, d["block_table"].numpy(), list(w.seq_lens), w.q_len,
                          w.page_size, w.cache_dtype, O.default_scale())
    w_uv = f64(d["w_uv"])
    o = f64(layer.o)
    for b, (ru, _) in ref.items():
        ro = O.out_proj(ru, w_uv)
        assert_close(o[b], ro, **tol_for(w), what=f"o seq {b}")
