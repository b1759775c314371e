"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol include/mla.h declares, its host-only functions agree with the
oracle, and argument validation fails synchronously before any device work."""
import os
import re

import numpy as np
import pytest

from oracle import mla_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from mla_latent_kv_16_gb300 import build
    build.build()
    from mla_latent_kv_16_gb300 import capi as C
    C.load()
    return C


def _declared():
    txt = open(os.path.join(ROOT, "include", "mla.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", txt)))


def test_exports_every_declared_symbol(capi):
    L = capi.load()
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(capi.EXPORTED)


def test_version_and_status_strings(capi):
    assert capi.load().mla_version() >= 100
    assert capi.status_string(capi.MLA_OK) == "MLA_OK"
    assert capi.status_string(capi.MLA_ERR_WORKSPACE_TOO_SMALL) == "MLA_ERR_WORKSPACE_TOO_SMALL"


def test_rope_table_bitwise_equal_to_oracle(capi):
    cos, sin = capi.mla_rope_table(3000)
    oc, os_ = O.rope_tables(3000)
    assert np.array_equal(cos.numpy().view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(sin.numpy().view(np.uint32), os_.view(np.uint32))


def test_rope_table_rejects_bad_args(capi):
    L = capi.load()
    assert L.mla_rope_table(0, 64, 10000.0, None, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_rope_table(4, 63, 10000.0, None, None) == capi.MLA_ERR_INVALID_ARG


def test_split_policy_and_workspace(capi):
    # explicit split counts are honoured and clamped to the page count
    assert capi.mla_decode_num_splits(4, 1, 2048, 64, 128, 128, "bf16") == 128
    assert capi.mla_decode_num_splits(4, 1, 10, 64, 128, 128, "bf16") == 10
    s = capi.mla_decode_num_splits(32, 1, 64, 64, 0, 128, "bf16")
    assert 1 <= s <= 64
    # workspace: fp32 partials [B][Lq][S][H][512] + lse, 256-byte aligned pieces
    ws = capi.mla_decode_workspace_size(4, 1, 2048, 64, 128, 128, "bf16")
    rows = 4 * 1 * 128 * 128
    assert ws == rows * 512 * 4 + ((rows * 4 + 255) // 256) * 256
    assert capi.mla_decode_workspace_size(4, 1, 2048, 64, 1, 128, "bf16") == 0
    assert capi.mla_decode_num_splits(4, 0, 2048, 64, 0, 128, "bf16") < 1


def test_validation_fails_before_device_work(capi):
    """Calls with bad arguments return an error code without touching a GPU."""
    L = capi.load()
    bad_dims = capi.MlaDims(128, 128, 256, 64, 128)
    assert L.mla_absorb_q(None, None, None, 4, bad_dims, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_absorb_q(None, None, None, 4, capi.dims(128), capi.MLA_E4M3, None) == capi.MLA_ERR_UNSUPPORTED
    assert L.mla_out_proj(None, None, None, -1, capi.dims(128), capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_absorb_q(None, None, None, 0, capi.dims(128), capi.MLA_BF16, None) == capi.MLA_OK  # no-op
    # E4M3 cache without scales, and an fp32 activation with an E4M3 cache
    assert L.mla_decode_paged(16, 16, 16, None, 16, 16, 1, 1, 1, 1, 64, 0.1, 0, None, 0, 16, None, None,
                              capi.dims(128), capi.MLA_BF16, capi.MLA_E4M3, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_decode_paged(16, 16, 16, 16, 16, 16, 1, 1, 1, 1, 64, 0.1, 0, None, 0, 16, None, None,
                              capi.dims(128), capi.MLA_F32, capi.MLA_E4M3, None) == capi.MLA_ERR_UNSUPPORTED
    # workspace too small for an explicit split count
    assert L.mla_decode_paged(16, 16, 16, None, 16, 16, 2, 1, 8, 16, 64, 0.1, 4, None, 0, 16, None, None,
                              capi.dims(128), capi.MLA_BF16, capi.MLA_BF16, None) == capi.MLA_ERR_WORKSPACE_TOO_SMALL
    assert L.mla_cache_append(16, 16, 16, 16, 16, 16, 1, 8, 16, None, 1, 64, capi.MLA_BF16, capi.MLA_E4M3, None,
                              None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_decode_paged(16, 16, 16, None, 16, 16, 1, 1, 1, 1, 64, float("nan"), 0, None, 0, 16, None, None,
                              capi.dims(128), capi.MLA_BF16, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG


def test_decode_out_proj_validation(capi):
    """mla_decode_out_proj: mla_decode_paged's checks, then a missing or
    misaligned W_UV / o buffer, all before any device work."""
    L = capi.load()
    D = capi.dims(128)
    args = (16, 16, 16, None, 16, 16, 1, 1, 1, 1, 64, 0.1, 0, None, 0)
    # decode's own checks come first: an E4M3 cache without scales
    assert L.mla_decode_out_proj(16, 16, 16, None, 16, 16, 1, 1, 1, 1, 64, 0.1, 0, None, 0, 16, 16, None, 16, None,
                                 D, capi.MLA_BF16, capi.MLA_E4M3, None) == capi.MLA_ERR_INVALID_ARG
    # no W_UV, no o, a misaligned o
    assert L.mla_decode_out_proj(*args, None, 16, None, 16, None, D, capi.MLA_BF16, capi.MLA_BF16, None) == \
        capi.MLA_ERR_INVALID_ARG
    assert L.mla_decode_out_proj(*args, 16, 16, None, None, None, D, capi.MLA_BF16, capi.MLA_BF16, None) == \
        capi.MLA_ERR_INVALID_ARG
    assert L.mla_decode_out_proj(*args, 16, 16, None, 24, None, D, capi.MLA_BF16, capi.MLA_BF16, None) == \
        capi.MLA_ERR_INVALID_ARG
    # workspace too small for an explicit split count
    assert L.mla_decode_out_proj(16, 16, 16, None, 16, 16, 2, 1, 8, 16, 64, 0.1, 4, None, 0, 16, 16, None, 16, None,
                                 D, capi.MLA_BF16, capi.MLA_BF16, None) == capi.MLA_ERR_WORKSPACE_TOO_SMALL
    # an empty batch is a no-op
    assert L.mla_decode_out_proj(None, None, None, None, None, None, 0, 1, 1, 1, 64, 0.1, 0, None, 0, None, None,
                                 None, None, None, D, capi.MLA_BF16, capi.MLA_BF16, None) == capi.MLA_OK


def test_fused_projection_validation(capi):
    """mla_fuse_out_weights / mla_out_proj_fused reject bad arguments before any
    device work; the workspace size covers one fp32 partial per K split."""
    L = capi.load()
    D = capi.dims(128)
    assert L.mla_fuse_out_weights(16, 16, 16, 0, D, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_fuse_out_weights(16, 16, 16, 7168, D, capi.MLA_E4M3, None) == capi.MLA_ERR_UNSUPPORTED
    assert L.mla_fuse_out_weights(None, 16, 16, 7168, D, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_fuse_out_weights(16, 16, 24, 7168, D, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_out_proj_fused(None, None, None, 0, 7168, None, 0, D, capi.MLA_BF16, None) == capi.MLA_OK
    assert L.mla_out_proj_fused(16, 16, 16, 4, 1 << 17, None, 0, D, capi.MLA_BF16, None) == \
        capi.MLA_ERR_INVALID_ARG
    need = capi.mla_out_proj_fused_workspace_size(32, 7168, 128)
    assert need > 0 and need % 256 == 0 and need % (32 * 7168 * 4) == 0
    assert L.mla_out_proj_fused(16, 16, 16, 32, 7168, None, 0, D, capi.MLA_BF16, None) == \
        capi.MLA_ERR_WORKSPACE_TOO_SMALL
    # the CUDA-core shapes (fp32, or n_in not a multiple of 64) never split K
    assert capi.mla_out_proj_fused_workspace_size(32, 7168, 128, "f32") == 0
    assert capi.mla_linear_workspace_size(32, 7000, 100) == 0
    assert capi.mla_linear_workspace_size(32, 7000, 7168) % (32 * 7000 * 4) == 0


def test_linear_and_front_validation(capi):
    L = capi.load()
    D = capi.dims(128)
    assert L.mla_linear(16, 16, 16, 4, 0, 64, None, 0, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_linear(16, 16, 16, 4, 64, 64, None, 0, capi.MLA_E4M3, None) == capi.MLA_ERR_UNSUPPORTED
    assert L.mla_linear(16, 16, 24, 4, 64, 64, None, 0, capi.MLA_BF16, None) == capi.MLA_ERR_INVALID_ARG
    assert L.mla_linear(None, None, None, 0, 64, 64, None, 0, capi.MLA_BF16, None) == capi.MLA_OK
    assert L.mla_linear(16, 16, 16, 32, 2112, 7168, None, 0, capi.MLA_BF16, None) == capi.MLA_ERR_WORKSPACE_TOO_SMALL
    args = [16] * 8
    ok = dict(max_pos=100, eps=1e-6, n=4, d=7168, dcq=1536)

    def front(max_pos=100, eps=1e-6, n=4, d=7168, dcq=1536, ws=16, ws_bytes=1 << 30, act=capi.MLA_BF16, outs=16):
        return L.mla_decode_front(*args, max_pos, eps, n, d, dcq, outs, 16, 16, 16, ws, ws_bytes, None, D, act, None)

    assert front(max_pos=0) == capi.MLA_ERR_INVALID_ARG
    assert front(eps=-1.0) == capi.MLA_ERR_INVALID_ARG
    assert front(eps=float("nan")) == capi.MLA_ERR_INVALID_ARG
    assert front(dcq=0) == capi.MLA_ERR_INVALID_ARG
    assert front(act=capi.MLA_E4M3) == capi.MLA_ERR_UNSUPPORTED
    assert front(outs=None) == capi.MLA_ERR_INVALID_ARG
    assert front(outs=24) == capi.MLA_ERR_INVALID_ARG
    assert front(ws_bytes=16) == capi.MLA_ERR_WORKSPACE_TOO_SMALL
    assert front(n=0) == capi.MLA_OK
    # workspace: the fp32 sums of both products plus c_q
    need = capi.mla_decode_front_workspace_size(32, 7168, 1536, 128)
    assert need >= 32 * (2112 + 24576) * 4 + 32 * 1536 * 2


def test_static_scratch_checks_arguments_before_its_size(capi):
    """mla_decode_paged_static_scratch returns mla_decode_paged's argument errors
    even for a problem whose partials would not fit its scratch array."""
    L = capi.load()
    D = capi.dims(128)
    # 64 sequences x 64 splits x 128 heads of fp32 partials: far beyond the array
    big = (64, 1, 64, 4096, 64, 0.1, 64)
    assert capi.mla_decode_workspace_size(64, 1, 64, 64, 64, 128, "bf16") > capi.MLA_STATIC_SCRATCH_BYTES

    def call(act, cache_dt, scales=16, q=16):
        B, Lq, maxp, npages, page, sc, splits = big
        return L.mla_decode_paged_static_scratch(q, 16, 16, scales, 16, 16, B, Lq, maxp, npages, page, sc, splits,
                                                 16, None, None, D, act, cache_dt, None)
    assert call(capi.MLA_F32, capi.MLA_E4M3) == capi.MLA_ERR_UNSUPPORTED       # fp32 activations, E4M3 cache
    assert call(capi.MLA_BF16, capi.MLA_E4M3, scales=None) == capi.MLA_ERR_INVALID_ARG  # E4M3 without scales
    assert call(capi.MLA_BF16, capi.MLA_BF16, scales=None, q=None) == capi.MLA_ERR_INVALID_ARG   # missing q_lat
    assert call(capi.MLA_BF16, capi.MLA_BF16, scales=None, q=8) == capi.MLA_ERR_INVALID_ARG      # misaligned q_lat
    assert call(capi.MLA_BF16, capi.MLA_BF16, scales=None) == capi.MLA_ERR_WORKSPACE_TOO_SMALL  # valid, too big
    # the same answers from mla_decode_paged (with no workspace)
    B, Lq, maxp, npages, page, sc, splits = big
    assert L.mla_decode_paged(16, 16, 16, 16, 16, 16, B, Lq, maxp, npages, page, sc, splits, None, 0, 16, None, None,
                              D, capi.MLA_F32, capi.MLA_E4M3, None) == capi.MLA_ERR_UNSUPPORTED


def test_decode_kernel_path_query(capi):
    """The kernel-choice query: argument errors, and the CUDA-core kernel for
    the cases the tensor-core kernel does not take (fp32, 16 heads, 100-token pages)."""
    L = capi.load()
    import ctypes
    out = ctypes.c_int32(0)
    assert L.mla_decode_kernel_path(16, None, 4, 64, capi.dims(128), capi.MLA_BF16, capi.MLA_BF16,
                                    None) == capi.MLA_ERR_INVALID_ARG
    for dims_, act, page in ((capi.dims(16), capi.MLA_F32, 256), (capi.dims(16), capi.MLA_BF16, 64),
                             (capi.dims(128), capi.MLA_BF16, 100)):
        assert L.mla_decode_kernel_path(16, None, 4, page, dims_, act, act, ctypes.byref(out)) == capi.MLA_OK
        assert out.value == capi.MLA_DECODE_PATH_CUDA_CORE
