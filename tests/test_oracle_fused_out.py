"""Pins for the oracle's fused output projection (W~ = W_O W_UV per head, then
one contraction over all heads): brute-force loops from the definition on
tiny shapes, the identity with the unfused projection and with the
materialised attention, and an identity output projection. CPU only."""
import math

import numpy as np

from oracle import mla_oracle as O


def _loops_fused(w_o2d, w_uv):
    """W~_i = (column block i of W_O) @ W_UV[i], with W_O given as the plain
    d x (H d_v) matrix, in scalar loops with math.fsum."""
    d = w_o2d.shape[0]
    H, d_v, d_c = w_uv.shape
    out = np.empty((d, H, d_c))
    for m in range(d):
        for i in range(H):
            for c in range(d_c):
                out[m, i, c] = math.fsum(w_o2d[m, i * d_v + e] * w_uv[i, e, c] for e in range(d_v))
    return out


def _tiny(seed=0, d=5, H=3, d_v=4, d_c=6):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((d, H * d_v)), rng.standard_normal((H, d_v, d_c))


def test_fused_weight_matches_column_block_loops():
    w_o2d, w_uv = _tiny()
    d, H, d_v = 5, 3, 4
    got = O.fuse_out_weights(w_o2d.reshape(d, H, d_v), w_uv)
    ref = _loops_fused(w_o2d, w_uv)
    assert np.max(np.abs(got - ref)) <= 1e-14 * np.max(np.abs(ref))


def test_fused_output_matches_loops():
    """y[m] = sum over heads and latent columns of W~[m,h,c] u[h,c], by loops."""
    rng = np.random.default_rng(1)
    w_f = rng.standard_normal((5, 3, 6))
    u = rng.standard_normal((2, 3, 6))
    got = O.out_proj_fused(u, w_f)
    for t in range(2):
        for m in range(5):
            ref = math.fsum(w_f[m, h, c] * u[t, h, c] for h in range(3) for c in range(6))
            assert abs(got[t, m] - ref) <= 1e-14 * max(1.0, abs(ref))


def test_fused_equals_unfused_projection():
    """Associativity: W~ u == W_O concat_h(W_UV[h] u_h) at the real head sizes."""
    rng = np.random.default_rng(2)
    H, d = 4, 96
    w_o = rng.standard_normal((d, H, 128)) / math.sqrt(H * 128)
    w_uv = rng.standard_normal((H, 128, 512)) / math.sqrt(512)
    u = rng.standard_normal((2, 3, H, 512))
    y_f = O.out_proj_fused(u, O.fuse_out_weights(w_o, w_uv))
    y_u = O.out_proj_model(O.out_proj(u, w_uv), w_o)
    assert y_f.shape == (2, 3, d)
    assert np.max(np.abs(y_f - y_u)) <= 1e-12 * np.max(np.abs(y_u))


def test_identity_output_projection_returns_head_outputs():
    """d = H*128 and W_O[m,h,e] = [m == 128 h + e]: y is the concatenation of the
    per-head outputs W_UV[h] u_h, in head order."""
    rng = np.random.default_rng(3)
    H = 3
    w_o = np.eye(H * 128).reshape(H * 128, H, 128)
    w_uv = rng.standard_normal((H, 128, 512))
    u = rng.standard_normal((4, H, 512))
    y = O.out_proj_fused(u, O.fuse_out_weights(w_o, w_uv))
    o = np.stack([np.stack([w_uv[h] @ u[t, h] for h in range(H)]) for t in range(4)])
    assert np.max(np.abs(y - o.reshape(4, H * 128))) <= 1e-13 * np.max(np.abs(o))


def test_fused_layer_equals_materialised_attention():
    """The decode output in the model dimension two ways: K and V materialised per
    head, then W_O over the concatenated heads; or the absorbed latent sum u
    times the fused weight."""
    rng = np.random.default_rng(4)
    H, T, d = 4, 17, 64
    q_nope = rng.standard_normal((H, 128))
    q_rope = rng.standard_normal((H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) / math.sqrt(512)
    w_uv = rng.standard_normal((H, 128, 512)) / math.sqrt(512)
    w_o = rng.standard_normal((d, H, 128)) / math.sqrt(H * 128)
    rows = rng.standard_normal((T, 576))
    sc = O.default_scale()
    o, _, _ = O.attend_nonabsorbed(q_nope, q_rope, w_uk, w_uv, rows, sc)
    u, _ = O.attend_absorbed(O.absorb_q(q_nope, w_uk), q_rope, rows, sc)
    y_mat = O.out_proj_model(o, w_o)
    y_abs = O.out_proj_fused(u, O.fuse_out_weights(w_o, w_uv))
    assert np.max(np.abs(y_mat - y_abs)) <= 1e-12 * np.max(np.abs(y_mat))


def test_fused_pins_catch_planted_mistakes(monkeypatch):
    """Index mistakes planted in the fused weight fail the loop pin."""
    w_o2d, w_uv = _tiny(seed=5, d=4, H=3, d_v=3, d_c=5)
    ref = _loops_fused(w_o2d, w_uv)
    good = O.fuse_out_weights(w_o2d.reshape(4, 3, 3), w_uv)
    assert np.allclose(good, ref, rtol=1e-13, atol=0)
    # 1) W_O's columns read head-minor ([d, d_v, H]) instead of head-major
    bad = O.fuse_out_weights(w_o2d.reshape(4, 3, 3).transpose(0, 2, 1), w_uv)
    assert not np.allclose(bad, ref)
    # 2) W_UV of the next head paired with each column block
    bad = O.fuse_out_weights(w_o2d.reshape(4, 3, 3), np.roll(w_uv, 1, axis=0))
    assert not np.allclose(bad, ref)
    # 3) W_UV[h] used transposed (square blocks make that shape-compatible)
    w_sq = np.random.default_rng(6).standard_normal((3, 3, 3))
    ref_sq = _loops_fused(w_o2d, w_sq)
    monkeypatch.setattr(O, "fuse_out_weights",
                        lambda a, b: np.einsum("mhe,hce->mhc", np.asarray(a, np.float64), np.asarray(b, np.float64)))
    assert not np.allclose(O.fuse_out_weights(w_o2d.reshape(4, 3, 3), w_sq), ref_sq)
