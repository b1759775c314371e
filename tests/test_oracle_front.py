"""Pins for the oracle's decode-layer front end (RMSNorm, the query and KV
projections, the query's RoPE): a library RMSNorm, closed forms, complex
multiplication for the rotation, and scalar loops on tiny shapes. CPU only."""
import math

import numpy as np
import torch

from oracle import mla_oracle as O


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 1536)) * 3.0
    g = 1.0 + 0.1 * rng.standard_normal(1536)
    for eps in (0.0, 2.0 ** -23, 1e-2):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (1536,), torch.from_numpy(g), eps).numpy()
        assert np.allclose(O.rms_norm(x, g, eps), ref, rtol=1e-14, atol=1e-14)


def test_rms_norm_closed_forms():
    g = np.linspace(0.5, 2.0, 8)
    # a constant vector c*1 normalises to sign(c) * gamma (eps = 0)
    assert np.allclose(O.rms_norm(np.full(8, -3.7), g, 0.0), -g, rtol=1e-15)
    # with gamma = 1 the output has unit RMS, and scaling the input changes nothing
    x = np.random.default_rng(1).standard_normal(512)
    y = O.rms_norm(x, np.ones(512), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    assert np.allclose(O.rms_norm(5.0 * x, np.ones(512), 0.0), y, rtol=1e-14)
    # eps adds to the mean square: a zero vector stays zero, a unit-RMS one shrinks by 1/sqrt(1+eps)
    assert np.array_equal(O.rms_norm(np.zeros(4), np.ones(4), 1e-6), np.zeros(4))
    assert np.allclose(O.rms_norm(y, np.ones(512), 0.25), y / math.sqrt(1.25), rtol=1e-14)


def _tiny_front(seed=2, n=3, d=6, d_cq=5, H=2):
    rng = np.random.default_rng(seed)
    return dict(h=rng.standard_normal((n, d)), w_dq=rng.standard_normal((d_cq, d)),
                g_q=1 + 0.1 * rng.standard_normal(d_cq), w_uq=rng.standard_normal((H * 128, d_cq)),
                w_qr=rng.standard_normal((H * 64, d_cq)), w_dkv=rng.standard_normal((512, d)),
                g_kv=1 + 0.1 * rng.standard_normal(512), w_kr=rng.standard_normal((64, d)),
                positions=np.array([0, 7, 4095])[:n])


def test_front_end_by_loops():
    """Scalar loops from the module's definition on tiny widths."""
    a = _tiny_front()
    eps = 1e-6
    q_nope, q_rope, c_kv, k_r = O.decode_front(**a, eps=eps)
    n, d = a["h"].shape
    d_cq = a["w_dq"].shape[0]
    for t in range(n):
        cq = [math.fsum(a["w_dq"][i, j] * a["h"][t, j] for j in range(d)) for i in range(d_cq)]
        inv = 1.0 / math.sqrt(math.fsum(v * v for v in cq) / d_cq + eps)
        cq = [cq[i] * inv * a["g_q"][i] for i in range(d_cq)]
        for hh, dd in ((0, 0), (1, 127), (1, 5)):
            ref = math.fsum(a["w_uq"][hh * 128 + dd, i] * cq[i] for i in range(d_cq))
            assert abs(q_nope[t, hh, dd] - ref) <= 1e-12 * max(1.0, abs(ref))
        # RoPE of pair i of head 1: angle pos * 10000^(-2i/64), adjacent elements
        for i in (0, 13, 31):
            x0 = math.fsum(a["w_qr"][64 + 2 * i, k] * cq[k] for k in range(d_cq))
            x1 = math.fsum(a["w_qr"][64 + 2 * i + 1, k] * cq[k] for k in range(d_cq))
            th = a["positions"][t] * 10000.0 ** (-2.0 * i / 64)
            assert abs(q_rope[t, 1, 2 * i] - (x0 * math.cos(th) - x1 * math.sin(th))) <= 1e-11 * max(1, abs(x0) + abs(x1))
            assert abs(q_rope[t, 1, 2 * i + 1] - (x0 * math.sin(th) + x1 * math.cos(th))) <= 1e-11 * max(1, abs(x0) + abs(x1))
        ckv = [math.fsum(a["w_dkv"][i, j] * a["h"][t, j] for j in range(d)) for i in range(512)]
        inv = 1.0 / math.sqrt(math.fsum(v * v for v in ckv) / 512 + eps)
        for i in (0, 200, 511):
            assert abs(c_kv[t, i] - ckv[i] * inv * a["g_kv"][i]) <= 1e-12
        for r in (0, 63):
            assert abs(k_r[t, r] - math.fsum(a["w_kr"][r, j] * a["h"][t, j] for j in range(d))) <= 1e-12


def test_front_query_rope_matches_complex_multiplication():
    """q_rope is the complex product of adjacent pairs with e^{i pos theta_k}, as
    the module's apply_rope computes it (here in complex128)."""
    a = _tiny_front(seed=3)
    q_nope, q_rope, _, _ = O.decode_front(**a, eps=0.0)
    c_q = O.rms_norm(a["h"] @ a["w_dq"].T, a["g_q"], 0.0)
    raw = torch.from_numpy((c_q @ a["w_qr"].T).reshape(3, 2, 32, 2))
    theta = torch.tensor([10000.0 ** (-2.0 * k / 64) for k in range(32)], dtype=torch.float64)
    ang = torch.from_numpy(a["positions"].astype(np.float64))[:, None, None] * theta
    rot = torch.view_as_real(torch.view_as_complex(raw) * torch.polar(torch.ones_like(ang), ang)).reshape(3, 2, 64)
    assert np.allclose(q_rope, rot.numpy(), rtol=1e-12, atol=1e-12)


def test_front_pins_catch_planted_mistakes():
    a = _tiny_front(seed=4)
    good = O.decode_front(**a, eps=0.0)
    # 1) RoPE applied to the two halves (i, i + 32) instead of adjacent pairs
    c_q = O.rms_norm(a["h"] @ a["w_dq"].T, a["g_q"], 0.0)
    raw = (c_q @ a["w_qr"].T).reshape(3, 2, 64)
    half = np.concatenate([raw[..., 0::2], raw[..., 1::2]], -1)
    bad = np.stack([O.rope_rotate_f64(half[t], float(a["positions"][t])) for t in range(3)])
    assert not np.allclose(bad, good[1])
    # 2) the norm taken before the projection instead of after
    bad_c = O.rms_norm(a["h"], np.ones(a["h"].shape[1]), 0.0) @ a["w_dkv"].T * a["g_kv"]
    assert not np.allclose(bad_c, good[2])
    # 3) mean of |x| instead of mean of x^2
    x = a["h"] @ a["w_dkv"].T
    bad_n = x / np.mean(np.abs(x), -1, keepdims=True) * a["g_kv"]
    assert not np.allclose(bad_n, good[2])


def test_linear_by_loops():
    rng = np.random.default_rng(5)
    x, w = rng.standard_normal((3, 7)), rng.standard_normal((4, 7))
    y = O.linear(x, w)
    for t in range(3):
        for o in range(4):
            assert abs(y[t, o] - math.fsum(w[o, i] * x[t, i] for i in range(7))) <= 1e-14
