"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix (printed figures, closed forms, library routines, brute force), never
against the oracle itself. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _eval(case):
    return getattr(O, case["formula"])(**case["args"])


# --------------------------------------------------------------------------- bytes

@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["id"])
def test_printed_cache_bytes(case):
    v = _eval(case) / case["unit"]
    if case.get("rounding") == "floor":
        assert math.floor(v) == case["printed"], (v, case["citation"])
    elif case["tol"] == 0:
        assert v == case["printed"], (v, case["citation"])
    else:
        assert abs(v - case["printed"]) <= case["tol"], (v, case["citation"])


@pytest.mark.parametrize("r", _golden()["ratios"], ids=lambda c: c["id"])
def test_printed_ratios(r):
    cases = {c["id"]: _eval(c) for c in _golden()["cases"]}
    q = cases[r["num"]] / cases[r["den"]]
    if "printed_pct_reduction" in r:
        assert round(100 * (1 - q), r["decimals"]) == r["printed_pct_reduction"]
    else:
        assert round(q, r["decimals"]) == r["printed_times"]


def test_inconsistent_figures_documented():
    for c in _golden()["inconsistent"]:
        assert _eval(c) == c["formula_gives"]


def test_row_bytes_per_dtype():
    # 576 values per token: 2304 B fp32, 1152 B bf16, 576 B e4m3 (+20 B of scales)
    assert O.mla_bytes_per_token(4) == 2304
    assert O.mla_bytes_per_token(2) == 1152
    assert O.mla_bytes_per_token(1) == 576
    assert len(O.E4M3_GROUPS) * 4 == 20


# --------------------------------------------------------------------------- formats

def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32) * 10.0 ** g.integers(-30, 30, 200000),
        # exact ties: bf16 value + half an ulp
        (np.arange(1, 5000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        (np.arange(1, 5000, dtype=np.uint32) << 16 | 0x7FFF).view(np.float32),
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(x), ref)


def test_e4m3_known_codes():
    assert O.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert O.e4m3_decode(np.uint8(0x38)) == 1.0
    assert O.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert O.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9
    assert O.e4m3_decode(np.uint8(0xFE)) == -448.0
    assert np.isnan(O.e4m3_decode(np.uint8(0x7F)))
    assert np.isnan(O.e4m3_decode(np.uint8(0xFF)))


def test_e4m3_all_codes_roundtrip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    back = O.e4m3_encode(vals.astype(np.float32))
    assert np.array_equal(back, codes)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_decode(codes)
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.all(both_nan | (ref == mine))


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.default_rng(1)
    grid = O.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2                       # exact ties
    x = np.concatenate([
        g.uniform(-448, 448, 300000),
        g.standard_normal(300000) * 10.0 ** g.uniform(-4, 2, 300000),
        mids, -mids, grid, -grid,
        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 1e4, 3e38], dtype=np.float32)
    assert np.all(O.e4m3_encode(x) == 0x7E)
    assert np.all(O.e4m3_encode(-x) == 0xFE)
    assert O.e4m3_encode(np.float32(-0.0)) == 0x80


# --------------------------------------------------------------------------- RoPE

def test_rope_table_spot_values():
    cos_t, sin_t = O.rope_tables(300)
    for p, i in [(0, 0), (1, 0), (7, 3), (255, 31), (299, 17)]:
        th = p * 10000.0 ** (-2.0 * i / 64)
        assert cos_t[p, i] == np.float32(math.cos(th))
        assert sin_t[p, i] == np.float32(math.sin(th))
    assert np.all(cos_t[0] == 1.0) and np.all(sin_t[0] == 0.0)


def test_rope_position_zero_is_identity_bit_exact():
    cos_t, sin_t = O.rope_tables(4)
    k = np.random.default_rng(2).standard_normal((5, 64)).astype(np.float32)
    out = O.rope_rotate_f32(k, np.zeros(5, dtype=np.int64), cos_t, sin_t)
    assert np.array_equal(out.view(np.uint32), k.view(np.uint32))


def test_rope_matches_complex_multiplication():
    # adjacent pairs as complex numbers times e^{i*pos*theta} (complex view)
    cos_t, sin_t = O.rope_tables(1000)
    g = np.random.default_rng(3)
    k = g.standard_normal((50, 64)).astype(np.float32)
    pos = g.integers(0, 1000, 50)
    z = k[:, 0::2].astype(np.float64) + 1j * k[:, 1::2].astype(np.float64)
    rot = z * (cos_t[pos].astype(np.float64) + 1j * sin_t[pos].astype(np.float64))
    ref = np.empty((50, 64))
    ref[:, 0::2] = rot.real
    ref[:, 1::2] = rot.imag
    out = O.rope_rotate_f32(k, pos, cos_t, sin_t).astype(np.float64)
    assert np.max(np.abs(out - ref)) <= 4 * np.finfo(np.float32).eps * np.max(np.abs(ref))


def test_rope_preserves_pair_norms_and_is_relative():
    g = np.random.default_rng(4)
    q = g.standard_normal(64)
    k = g.standard_normal(64)
    for m in (0, 3, 100):
        rq = O.rope_rotate_f64(q, m)
        assert np.allclose(rq[0::2] ** 2 + rq[1::2] ** 2, q[0::2] ** 2 + q[1::2] ** 2, rtol=1e-13)
    d1 = O.rope_rotate_f64(q, 50) @ O.rope_rotate_f64(k, 20)
    d2 = O.rope_rotate_f64(q, 130) @ O.rope_rotate_f64(k, 100)
    d3 = O.rope_rotate_f64(q, 30) @ O.rope_rotate_f64(k, 0)
    assert abs(d1 - d2) < 1e-11 and abs(d1 - d3) < 1e-11


# --------------------------------------------------------------------------- attention

def _rand_case(H=4, T=37, seed=5):
    g = np.random.default_rng(seed)
    q_nope = g.standard_normal((H, 128))
    q_rope = g.standard_normal((H, 64))
    w_uk = g.standard_normal((H, 128, 512)) / math.sqrt(512)
    w_uv = g.standard_normal((H, 128, 512)) / math.sqrt(512)
    rows = g.standard_normal((T, 576))
    return q_nope, q_rope, w_uk, w_uv, rows


def test_absorbed_equals_nonabsorbed():
    q_nope, q_rope, w_uk, w_uv, rows = _rand_case()
    sc = O.default_scale()
    o, u, lse = O.attend_nonabsorbed(q_nope, q_rope, w_uk, w_uv, rows, sc)
    u2, lse2 = O.attend_absorbed(O.absorb_q(q_nope, w_uk), q_rope, rows, sc)
    o2 = O.out_proj(u2, w_uv)
    assert np.max(np.abs(u - u2)) <= 1e-12 * np.max(np.abs(u))
    assert np.max(np.abs(o - o2)) <= 1e-12 * np.max(np.abs(o))
    assert np.max(np.abs(lse - lse2)) <= 1e-12 * np.max(np.abs(lse))


def test_scale_is_one_over_sqrt_192():
    assert O.default_scale() == 1.0 / math.sqrt(192.0)


def test_single_token_sequence():
    q_nope, q_rope, w_uk, w_uv, rows = _rand_case(T=1)
    o, u, lse = O.attend_nonabsorbed(q_nope, q_rope, w_uk, w_uv, rows, O.default_scale())
    assert np.array_equal(u, np.broadcast_to(rows[0, :512], u.shape))
    assert np.allclose(o, w_uv @ rows[0, :512], rtol=0, atol=1e-14)


def test_mqa_reduction_matches_torch_sdpa():
    """W_UK[h] = W_UV[h] = [I_128 | 0]: each head attends with key [c[:128]; k_R]
    and value c[:128] shared by all heads -- textbook MQA, which torch's
    scaled_dot_product_attention computes in float64."""
    H, T = 6, 23
    q_nope, q_rope, _, _, rows = _rand_case(H=H, T=T, seed=6)
    eye = np.zeros((H, 128, 512))
    eye[:, :, :128] = np.eye(128)
    o, _, _ = O.attend_nonabsorbed(q_nope, q_rope, eye, eye, rows, O.default_scale())
    q = torch.from_numpy(np.concatenate([q_nope, q_rope], 1))[None, :, None, :]     # [1,H,1,192]
    k = torch.from_numpy(np.concatenate([rows[:, :128], rows[:, 512:]], 1))[None, None].expand(1, H, T, 192)
    v = torch.from_numpy(rows[:, :128])[None, None].expand(1, H, T, 128)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=1 / math.sqrt(192))
    assert np.allclose(o, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_zero_q_rope_ignores_k_r():
    q_nope, q_rope, w_uk, w_uv, rows = _rand_case(seed=7)
    rows2 = rows.copy()
    rows2[:, 512:] = np.random.default_rng(8).standard_normal((rows.shape[0], 64)) * 100
    z = np.zeros_like(q_rope)
    a = O.attend_nonabsorbed(q_nope, z, w_uk, w_uv, rows, O.default_scale())
    b = O.attend_nonabsorbed(q_nope, z, w_uk, w_uv, rows2, O.default_scale())
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    # and with q_rope != 0 the rope rows do matter
    c = O.attend_nonabsorbed(q_nope, q_rope, w_uk, w_uv, rows2, O.default_scale())
    assert not np.allclose(a[0], c[0])


def test_brute_force_tiny():
    """Scalar loops with math.fsum for 2 heads x 5 tokens, against the oracle."""
    q_nope, q_rope, w_uk, w_uv, rows = _rand_case(H=2, T=5, seed=9)
    sc = 1.0 / math.sqrt(192)
    o, u, lse = O.attend_nonabsorbed(q_nope, q_rope, w_uk, w_uv, rows, sc)
    for h in range(2):
        s = []
        for t in range(5):
            kc = [math.fsum(w_uk[h, d, c] * rows[t, c] for c in range(512)) for d in range(128)]
            dot = math.fsum([q_nope[h, d] * kc[d] for d in range(128)] +
                            [q_rope[h, r] * rows[t, 512 + r] for r in range(64)])
            s.append(dot * sc)
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = math.fsum(e)
        p = [x / z for x in e]
        assert abs(lse[h] - (m + math.log(z))) < 1e-12
        for d in (0, 17, 127):
            v = [math.fsum(w_uv[h, d, c] * rows[t, c] for c in range(512)) for t in range(5)]
            assert abs(o[h, d] - math.fsum(p[t] * v[t] for t in range(5))) < 1e-12
        for c in (0, 300, 511):
            assert abs(u[h, c] - math.fsum(p[t] * rows[t, c] for t in range(5))) < 1e-12


def test_lse_matches_scipy():
    from scipy.special import logsumexp
    s = np.random.default_rng(10).standard_normal((3, 40)) * 7
    _, lse = O.softmax_stats(s)
    assert np.allclose(lse, logsumexp(s, axis=-1), rtol=1e-14)


def test_softmax_shift_invariance_with_large_logits():
    s = np.random.default_rng(11).standard_normal((2, 64))
    p1, l1 = O.softmax_stats(s)
    p2, l2 = O.softmax_stats(s + 1000.0)
    assert np.allclose(p1, p2, rtol=1e-10) and np.allclose(l2 - l1, 1000.0, rtol=1e-13)


# --------------------------------------------------------------------------- paging

def _small_workload(**kw):
    from mla_latent_kv_16_gb300 import workloads as W
    base = dict(batch=3, heads=8, seq_lens=[70, 129, 5])
    base.update(kw)
    return W.preset("dsv3_bf16", **base)


def _build_pool(w, d):
    cos_t, sin_t = O.rope_tables(w.max_pos)
    pool, sc = O.new_pool(w.num_pages, w.page_size, w.cache_dtype)
    to_np = (lambda t: t.view(torch.int16).numpy().view(np.uint16)) if w.act_dtype == "bf16" \
        else (lambda t: t.numpy())
    O.append(pool, sc, to_np(d["ctx_c_kv"]), to_np(d["ctx_k_r"]), d["ctx_positions"].numpy(),
             d["ctx_slots"].numpy(), cos_t, sin_t, w.act_dtype, w.cache_dtype)
    return pool, sc


def test_slots_and_block_table_agree():
    from mla_latent_kv_16_gb300 import workloads as W
    w = _small_workload()
    d = W.make_inputs(w)
    pool, sc = _build_pool(w, d)
    off = 0
    c = d["ctx_c_kv"].view(torch.int16).numpy().view(np.uint16)
    for b, L in enumerate(w.seq_lens):
        rows = O.gather_rows(pool, sc, d["block_table"][b].numpy(), L, w.page_size, "bf16")
        assert np.array_equal(rows[:, :512], O.bf16_bits_to_f64(c[off:off + L]))
        off += L
    # unwritten tail rows stay poisoned
    assert np.isnan(O.bf16_bits_to_f64(pool[:, 0])).sum() == w.num_pages * w.page_size - w.total_tokens


def test_decode_independent_of_page_permutation():
    from mla_latent_kv_16_gb300 import workloads as W
    w1 = _small_workload(shuffle_pages=False)
    w2 = _small_workload(shuffle_pages=True)
    d1, d2 = W.make_inputs(w1), W.make_inputs(w2)
    assert not torch.equal(d1["block_table"], d2["block_table"])
    outs = []
    for w, d in ((w1, d1), (w2, d2)):
        pool, sc = _build_pool(w, d)
        q_lat = O.absorb_q(d["q_nope"].float().numpy(), d["w_uk"].float().numpy())
        outs.append(O.decode_latent(q_lat, d["q_rope"].float().numpy(), pool, sc,
                                    d["block_table"].numpy(), w.seq_lens, 1, w.page_size,
                                    "bf16", O.default_scale()))
    for b in outs[0]:
        assert np.array_equal(outs[0][b][0], outs[1][b][0])


def test_e4m3_readback_values_by_hand():
    """E4M3 rows read back as decode(byte) * scale, exactly (in fp64), each
    element scaled by its own group's factor. Expected values worked by hand:
    0x38 is 1.0 and 0x3A is 1.25 (exponent field 7, mantissa 010); 0x7E is 448;
    0xB8 is -1.0. fl32(0.1) = 13421773 * 2^-27 exactly, fl32(1/3) = 11184811 *
    2^-25; 1.25 * fl32(1/3) = 55924055 * 2^-27; 448 * 3 = 1344."""
    pool = np.full((2, O.ROW), 0x38, dtype=np.uint8)
    sc = np.ones((2, len(O.E4M3_GROUPS)), dtype=np.float32)
    sc[1] = [0.1, 1.0 / 3.0, 3.0, 2.0, 0.5]
    pool[1, 128] = 0x3A
    pool[1, 256] = 0x7E
    pool[1, 512] = 0xB8                      # -1.0 in the RoPE group
    rows = O.gather_rows(pool, sc, np.array([0]), 2, 2, "e4m3")
    assert np.all(rows[0] == 1.0)            # unit scale: the codes themselves
    assert rows[1, 0] == 13421773 * 2.0 ** -27 and rows[1, 127] == 13421773 * 2.0 ** -27
    assert rows[1, 129] == 11184811 * 2.0 ** -25
    assert rows[1, 128] == 55924055 * 2.0 ** -27   # not representable in fp32 or bf16: no rounding
    assert rows[1, 256] == 1344.0
    assert rows[1, 511] == 2.0               # last latent element: group 3
    assert rows[1, 512] == -0.5 and rows[1, 575] == 0.5   # RoPE part: group 4


def test_e4m3_append_bounds():
    from mla_latent_kv_16_gb300 import workloads as W
    w = W.preset("fp8_lq2", batch=2, heads=8, seq_lens=[77, 64])
    d = W.make_inputs(w)
    pool, sc = _build_pool(w, d)
    cos_t, sin_t = O.rope_tables(w.max_pos)
    c = O.bf16_bits_to_f32(d["ctx_c_kv"].view(torch.int16).numpy().view(np.uint16))
    k = O.rope_rotate_f32(O.bf16_bits_to_f32(d["ctx_k_r"].view(torch.int16).numpy().view(np.uint16)),
                          d["ctx_positions"].numpy().astype(np.int64), cos_t, sin_t)
    x = np.concatenate([c, k], 1).astype(np.float64)
    slots = d["ctx_slots"].numpy()
    vals = O.e4m3_decode(pool[slots])
    for gi, (a, b) in enumerate(O.E4M3_GROUPS):
        s = sc[slots, gi].astype(np.float64)
        seg = x[:, a:b]
        deq = vals[:, a:b] * s[:, None]
        # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 for normals,
        # absolute <= 2^-10 * scale in the subnormal range
        err = np.abs(deq - seg)
        bound = np.maximum(np.abs(seg) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * 1.0001
        assert np.all(err <= bound)
        # the largest element of each group encodes to +-448
        amax_idx = np.argmax(np.abs(seg), axis=1)
        codes = pool[slots, a + amax_idx]
        assert np.all((codes & 0x7F) == 0x7E)


# --------------------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible oracle mistakes and show that a pin above fails."""
    q_nope, q_rope, w_uk, w_uv, rows = _rand_case(H=3, T=9, seed=12)
    H, T = 3, 9
    eye = np.zeros((H, 128, 512))
    eye[:, :, :128] = np.eye(128)
    q = torch.from_numpy(np.concatenate([q_nope, q_rope], 1))[None, :, None, :]
    k = torch.from_numpy(np.concatenate([rows[:, :128], rows[:, 512:]], 1))[None, None].expand(1, H, T, 192)
    v = torch.from_numpy(rows[:, :128])[None, None].expand(1, H, T, 128)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=1 / math.sqrt(192))[0, :, 0].numpy()

    # 1) dropped RoPE term in the score
    o, _, _ = O.attend_nonabsorbed(q_nope, np.zeros_like(q_rope), eye, eye, rows, O.default_scale())
    assert not np.allclose(o, ref, rtol=1e-6)
    # 2) wrong scale 1/sqrt(128)
    o, _, _ = O.attend_nonabsorbed(q_nope, q_rope, eye, eye, rows, 1 / math.sqrt(128))
    assert not np.allclose(o, ref, rtol=1e-6)
    # 3) sign error in the rotation is caught by the complex-multiply pin
    cos_t, sin_t = O.rope_tables(50)
    kk = np.random.default_rng(13).standard_normal((4, 64)).astype(np.float32)
    pos = np.array([1, 5, 9, 40])
    good = O.rope_rotate_f32(kk, pos, cos_t, sin_t)
    bad = O.rope_rotate_f32(kk, pos, cos_t, -sin_t)
    assert not np.allclose(good, bad)
    # 4) a page-table off-by-one changes what gather_rows returns
    pool = np.arange(8 * 4 * 576, dtype=np.float32).reshape(32, 576)
    bt = np.array([3, 1])
    r1 = O.gather_rows(pool, None, bt, 7, 4, "f32")
    r2 = O.gather_rows(pool, None, bt + 1, 7, 4, "f32")
    assert not np.array_equal(r1, r2)
    assert np.array_equal(r1[0], pool[12]) and np.array_equal(r1[4], pool[4])
