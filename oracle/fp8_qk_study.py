"""Accuracy study for an FP8 (E4M3) score path on an E4M3 cache. TEST
INFRASTRUCTURE, like the rest of this package: it runs the oracle only.

An E4M3 cache stores codes with one fp32 scale per token and group ("Multi-Head
Latent Attention (MLA)" page, "High-Throughput Serving Kernels": FP8 E4M3 with
per-block scaling factors). A tensor-core score path that multiplies codes
directly would compute, per head h and token t,

    s = scale * sum_g  sq[h, g] * sk[t, g] * (qcode_g[h] . kcode_g[t])

with q_lat and q_rope quantised to E4M3 too (scales sq per head and group).
This script measures what that does to the decode output against the exact
fp64 result (the cache read back as code x scale, no rounding), next to the
current path (code x scale rounded to bf16, q_lat in bf16), on seeded inputs
of the E4M3 workload's recipe; also with the query as two E4M3 terms (the code
and the code of its residual), which doubles the FP8 score MMAs. In those rows
the latent sum u = P V uses the exact read-back, so only the score path
differs. The last rows take the latent sum to FP8 as well: each token's group
scale folded into P (P_g[h, t] = p[h, t] * sk[t, g]), P_g quantised to E4M3
per head (one or two terms), times the codes.

    python -m oracle.fp8_qk_study [n_seq] [seq_len]
"""
from __future__ import annotations

import sys

import numpy as np

from . import mla_oracle as O
from .harness import f64, oracle_pool


def quantise_e4m3(x: np.ndarray, groups) -> tuple:
    """Per-row E4M3 codes and scales of x [..., width] for the column groups
    given, by the cache's own rule (scale = fl32(amax / 448), 1 if amax = 0)."""
    x = np.asarray(x, np.float64)
    codes = np.zeros(x.shape, np.uint8)
    scales = np.ones(x.shape[:-1] + (len(groups),), np.float32)
    for gi, (a, b) in enumerate(groups):
        seg = x[..., a:b].astype(np.float32)
        amax = np.max(np.abs(seg), axis=-1)
        sc = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
        scales[..., gi] = sc
        codes[..., a:b] = O.e4m3_encode((seg / sc[..., None]).astype(np.float32))
    return codes, scales


def dequantise(codes, scales, groups) -> np.ndarray:
    out = np.zeros(codes.shape, np.float64)
    for gi, (a, b) in enumerate(groups):
        out[..., a:b] = O.e4m3_decode(codes[..., a:b]) * scales[..., gi:gi + 1].astype(np.float64)
    return out


def study(n_seq: int = 3, seq_len: int = 2048, seed: int = 4):
    from mla_latent_kv_16_gb300 import workloads as W

    w = W.preset("fp8_lq2", batch=n_seq, seq_lens=[seq_len] * n_seq, seed=seed)
    d = W.make_inputs(w)
    pool, sc = oracle_pool(w, d)
    q_lat = O.absorb_q(f64(d["q_nope"]), f64(d["w_uk"]))  # exact
    q_rope = f64(d["q_rope"])
    scale = O.default_scale()
    groups = O.E4M3_GROUPS
    errs = {"bf16 q_lat, bf16 dequantised cache (current)": [], "E4M3 q per (head, group), E4M3 cache codes": [],
            "E4M3 q per head (one scale), E4M3 cache codes": [],
            "E4M3 q + E4M3 residual (two terms), E4M3 cache codes": [],
            "two-term q; P in E4M3 per (head, group), one term": [],
            "two-term q; P in E4M3 per (head, group), two terms": []}
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        # exact read-back (code x scale in fp64): the definition, and what an FP8
        # score path multiplies; the current kernel rounds it to bf16 first
        rows_exact = O.gather_rows(pool, sc, d["block_table"].numpy()[b], L, w.page_size, "e4m3")
        rows_bf16 = O.round_bf16(rows_exact)
        slots = [int(d["block_table"][b, t // w.page_size]) * w.page_size + t % w.page_size for t in range(L)]
        codes_k = pool.reshape(-1, 576)[slots]
        sc_k = sc.reshape(-1, 5)[slots]
        rows_exact_codes = dequantise(codes_k, sc_k, groups)
        for j in range(w.q_len):
            T = O.visible_tokens(L, w.q_len, j)
            u_ref, lse_ref = O.attend_absorbed(q_lat[b, j], q_rope[b, j], rows_exact[:T], scale)
            qfull = np.concatenate([q_lat[b, j], q_rope[b, j]], axis=-1)  # [H, 576]

            def run(q_eff, k_rows, pv=None):
                s = (q_eff @ k_rows[:T].T) * scale
                p, lse = O.softmax_stats(s)
                return (p @ k_rows[:T, :512] if pv is None else pv(p)), lse

            def pv_fp8(p, terms):
                # u[:, g] = sum_t (p[:, t] sk[t, g]) code[t, g]: P_g quantised per head
                u = np.zeros((p.shape[0], 512))
                kc = O.e4m3_decode(codes_k[:T, :512]).astype(np.float64)
                for gi, (a, bb) in enumerate(groups[:4]):
                    pg = p * sc_k[:T, gi].astype(np.float64)[None, :]
                    approx = np.zeros_like(pg)
                    for _ in range(terms):
                        c_, s_ = quantise_e4m3(pg - approx, ((0, T),))
                        approx = approx + dequantise(c_, s_, ((0, T),))
                    u[:, a:bb] = approx @ kc[:, a:bb]
                return u

            # current: q_lat rounded to bf16 (q_rope is given in bf16), bf16-rounded dequantised rows
            q_cur = np.concatenate([O.round_bf16(q_lat[b, j]), q_rope[b, j]], axis=-1)
            errs["bf16 q_lat, bf16 dequantised cache (current)"].append((run(q_cur, rows_bf16), (u_ref, lse_ref)))
            qc, qs = quantise_e4m3(qfull, groups)
            q8 = dequantise(qc, qs, groups)
            errs["E4M3 q per (head, group), E4M3 cache codes"].append((run(q8, rows_exact_codes), (u_ref, lse_ref)))
            rc, rs = quantise_e4m3(qfull - q8, groups)  # the residual, quantised the same way
            errs["E4M3 q + E4M3 residual (two terms), E4M3 cache codes"].append(
                (run(q8 + dequantise(rc, rs, groups), rows_exact_codes), (u_ref, lse_ref)))
            q2 = q8 + dequantise(rc, rs, groups)
            errs["two-term q; P in E4M3 per (head, group), one term"].append(
                (run(q2, rows_exact_codes, lambda p: pv_fp8(p, 1)), (u_ref, lse_ref)))
            errs["two-term q; P in E4M3 per (head, group), two terms"].append(
                (run(q2, rows_exact_codes, lambda p: pv_fp8(p, 2)), (u_ref, lse_ref)))
            qc1, qs1 = quantise_e4m3(qfull, ((0, 576),))
            q81 = dequantise(qc1, qs1, ((0, 576),))
            errs["E4M3 q per head (one scale), E4M3 cache codes"].append((run(q81, rows_exact_codes),
                                                                          (u_ref, lse_ref)))
    out = {}
    for name, pairs in errs.items():
        u = np.stack([g[0] for g, _ in pairs])
        ur = np.stack([r[0] for _, r in pairs])
        l = np.stack([g[1] for g, _ in pairs])
        lr = np.stack([r[1] for _, r in pairs])
        out[name] = dict(u_rel_l2=float(np.linalg.norm(u - ur) / np.linalg.norm(ur)),
                         u_max_abs=float(np.max(np.abs(u - ur))),
                         lse_max_rel=float(np.max(np.abs(l - lr) / np.abs(lr))))
    return out


if __name__ == "__main__":
    n = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    L = int(sys.argv[2]) if len(sys.argv) > 2 else 2048
    for name, r in study(n, L).items():
        print(f"{name:55s} u rel-L2 {r['u_rel_l2']:.2e}  u max-abs {r['u_max_abs']:.2e}  "
              f"lse max rel {r['lse_max_rel']:.2e}")
