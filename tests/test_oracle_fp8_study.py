"""Pins the conclusions of the FP8 score-path study (oracle/fp8_qk_study.py) on a
small seeded E4M3 case: a single E4M3 term for the query (or for P) misses the
rel-L2 <= 5e-3 bound on the latent output; two terms (the code and the code of
its residual) meet it, for the scores alone and with the latent sum in FP8 too.
CPU only."""
from oracle import fp8_qk_study as S

BOUND = 5e-3


def test_fp8_score_path_needs_two_query_terms():
    r = S.study(n_seq=2, seq_len=512, seed=7)
    assert r["bf16 q_lat, bf16 dequantised cache (current)"]["u_rel_l2"] <= BOUND
    assert r["E4M3 q per (head, group), E4M3 cache codes"]["u_rel_l2"] > BOUND
    assert r["E4M3 q per head (one scale), E4M3 cache codes"]["u_rel_l2"] > BOUND
    assert r["E4M3 q + E4M3 residual (two terms), E4M3 cache codes"]["u_rel_l2"] <= BOUND
    assert r["two-term q; P in E4M3 per (head, group), one term"]["u_rel_l2"] > BOUND
    assert r["two-term q; P in E4M3 per (head, group), two terms"]["u_rel_l2"] <= BOUND
