"""CPU oracle for MLA decode with matrix absorption over a paged latent cache.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this module. The product path never does, and
this module imports nothing from the product (only the seeded input generator
module, which holds no arithmetic of the method, is shared).

Plain and slow on purpose: numpy in fp64, no blocking, no fusion, one head at a
time. Each function names the passage it follows. Sources, by page title:

  [P1] "Model Architecture Driving Inference Systems: From MHA/GQA to DeepSeek
       MLA Matrix Absorption and Memory Minimalism" (dev.to)
  [P2] "Multi-Head Latent Attention (MLA): Mathematical Foundations, Low-Rank KV
       Compression, Decoupled Rotary Positional Embeddings, and Inference Matrix
       Absorption" (llms.blog)
  [P4] "DeepSeek's attention evolution - [MLA]" (blog.0xnullpath.cc)
  [P5] "Tech Radar: DeepSeek-V3 Multi-Head Latent Attention (MLA) Architecture &
       KV Cache Compression" (tanhdev.com)

Readings taken where the pages are silent (each one is also a test):
  * RoPE pairs are adjacent elements (2i, 2i+1), the complex view of [P2]
    "PyTorch Reference Implementation" (apply_rope); theta_i = base^(-2i/64),
    base 10000, angle = position * theta_i, position 0-based.
  * cos/sin are evaluated in fp64 by libm and rounded to fp32; the rotation
    is done in fp32 with every product and sum rounded separately (no FMA).
  * q_rope arrives already rotated; append rotates k_R only.
  * W_UK[h], W_UV[h] are [128 x 512] (the view(n_heads, d_head, d_c) of [P2]).
  * The score scale is 1/sqrt(d_h + d_R) = 1/sqrt(192) ([P1] §3.1, [P5] §2).
  * seq_len counts the step's q_len new tokens, appended before attending
    ([P2] forward_decode_absorbed concatenates first); query j of q_len sees
    tokens 0 .. seq_len - q_len + j.
  * E4M3 cache: one fp32 scale per token per group, groups [0,128), [128,256),
    [256,384), [384,512) of c_KV and [512,576) of k_R; scale = fl32(amax/448)
    (1.0 when amax is 0); byte = E4M3FN(fl32(x/scale)) rounded to nearest even,
    saturating to +-448; value = decode(byte) * scale.
  * lse is the natural-log log-sum-exp of the scaled scores.
  * W_O in R^{d x (H d_v)} is stored [d][H][d_v] (the view(d_model, n_heads,
    d_head) of [P2]); the fused weight W~ is [d][H][d_c].
"""
from __future__ import annotations

import math

import numpy as np

D_NOPE = 128
D_ROPE = 64
D_C = 512
D_V = 128
ROW = D_C + D_ROPE
E4M3_GROUPS = ((0, 128), (128, 256), (256, 384), (384, 512), (512, 576))
E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# Cache footprint closed forms
# ---------------------------------------------------------------------------

def kv_bytes_per_token(n_layers: int, n_kv_heads: int, d_head: int, dtype_bytes: int) -> int:
    """Per-token K+V bytes: 2 * n_layers * n_kv_heads * d_head * sizeof(dtype).
    [P1] Introduction, "KV Cache Bytes per Token" equation."""
    return 2 * n_layers * n_kv_heads * d_head * dtype_bytes


def kv_cache_bytes(batch: int, seq_len: int, n_layers: int, d_head: int, n_heads: int,
                   dtype_bytes: int) -> int:
    """Whole-cache size 2*B*L*N*d_head*n_heads*bytes. [P5] §1 "KV Cache Size"."""
    return 2 * batch * seq_len * n_layers * d_head * n_heads * dtype_bytes


def mla_bytes_per_token(dtype_bytes: float, n_layers: int = 1, d_c: int = D_C,
                        d_r: int = D_ROPE) -> float:
    """MLA caches only c_KV (d_c) and the shared k_R (d_R) per token per layer.
    [P1] §2.4 table; [P2] "What the Inference Engine Caches"."""
    return n_layers * (d_c + d_r) * dtype_bytes


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits.
    Inputs must be finite."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def e4m3_decode(b) -> np.ndarray:
    """OCP FP8 E4M3FN byte -> value (fp64): bias 7, subnormals 2^-6 * m/8,
    0x7F/0xFF are NaN, no infinities."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32)))
    out = s * mag
    return np.where((b & 0x7F) == 0x7F, np.nan, out)


def e4m3_encode(x) -> np.ndarray:
    """fp32 -> OCP FP8 E4M3FN byte, round to nearest even, saturating to
    +-448 (finite inputs). Written from the format definition: the grid step
    is 2^-9 below the smallest normal 2^-6, else 2^(floor(log2|x|)-3)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    _, ex = np.frexp(a)                     # a = f * 2^ex, f in [0.5, 1)
    e_unb = ex - 1                          # floor(log2 a) for a > 0
    step_exp = np.where(a < 2.0 ** -6, -9, e_unb - 3)
    step_exp = np.where(a == 0, -9, step_exp)
    q = np.rint(np.ldexp(a, -step_exp.astype(np.int32)))   # exact scaling, RNE
    v = np.ldexp(q, step_exp.astype(np.int32))              # rounded magnitude
    v = np.minimum(v, E4M3_MAX)                              # saturate
    # encode magnitude v (now exactly on the grid)
    _, ev = np.frexp(v)
    ev = ev - 1
    normal = v >= 2.0 ** -6
    e_field = np.where(normal, ev + 7, 0)
    m_field = np.where(normal,
                       np.rint(np.ldexp(v, (-ev).astype(np.int32)) * 8.0 - 8.0),
                       np.rint(np.ldexp(v, 9)))
    byte = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    byte = np.where(sign, byte | 0x80, byte)
    return byte.astype(np.uint8)


# ---------------------------------------------------------------------------
# Decoupled RoPE on k_R  ([P1] §2.3, [P2] "The Decoupled RoPE Solution")
# ---------------------------------------------------------------------------

_ROPE_CACHE: dict = {}


def rope_tables(max_pos: int, d_rope: int = D_ROPE, base: float = 10000.0):
    """cos/sin [max_pos, d_rope/2] fp32 of angle pos*theta_i, theta_i =
    base^(-(2i)/d_rope), each evaluated by libm in fp64 and rounded once."""
    key = (max_pos, d_rope, base)
    if key in _ROPE_CACHE:
        return _ROPE_CACHE[key]
    half = d_rope // 2
    theta = [math.pow(base, -(2.0 * i) / d_rope) for i in range(half)]
    cos = np.empty((max_pos, half), dtype=np.float64)
    sin = np.empty((max_pos, half), dtype=np.float64)
    for p in range(max_pos):
        fp = float(p)
        cos[p] = [math.cos(fp * t) for t in theta]
        sin[p] = [math.sin(fp * t) for t in theta]
    out = (cos.astype(np.float32), sin.astype(np.float32))
    _ROPE_CACHE[key] = out
    return out


def rope_rotate_f32(k: np.ndarray, positions: np.ndarray, cos_t: np.ndarray,
                    sin_t: np.ndarray) -> np.ndarray:
    """Rotate adjacent pairs (x0, x1) = (k[2i], k[2i+1]) by angle pos*theta_i in
    fp32: r0 = x0*c - x1*s, r1 = x0*s + x1*c, every operation rounded to fp32
    (numpy float32 ufuncs never fuse). k: [N, 64] float32."""
    k = np.asarray(k, dtype=np.float32)
    c = cos_t[positions]
    s = sin_t[positions]
    x0 = k[:, 0::2]
    x1 = k[:, 1::2]
    r0 = np.subtract(np.multiply(x0, c), np.multiply(x1, s))
    r1 = np.add(np.multiply(x0, s), np.multiply(x1, c))
    out = np.empty_like(k)
    out[:, 0::2] = r0
    out[:, 1::2] = r1
    return out


def rope_rotate_f64(v: np.ndarray, pos: float, base: float = 10000.0) -> np.ndarray:
    """Exact-angle fp64 rotation of one vector, for the RoPE property checks."""
    half = v.shape[-1] // 2
    out = np.empty_like(v, dtype=np.float64)
    for i in range(half):
        th = pos * math.pow(base, -(2.0 * i) / v.shape[-1])
        c, s = math.cos(th), math.sin(th)
        out[..., 2 * i] = v[..., 2 * i] * c - v[..., 2 * i + 1] * s
        out[..., 2 * i + 1] = v[..., 2 * i] * s + v[..., 2 * i + 1] * c
    return out


# ---------------------------------------------------------------------------
# Paged cache: append and read back
# ---------------------------------------------------------------------------

def new_pool(num_pages: int, page_size: int, cache_dtype: str):
    """An empty page pool, every byte poisoned (NaN values, NaN scales), so that
    reading an unwritten row shows up in the result."""
    n = num_pages * page_size
    if cache_dtype == "f32":
        return np.full((n, ROW), np.nan, dtype=np.float32), None
    if cache_dtype == "bf16":
        return np.full((n, ROW), 0x7FC0, dtype=np.uint16), None
    return (np.full((n, ROW), 0x7F, dtype=np.uint8),
            np.full((n, len(E4M3_GROUPS)), np.nan, dtype=np.float32))


def _to_f32(x, act_dtype: str) -> np.ndarray:
    """Input rows as exact fp32 (bf16 inputs arrive as uint16 bits)."""
    if act_dtype == "bf16":
        return bf16_bits_to_f32(x)
    return np.asarray(x, dtype=np.float32)


def append(pool, scales, c_kv, k_r, positions, slots, cos_t, sin_t, act_dtype: str,
           cache_dtype: str):
    """Write tokens into the paged latent cache ([P2] forward_decode_absorbed
    step 2; [P1] §2.4 row = 512 c_KV + 64 k_R; E4M3 with per-group scales per
    [P2] "High-Throughput Serving Kernels"). Row slot s holds the token; c_KV
    is stored unchanged (rounded to the cache dtype), k_R is rotated first.
    Returns (pool, scales), modified in place."""
    c = _to_f32(c_kv, act_dtype)
    k = _to_f32(k_r, act_dtype)
    kr = rope_rotate_f32(k, np.asarray(positions, dtype=np.int64), cos_t, sin_t)
    x = np.concatenate([c, kr], axis=1)                     # fp32 [N, 576]
    slots = np.asarray(slots, dtype=np.int64)
    if cache_dtype == "f32":
        pool[slots] = x
    elif cache_dtype == "bf16":
        pool[slots] = f32_to_bf16_bits(x)
    else:
        q = np.empty(x.shape, dtype=np.uint8)
        sc = np.empty((x.shape[0], len(E4M3_GROUPS)), dtype=np.float32)
        for gi, (a, b) in enumerate(E4M3_GROUPS):
            seg = x[:, a:b]
            amax = np.max(np.abs(seg), axis=1).astype(np.float32)
            s = np.where(amax == 0, np.float32(1.0),
                         np.divide(amax, np.float32(E4M3_MAX), dtype=np.float32))
            s = s.astype(np.float32)
            sc[:, gi] = s
            q[:, a:b] = e4m3_encode(np.divide(seg, s[:, None], dtype=np.float32))
        pool[slots] = q
        scales[slots] = sc
    return pool, scales


def gather_rows(pool, scales, block_table_row, n_tokens: int, page_size: int,
                cache_dtype: str) -> np.ndarray:
    """Logical rows 0..n_tokens-1 of one sequence, decoded to fp64, read through
    its block table (paged layout, [P1] §4.1 'block size 64 page allocations').
    E4M3 rows come back exactly dequantised: decode(byte) * scale of the
    element's group, in fp64 ([P2] "High-Throughput Serving Kernels": E4M3
    values with per-block scaling factors)."""
    pos = np.arange(n_tokens)
    pages = np.asarray(block_table_row, dtype=np.int64)[pos // page_size]
    slots = pages * page_size + pos % page_size
    raw = pool[slots]
    if cache_dtype == "f32":
        return raw.astype(np.float64)
    if cache_dtype == "bf16":
        return bf16_bits_to_f64(raw)
    vals = e4m3_decode(raw)
    sc = scales[slots].astype(np.float64)
    for gi, (a, b) in enumerate(E4M3_GROUPS):
        vals[:, a:b] *= sc[:, gi:gi + 1]
    return vals


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def softmax_stats(s: np.ndarray):
    """Max-subtracted softmax in fp64 over the last axis. Returns (p, lse)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    l_ = np.sum(e, axis=-1, keepdims=True)
    return e / l_, (m + np.log(l_))[..., 0]


def absorb_q(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_lat[..., h, :] = W_UK[h]^T q_nope[..., h, :]  (128 -> 512).
    [P1] §3.1 "absorbed query"; [P2] einsum('bthd,hdc->bhtc')."""
    return np.einsum("...hd,hdc->...hc", np.asarray(q_nope, np.float64),
                     np.asarray(w_uk, np.float64))


def out_proj(u: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """o[..., h, :] = W_UV[h] u[..., h, :]  (512 -> 128). [P1] §3.2."""
    return np.einsum("...hc,hdc->...hd", np.asarray(u, np.float64),
                     np.asarray(w_uv, np.float64))


def attend_absorbed(q_lat: np.ndarray, q_rope: np.ndarray, rows: np.ndarray, scale: float):
    """One query position, all heads, absorbed form over visible rows:
    s_t = (q_lat . c_t + q_rope . k_R,t) * scale; u = sum_t p_t c_t.
    [P1] §3.1 final score; §3.2 latent sum. q_lat [H,512], q_rope [H,64],
    rows [T,576] fp64. Returns u [H,512], lse [H]."""
    C = rows[:, :D_C]
    KR = rows[:, D_C:]
    s = (np.asarray(q_lat, np.float64) @ C.T + np.asarray(q_rope, np.float64) @ KR.T) * scale
    p, lse = softmax_stats(s)
    return p @ C, lse


def attend_nonabsorbed(q_nope, q_rope, w_uk, w_uv, rows: np.ndarray, scale: float):
    """One query position, the MHA form with K and V materialised per head:
    K_h[t] = [W_UK[h] c_t ; k_R,t] (192), V_h[t] = W_UV[h] c_t (128),
    s = q_h . K_h / sqrt(192), o = sum p V. ([P1] §2.3 k = [k^C ; k^R],
    §3.1 score; §3.2 o = sum_j P W_UV c_j; [P4] §2.5 MHA form.)
    Returns o [H,128], u [H,512] (= sum p c, for intermediate checks), lse [H]."""
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    C = rows[:, :D_C]
    KR = rows[:, D_C:]
    H = q_nope.shape[0]
    o = np.empty((H, D_V))
    u = np.empty((H, D_C))
    lse = np.empty(H)
    for h in range(H):
        K = np.concatenate([C @ w_uk[h].T, KR], axis=1)
        V = C @ w_uv[h].T
        q = np.concatenate([q_nope[h], q_rope[h]])
        s = (K @ q) * scale
        p, l_ = softmax_stats(s)
        o[h] = p @ V
        u[h] = p @ C
        lse[h] = l_
    return o, u, lse


def round_bf16(x) -> np.ndarray:
    """fp64 values rounded as a GPU stores an fp32 result in bf16: to fp32
    (nearest) and then to bf16 (nearest-even); returned as fp64."""
    return bf16_bits_to_f64(f32_to_bf16_bits(np.asarray(x, np.float64).astype(np.float32)))


def default_scale(d_nope: int = D_NOPE, d_rope: int = D_ROPE) -> float:
    """1/sqrt(d_h + d_R). [P1] §3.1; [P2] self.scale; [P5] §2."""
    return 1.0 / math.sqrt(d_nope + d_rope)


def visible_tokens(seq_len: int, q_len: int, j: int) -> int:
    """Number of rows query j (0-based) of a q_len-token step attends to."""
    return seq_len - q_len + j + 1


def decode_latent(q_lat, q_rope, pool, scales, block_table, seq_lens, q_len: int,
                  page_size: int, cache_dtype: str, scale: float, batch_index=None):
    """The decode step from the absorbed query to the latent output u and lse,
    for the listed sequences (all by default). q_lat [B,Lq,H,512], q_rope
    [B,Lq,H,64]. Returns dict b -> (u [Lq,H,512], lse [Lq,H])."""
    out = {}
    B = len(seq_lens)
    for b in (range(B) if batch_index is None else batch_index):
        L = int(seq_lens[b])
        rows = gather_rows(pool, scales, block_table[b], L, page_size, cache_dtype)
        us, ls = [], []
        for j in range(q_len):
            T = visible_tokens(L, q_len, j)
            u, lse = attend_absorbed(q_lat[b, j], q_rope[b, j], rows[:T], scale)
            us.append(u)
            ls.append(lse)
        out[b] = (np.stack(us), np.stack(ls))
    return out


def decode_full(q_nope, q_rope, w_uk, w_uv, pool, scales, block_table, seq_lens,
                q_len: int, page_size: int, cache_dtype: str, scale: float,
                batch_index=None, heads=None):
    """The whole decode output o in the non-absorbed form, for the listed
    sequences and heads. Returns dict b -> (o [Lq,h,128], u [Lq,h,512], lse [Lq,h])."""
    out = {}
    B = len(seq_lens)
    H = q_nope.shape[2]
    hs = list(range(H)) if heads is None else list(heads)
    w_uk_s = np.asarray(w_uk)[hs]
    w_uv_s = np.asarray(w_uv)[hs]
    for b in (range(B) if batch_index is None else batch_index):
        L = int(seq_lens[b])
        rows = gather_rows(pool, scales, block_table[b], L, page_size, cache_dtype)
        os_, us, ls = [], [], []
        for j in range(q_len):
            T = visible_tokens(L, q_len, j)
            o, u, lse = attend_nonabsorbed(np.asarray(q_nope)[b, j][hs], np.asarray(q_rope)[b, j][hs],
                                           w_uk_s, w_uv_s, rows[:T], scale)
            os_.append(o)
            us.append(u)
            ls.append(lse)
        out[b] = (np.stack(os_), np.stack(us), np.stack(ls))
    return out


# ---------------------------------------------------------------------------
# Output projection with W_UV folded in (the weights are fused at load time)
# ---------------------------------------------------------------------------

def fuse_out_weights(w_o: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """Pre-fused output weight, per head the d x d_v column block of W_O times
    W_UV[h] (d_v x d_c): W~[m, h, c] = sum_e W_O[m, h, e] W_UV[h, e, c].
    [P1] §3.2 (W~^O_i = W^O_i W^UV_i in R^{d x d_c}, fused before decoding);
    [P2] "Value Output Matrix Absorption" (W_O^i W_UV,i is static and computed
    once). w_o [d, H, d_v] is W_O in R^{d x (H d_v)} viewed per head."""
    w_o = np.asarray(w_o, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    out = np.empty((w_o.shape[0], w_uv.shape[0], w_uv.shape[2]))
    for h in range(w_uv.shape[0]):
        out[:, h, :] = w_o[:, h, :] @ w_uv[h]
    return out


def out_proj_fused(u: np.ndarray, w_fused: np.ndarray) -> np.ndarray:
    """y[..., m] = sum_h sum_c W~[m, h, c] u[..., h, c]: the attention block's
    output in the model dimension straight from the latent outputs u, as one
    product with the heads' latent vectors concatenated.
    [P1] §3.2 (the 512-dimensional latent sum times the pre-fused matrix);
    [P2] "Value Output Matrix Absorption" (final projection from latent space)."""
    u = np.asarray(u, np.float64)
    w = np.asarray(w_fused, np.float64)
    return u.reshape(*u.shape[:-2], -1) @ w.reshape(w.shape[0], -1).T


def out_proj_model(o: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """y[..., m] = sum_h sum_e W_O[m, h, e] o[..., h, e]: the unfused output
    projection, W_O times the concatenated head outputs o [..., H, d_v].
    [P2] "Value Output Matrix Absorption" (W_O = [W_O^1, ..., W_O^nh] in
    R^{d x (nh d_v)})."""
    o = np.asarray(o, np.float64)
    w = np.asarray(w_o, np.float64)
    return o.reshape(*o.shape[:-2], -1) @ w.reshape(w.shape[0], -1).T


# ---------------------------------------------------------------------------
# Decode-layer front end: hidden state -> q_nope, q_rope, c_KV, k_R
# ---------------------------------------------------------------------------

def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis. [P2] "PyTorch
    Reference Implementation" (q_norm and kv_norm are RMS norms over d_c_q and
    d_c_kv)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gamma, np.float64)


def decode_front(h, w_dq, g_q, w_uq, w_qr, w_dkv, g_kv, w_kr, positions, eps: float,
                 base: float = 10000.0):
    """The step's projections from the hidden states h [n, d] of its new tokens,
    [P2] "PyTorch Reference Implementation" (forward_decode_absorbed, steps 1
    and 2; [P1] §2.1 c^KV = W^DKV h, §2.3 decoupled RoPE keys and queries):
      c_q    = RMSNorm(W_DQ h)                 (d_c_q)
      q_nope = W_UQ c_q, per head 128          ([n, H, 128])
      q_rope = RoPE_pos(W_QR c_q), per head 64 ([n, H, 64], rotated)
      c_kv   = RMSNorm(W_DKV h)                ([n, 512])
      k_r    = W_KR h                          ([n, 64], before its rotation, which append applies)
    Weights are nn.Linear layouts [out, in]: w_dq [d_c_q, d], w_uq [H*128, d_c_q],
    w_qr [H*64, d_c_q], w_dkv [512, d], w_kr [64, d]. Exact fp64 throughout."""
    h = np.asarray(h, np.float64)
    n = h.shape[0]
    c_q = rms_norm(h @ np.asarray(w_dq, np.float64).T, g_q, eps)
    q_nope = (c_q @ np.asarray(w_uq, np.float64).T).reshape(n, -1, D_NOPE)
    q_r = (c_q @ np.asarray(w_qr, np.float64).T).reshape(n, -1, D_ROPE)
    q_rope = np.stack([rope_rotate_f64(q_r[t], float(positions[t]), base) for t in range(n)]) if n else q_r
    c_kv = rms_norm(h @ np.asarray(w_dkv, np.float64).T, g_kv, eps)
    k_r = h @ np.asarray(w_kr, np.float64).T
    return q_nope, q_rope, c_kv, k_r


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y[..., o] = sum_i w[o, i] x[..., i]: a bias-free nn.Linear with weight
    w [out, in] ([P2] "PyTorch Reference Implementation" declares every
    projection so)."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


# ---------------------------------------------------------------------------
# Prefill in the MHA form: per-head K and V expanded from the latent rows
# ---------------------------------------------------------------------------

def expand_kv(rows: np.ndarray, w_uk: np.ndarray, w_uv: np.ndarray):
    """Per-head keys and values of cached rows [T, 576] (c_KV, rotated k_R):
    K[t, h] = [W_UK[h] c_t ; k_R,t] (192) and V[t, h] = W_UV[h] c_t (128).
    [P4] §2.5 (the MHA form expands the shared latent into per-head K/V);
    [P1] §2.3 (k = [k^C ; k^R], the RoPE key shared by all heads)."""
    rows = np.asarray(rows, np.float64)
    C, KR = rows[:, :D_C], rows[:, D_C:]
    kc = np.einsum("tc,hec->the", C, np.asarray(w_uk, np.float64))
    v = np.einsum("tc,hec->the", C, np.asarray(w_uv, np.float64))
    k = np.concatenate([kc, np.broadcast_to(KR[:, None, :], (rows.shape[0], kc.shape[1], D_ROPE))], axis=-1)
    return k, v


def prefill_mha(q_nope: np.ndarray, q_rope: np.ndarray, rows: np.ndarray, w_uk: np.ndarray,
                w_uv: np.ndarray, scale: float):
    """Causal attention of the last Tq tokens of a sequence over all its rows,
    in the MHA form: K and V expanded once, S = Q K^T * scale per head with
    query j (of Tq) seeing rows 0 .. T - Tq + j, softmax, O = P V.
    [P1] Q2 (prefill runs uncompressed, absorption is for decode); [P4] §2.5.
    q_nope [Tq, H, 128], q_rope [Tq, H, 64] (rotated), rows [T, 576].
    Returns o [Tq, H, 128] and lse [Tq, H]."""
    k, v = expand_kv(rows, w_uk, w_uv)
    q = np.concatenate([np.asarray(q_nope, np.float64), np.asarray(q_rope, np.float64)], axis=-1)
    Tq, T = q.shape[0], rows.shape[0]
    s = np.einsum("jhd,thd->hjt", q, k) * scale
    visible = np.arange(T)[None, :] <= (T - Tq + np.arange(Tq))[:, None]
    s = np.where(visible[None], s, -np.inf)
    p, lse = softmax_stats(s)
    return np.einsum("hjt,the->jhe", p, v), lse.T
