"""Thin Python binding of the C ABI in include/mla.h.

Argument marshalling only: every step of the decode path runs in the library's
CUDA kernels. Functions carry the ABI's names and take torch CUDA tensors
(PyTorch provides device memory and streams). Output tensors are allocated with
torch when the caller does not pass them. If the shared library is missing, the
import of the library fails loudly; there is no other implementation to fall
back to.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import build as _build

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_WORKSPACE_TOO_SMALL, \
    MLA_ERR_DEVICE_FLAG = range(6)
MLA_F32, MLA_BF16, MLA_E4M3 = 0, 1, 2
DTYPE_CODE = {"f32": MLA_F32, "bf16": MLA_BF16, "e4m3": MLA_E4M3}
MLA_DEVERR_BAD_PAGE, MLA_DEVERR_BAD_SEQLEN, MLA_DEVERR_BAD_SLOT, MLA_DEVERR_BAD_POSITION = 1, 2, 4, 8
MLA_DEVERR_TIMEOUT = 16
MLA_STATIC_SCRATCH_BYTES = 32 << 20  # size of the library's fixed split-KV scratch array
MLA_DECODE_PATH_TENSOR_CORE, MLA_DECODE_PATH_CUDA_CORE = 1, 2

EXPORTED = ("mla_status_string", "mla_version", "mla_rope_table", "mla_cache_append", "mla_absorb_q",
            "mla_decode_num_splits", "mla_decode_workspace_size", "mla_decode_paged", "mla_out_proj",
            "mla_read_device_error", "mla_decode_paged_static_scratch", "mla_fuse_out_weights",
            "mla_out_proj_fused_workspace_size", "mla_out_proj_fused", "mla_linear_workspace_size", "mla_linear",
            "mla_decode_front_workspace_size", "mla_decode_front", "mla_decode_kernel_path",
            "mla_prefill_workspace_size", "mla_prefill_mha", "mla_decode_out_proj")


class MlaDims(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("d_nope", ctypes.c_int32), ("d_c", ctypes.c_int32),
                ("d_rope", ctypes.c_int32), ("d_v", ctypes.c_int32)]


def dims(num_heads: int) -> MlaDims:
    return MlaDims(num_heads, 128, 512, 64, 128)


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)}")
        self.status = status


_LIB = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load (once) and return the ctypes handle of libmla_gb300.so."""
    global _LIB
    if _LIB is not None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libmla_gb300.so is not built ({p}); run mla_latent_kv_16_gb300.build.build()")
    L = ctypes.CDLL(p)
    vp, i32, i64, sz, f32, f64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                                  ctypes.c_float, ctypes.c_double)
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_status_string.argtypes = [ctypes.c_int]
    L.mla_version.restype = i32
    L.mla_rope_table.restype = ctypes.c_int
    L.mla_rope_table.argtypes = [i32, i32, f64, vp, vp]
    L.mla_cache_append.restype = ctypes.c_int
    L.mla_cache_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i64, i32, ctypes.c_int,
                                   ctypes.c_int, vp, vp]
    L.mla_absorb_q.restype = ctypes.c_int
    L.mla_absorb_q.argtypes = [vp, vp, vp, i32, MlaDims, ctypes.c_int, vp]
    L.mla_out_proj.restype = ctypes.c_int
    L.mla_out_proj.argtypes = [vp, vp, vp, i32, MlaDims, ctypes.c_int, vp]
    L.mla_decode_num_splits.restype = i32
    L.mla_decode_num_splits.argtypes = [i32, i32, i32, i32, i32, MlaDims, ctypes.c_int]
    L.mla_decode_workspace_size.restype = sz
    L.mla_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, MlaDims, ctypes.c_int]
    L.mla_decode_paged.restype = ctypes.c_int
    L.mla_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, f32, i32, vp, sz, vp, vp,
                                   vp, MlaDims, ctypes.c_int, ctypes.c_int, vp]
    L.mla_decode_out_proj.restype = ctypes.c_int
    L.mla_decode_out_proj.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, f32, i32, vp, sz, vp, vp,
                                      vp, vp, vp, MlaDims, ctypes.c_int, ctypes.c_int, vp]
    L.mla_decode_paged_static_scratch.restype = ctypes.c_int
    L.mla_decode_paged_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, f32, i32, vp,
                                                  vp, vp, MlaDims, ctypes.c_int, ctypes.c_int, vp]
    L.mla_fuse_out_weights.restype = ctypes.c_int
    L.mla_fuse_out_weights.argtypes = [vp, vp, vp, i32, MlaDims, ctypes.c_int, vp]
    L.mla_out_proj_fused_workspace_size.restype = sz
    L.mla_out_proj_fused_workspace_size.argtypes = [i32, i32, MlaDims, ctypes.c_int]
    L.mla_out_proj_fused.restype = ctypes.c_int
    L.mla_out_proj_fused.argtypes = [vp, vp, vp, i32, i32, vp, sz, MlaDims, ctypes.c_int, vp]
    L.mla_linear_workspace_size.restype = sz
    L.mla_linear_workspace_size.argtypes = [i32, i32, i32, ctypes.c_int]
    L.mla_linear.restype = ctypes.c_int
    L.mla_linear.argtypes = [vp, vp, vp, i32, i32, i32, vp, sz, ctypes.c_int, vp]
    L.mla_decode_front_workspace_size.restype = sz
    L.mla_decode_front_workspace_size.argtypes = [i32, i32, i32, MlaDims, ctypes.c_int]
    L.mla_decode_front.restype = ctypes.c_int
    L.mla_decode_front.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, f32, i32, i32, i32, vp, vp, vp, vp, vp, sz,
                                   vp, MlaDims, ctypes.c_int, vp]
    L.mla_read_device_error.restype = ctypes.c_int
    L.mla_decode_kernel_path.restype = ctypes.c_int
    L.mla_prefill_workspace_size.restype = sz
    L.mla_prefill_workspace_size.argtypes = [i32, MlaDims]
    L.mla_prefill_mha.restype = ctypes.c_int
    L.mla_prefill_mha.argtypes = [vp, vp, vp, vp, vp, i32, i32, f32, vp, sz, vp, vp, vp, MlaDims, ctypes.c_int, vp]
    L.mla_decode_kernel_path.argtypes = [vp, vp, i64, i32, MlaDims, ctypes.c_int, ctypes.c_int, vp]
    L.mla_read_device_error.argtypes = [vp, vp, vp]
    _LIB = L
    return L


def status_string(status: int) -> str:
    return load().mla_status_string(status).decode()


def _check(fn: str, status: int):
    if status != MLA_OK:
        raise MlaError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _act_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MLA_F32
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def _contig_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# --------------------------------------------------------------------------- host helpers

def mla_rope_table(max_pos: int, d_rope: int = 64, base: float = 10000.0):
    """(cos, sin) host fp32 tensors [max_pos, d_rope/2] computed by the library."""
    cos = torch.empty(max_pos, d_rope // 2, dtype=torch.float32)
    sin = torch.empty_like(cos)
    _check("mla_rope_table", load().mla_rope_table(max_pos, d_rope, base, _ptr(cos), _ptr(sin)))
    return cos, sin


def mla_decode_num_splits(batch, q_len, max_pages_per_seq, page_size, num_splits, num_heads, cache_dtype):
    return load().mla_decode_num_splits(batch, q_len, max_pages_per_seq, page_size, num_splits, dims(num_heads),
                                        DTYPE_CODE[cache_dtype])


def mla_decode_workspace_size(batch, q_len, max_pages_per_seq, page_size, num_splits, num_heads, cache_dtype):
    return load().mla_decode_workspace_size(batch, q_len, max_pages_per_seq, page_size, num_splits,
                                            dims(num_heads), DTYPE_CODE[cache_dtype])


# --------------------------------------------------------------------------- device calls

def mla_cache_append(c_kv, k_r, positions, slot_mapping, rope_cos, rope_sin, cache, scales, page_size,
                     cache_dtype: str, dev_error=None, stream=None):
    _contig_cuda(c_kv, k_r, positions, slot_mapping, rope_cos, rope_sin, cache, scales, dev_error)
    n = c_kv.shape[0]
    rows = cache.shape[0] * cache.shape[1] if cache.dim() == 3 else cache.shape[0]
    num_pages = rows // page_size
    st = load().mla_cache_append(_ptr(c_kv), _ptr(k_r), _ptr(positions), _ptr(slot_mapping), _ptr(rope_cos),
                                 _ptr(rope_sin), n, rope_cos.shape[0], _ptr(cache), _ptr(scales), num_pages,
                                 page_size, _act_code(c_kv), DTYPE_CODE[cache_dtype], _ptr(dev_error),
                                 _stream(stream))
    _check("mla_cache_append", st)


def mla_absorb_q(q_nope, w_uk, q_lat=None, stream=None):
    """q_nope [..., H, 128], w_uk [H, 128, 512] -> q_lat [..., H, 512]."""
    _contig_cuda(q_nope, w_uk, q_lat)
    H = w_uk.shape[0]
    n = q_nope.numel() // (H * 128)
    if q_lat is None:
        q_lat = torch.empty(*q_nope.shape[:-1], 512, dtype=q_nope.dtype, device=q_nope.device)
    _check("mla_absorb_q", load().mla_absorb_q(_ptr(q_nope), _ptr(w_uk), _ptr(q_lat), n, dims(H),
                                                _act_code(q_nope), _stream(stream)))
    return q_lat


def mla_out_proj(u, w_uv, o=None, stream=None):
    """u [..., H, 512], w_uv [H, 128, 512] -> o [..., H, 128]."""
    _contig_cuda(u, w_uv, o)
    H = w_uv.shape[0]
    n = u.numel() // (H * 512)
    if o is None:
        o = torch.empty(*u.shape[:-1], 128, dtype=u.dtype, device=u.device)
    _check("mla_out_proj", load().mla_out_proj(_ptr(u), _ptr(w_uv), _ptr(o), n, dims(H), _act_code(u),
                                                _stream(stream)))
    return o


def mla_fuse_out_weights(w_o, w_uv, w_fused=None, stream=None):
    """w_o [d_model, H, 128], w_uv [H, 128, 512] -> W~ [d_model, H, 512] (load time)."""
    _contig_cuda(w_o, w_uv, w_fused)
    d_model, H = w_o.shape[0], w_uv.shape[0]
    if w_fused is None:
        w_fused = torch.empty(d_model, H, 512, dtype=w_o.dtype, device=w_o.device)
    _check("mla_fuse_out_weights", load().mla_fuse_out_weights(_ptr(w_o), _ptr(w_uv), _ptr(w_fused), d_model,
                                                                dims(H), _act_code(w_o), _stream(stream)))
    return w_fused


def mla_out_proj_fused_workspace_size(n_tokens: int, d_model: int, num_heads: int, act: str = "bf16") -> int:
    return load().mla_out_proj_fused_workspace_size(n_tokens, d_model, dims(num_heads), DTYPE_CODE[act])


def mla_out_proj_fused(u, w_fused, y=None, workspace=None, stream=None):
    """u [..., H, 512], W~ [d_model, H, 512] -> y [..., d_model]."""
    _contig_cuda(u, w_fused, y, workspace)
    d_model, H = w_fused.shape[0], w_fused.shape[1]
    n = u.numel() // (H * 512)
    if y is None:
        y = torch.empty(*u.shape[:-2], d_model, dtype=u.dtype, device=u.device)
    act = "f32" if u.dtype == torch.float32 else "bf16"
    need = mla_out_proj_fused_workspace_size(n, d_model, H, act) if n > 0 else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=u.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_out_proj_fused", load().mla_out_proj_fused(_ptr(u), _ptr(w_fused), _ptr(y), n, d_model,
                                                            _ptr(workspace), ws_bytes, dims(H), _act_code(u),
                                                            _stream(stream)))
    return y


def mla_linear_workspace_size(n_tokens: int, n_out: int, n_in: int, act: str = "bf16") -> int:
    return load().mla_linear_workspace_size(n_tokens, n_out, n_in, DTYPE_CODE[act])


def mla_linear(x, w, y=None, workspace=None, stream=None):
    """x [..., n_in], w [n_out, n_in] -> y [..., n_out] = x w^T."""
    _contig_cuda(x, w, y, workspace)
    n_out, n_in = w.shape
    n = x.numel() // n_in
    if y is None:
        y = torch.empty(*x.shape[:-1], n_out, dtype=x.dtype, device=x.device)
    act = "f32" if x.dtype == torch.float32 else "bf16"
    need = mla_linear_workspace_size(n, n_out, n_in, act) if n > 0 else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_linear", load().mla_linear(_ptr(x), _ptr(w), _ptr(y), n, n_out, n_in, _ptr(workspace), ws_bytes,
                                            _act_code(x), _stream(stream)))
    return y


def mla_decode_front_workspace_size(n_tokens: int, d_model: int, d_cq: int, num_heads: int, act: str = "bf16") -> int:
    return load().mla_decode_front_workspace_size(n_tokens, d_model, d_cq, dims(num_heads), DTYPE_CODE[act])


def mla_decode_front(h, w_dqkv, g_q, g_kv, w_uqr, positions, rope_cos, rope_sin, eps: float, num_heads: int,
                     q_nope=None, q_rope=None, c_kv=None, k_r=None, workspace=None, dev_error=None, stream=None):
    """h [n, d_model] -> (q_nope [n, H, 128], q_rope [n, H, 64] rotated, c_kv [n, 512], k_r [n, 64])."""
    _contig_cuda(h, w_dqkv, g_q, g_kv, w_uqr, positions, rope_cos, rope_sin, q_nope, q_rope, c_kv, k_r, workspace,
                 dev_error)
    n, d_model = h.shape
    d_cq = g_q.shape[0]
    H = num_heads
    mk = lambda *shape: torch.empty(*shape, dtype=h.dtype, device=h.device)
    q_nope = mk(n, H, 128) if q_nope is None else q_nope
    q_rope = mk(n, H, 64) if q_rope is None else q_rope
    c_kv = mk(n, 512) if c_kv is None else c_kv
    k_r = mk(n, 64) if k_r is None else k_r
    act = "f32" if h.dtype == torch.float32 else "bf16"
    need = mla_decode_front_workspace_size(n, d_model, d_cq, H, act) if n > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=h.device)
    st = load().mla_decode_front(_ptr(h), _ptr(w_dqkv), _ptr(g_q), _ptr(g_kv), _ptr(w_uqr), _ptr(positions),
                                 _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0], eps, n, d_model, d_cq,
                                 _ptr(q_nope), _ptr(q_rope), _ptr(c_kv), _ptr(k_r), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(dev_error), dims(H),
                                 _act_code(h), _stream(stream))
    _check("mla_decode_front", st)
    return q_nope, q_rope, c_kv, k_r


def mla_decode_paged(q_lat, q_rope, cache, scales, block_table, seq_lens, page_size: int, cache_dtype: str,
                     softmax_scale: Optional[float] = None, num_splits: int = 0, workspace=None, u_out=None,
                     lse_out=None, dev_error=None, stream=None, want_lse: bool = True):
    """q_lat [B, Lq, H, 512], q_rope [B, Lq, H, 64] -> (u [B, Lq, H, 512], lse [B, Lq, H] or None)."""
    _contig_cuda(q_lat, q_rope, cache, scales, block_table, seq_lens, workspace, u_out, lse_out, dev_error)
    B, Lq, H = q_lat.shape[0], q_lat.shape[1], q_lat.shape[2]
    maxp = block_table.shape[1]
    rows = cache.shape[0] * cache.shape[1] if cache.dim() == 3 else cache.shape[0]
    num_pages = rows // page_size
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(128 + 64)
    if u_out is None:
        u_out = torch.empty(B, Lq, H, 512, dtype=q_lat.dtype, device=q_lat.device)
    if lse_out is None and want_lse:
        lse_out = torch.empty(B, Lq, H, dtype=torch.float32, device=q_lat.device)
    need = mla_decode_workspace_size(B, Lq, maxp, page_size, num_splits, H, cache_dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_lat.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().mla_decode_paged(_ptr(q_lat), _ptr(q_rope), _ptr(cache), _ptr(scales), _ptr(block_table),
                                 _ptr(seq_lens), B, Lq, maxp, num_pages, page_size, softmax_scale, num_splits,
                                 _ptr(workspace), ws_bytes, _ptr(u_out), _ptr(lse_out), _ptr(dev_error), dims(H),
                                 _act_code(q_lat), DTYPE_CODE[cache_dtype], _stream(stream))
    _check("mla_decode_paged", st)
    return u_out, lse_out


def mla_decode_out_proj(q_lat, q_rope, cache, scales, block_table, seq_lens, page_size: int, cache_dtype: str,
                        w_uv, softmax_scale: Optional[float] = None, num_splits: int = 0, workspace=None,
                        u_out=None, lse_out=None, o_out=None, dev_error=None, stream=None):
    """mla_decode_paged then mla_out_proj as one call -> (u [B, Lq, H, 512], lse [B, Lq, H], o [B, Lq, H, 128])."""
    _contig_cuda(q_lat, q_rope, cache, scales, block_table, seq_lens, w_uv, workspace, u_out, lse_out, o_out,
                 dev_error)
    B, Lq, H = q_lat.shape[0], q_lat.shape[1], q_lat.shape[2]
    maxp = block_table.shape[1]
    rows = cache.shape[0] * cache.shape[1] if cache.dim() == 3 else cache.shape[0]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(128 + 64)
    if u_out is None:
        u_out = torch.empty(B, Lq, H, 512, dtype=q_lat.dtype, device=q_lat.device)
    if lse_out is None:
        lse_out = torch.empty(B, Lq, H, dtype=torch.float32, device=q_lat.device)
    if o_out is None:
        o_out = torch.empty(B, Lq, H, 128, dtype=q_lat.dtype, device=q_lat.device)
    need = mla_decode_workspace_size(B, Lq, maxp, page_size, num_splits, H, cache_dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_lat.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().mla_decode_out_proj(_ptr(q_lat), _ptr(q_rope), _ptr(cache), _ptr(scales), _ptr(block_table),
                                    _ptr(seq_lens), B, Lq, maxp, rows // page_size, page_size, softmax_scale,
                                    num_splits, _ptr(workspace), ws_bytes, _ptr(w_uv), _ptr(u_out), _ptr(lse_out),
                                    _ptr(o_out), _ptr(dev_error), dims(H), _act_code(q_lat), DTYPE_CODE[cache_dtype],
                                    _stream(stream))
    _check("mla_decode_out_proj", st)
    return u_out, lse_out, o_out


def mla_decode_paged_static_scratch(q_lat, q_rope, cache, scales, block_table, seq_lens, page_size: int,
                                    cache_dtype: str, softmax_scale: Optional[float] = None, num_splits: int = 0,
                                    u_out=None, lse_out=None, dev_error=None, stream=None):
    """mla_decode_paged with the split-KV partials in the library's fixed device
    array (no workspace argument). u_out and lse_out must be passed in."""
    _contig_cuda(q_lat, q_rope, cache, scales, block_table, seq_lens, u_out, lse_out, dev_error)
    if u_out is None:
        raise ValueError("u_out is required")
    B, Lq, H = q_lat.shape[0], q_lat.shape[1], q_lat.shape[2]
    rows = cache.shape[0] * cache.shape[1] if cache.dim() == 3 else cache.shape[0]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(128 + 64)
    st = load().mla_decode_paged_static_scratch(
        _ptr(q_lat), _ptr(q_rope), _ptr(cache), _ptr(scales), _ptr(block_table), _ptr(seq_lens), B, Lq,
        block_table.shape[1], rows // page_size, page_size, softmax_scale, num_splits, _ptr(u_out), _ptr(lse_out),
        _ptr(dev_error), dims(H), _act_code(q_lat), DTYPE_CODE[cache_dtype], _stream(stream))
    _check("mla_decode_paged_static_scratch", st)
    return u_out, lse_out


def mla_prefill_workspace_size(n_tokens: int, heads: int) -> int:
    return load().mla_prefill_workspace_size(n_tokens, dims(heads))


def mla_prefill_mha(q_nope, q_rope, rows, w_uk, w_uv, softmax_scale: Optional[float] = None, workspace=None,
                    o_out=None, lse_out=None, dev_error=None, stream=None, want_lse: bool = True):
    """Prefill in the MHA form for one sequence: q_nope [Tq, H, 128], q_rope [Tq, H, 64],
    rows [T, 576] (the sequence's cache rows) -> (o [Tq, H, 128], lse [Tq, H] or None)."""
    _contig_cuda(q_nope, q_rope, rows, w_uk, w_uv, workspace, o_out, lse_out, dev_error)
    Tq, H = q_nope.shape[0], q_nope.shape[1]
    T = rows.shape[0]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(128 + 64)
    if o_out is None:
        o_out = torch.empty(Tq, H, 128, dtype=q_nope.dtype, device=q_nope.device)
    if lse_out is None and want_lse:
        lse_out = torch.empty(Tq, H, dtype=torch.float32, device=q_nope.device)
    need = mla_prefill_workspace_size(T, H)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_nope.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().mla_prefill_mha(_ptr(q_nope), _ptr(q_rope), _ptr(rows), _ptr(w_uk), _ptr(w_uv), T, Tq,
                                softmax_scale, _ptr(workspace), ws_bytes, _ptr(o_out), _ptr(lse_out), _ptr(dev_error),
                                dims(H), _act_code(q_nope), _stream(stream))
    _check("mla_prefill_mha", st)
    return o_out, lse_out


def merge_kernel_launches(path: int, splits: int, with_out_proj: bool) -> int:
    """Split-merge kernel launches of a decode call: none for one split, none
    when mla_decode_out_proj merges 2..4 splits of the tensor-core decode inside
    its projection kernel, else one."""
    if splits <= 1 or (with_out_proj and path == MLA_DECODE_PATH_TENSOR_CORE and splits <= 4):
        return 0
    return 1


def mla_decode_kernel_path(cache, scales, page_size: int, heads: int, act: str, cache_dtype: str) -> int:
    """Which decode kernel mla_decode_paged runs on this cache: MLA_DECODE_PATH_TENSOR_CORE
    or MLA_DECODE_PATH_CUDA_CORE."""
    rows = cache.shape[0] * cache.shape[1] if cache.dim() == 3 else cache.shape[0]
    out = ctypes.c_int32(0)
    st = load().mla_decode_kernel_path(_ptr(cache), _ptr(scales), rows // page_size, page_size, dims(heads),
                                       DTYPE_CODE[act], DTYPE_CODE[cache_dtype], ctypes.byref(out))
    _check("mla_decode_kernel_path", st)
    return out.value


def mla_read_device_error(dev_error, stream=None) -> int:
    code = ctypes.c_int32(0)
    st = load().mla_read_device_error(_ptr(dev_error), _stream(stream), ctypes.byref(code))
    if st not in (MLA_OK, MLA_ERR_DEVICE_FLAG):
        _check("mla_read_device_error", st)
    return code.value
