"""One MLA decode layer over a paged latent cache, driven through the C ABI.

MLADecodeLayer owns the device state of one attention layer: the weights
W_UK, W_UV, the paged latent cache (and E4M3 scales), the RoPE tables, the
block table / sequence lengths, and reusable workspace and output buffers. A
decode step is

    append(new tokens) -> absorb_q -> decode_out_proj (decode_paged + out_proj)

on one stream, with no allocation in the step once the buffers exist; with
2 to 4 KV splits the split merge runs inside the projection kernel.

With the model-level weights attached (attach_front, attach_output), a step can
start from the hidden states of the new tokens and end in the model dimension:

    decode_front(h) -> append -> absorb_q -> decode_paged -> out_proj_fused (or out_proj, W_O)
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import capi
from .workloads import BF16, E4M3, F32, ROW, TORCH_DTYPE, Workload

CACHE_TORCH = {F32: torch.float32, BF16: torch.bfloat16, E4M3: torch.uint8}


class MLADecodeLayer:
    def __init__(self, w: Workload, w_uk: torch.Tensor, w_uv: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, device="cuda", poison: bool = True, num_splits: Optional[int] = None):
        self.w = w
        self.device = torch.device(device)
        self.H = w.heads
        self.P = w.page_size
        self.cache_dtype = w.cache_dtype
        self.act = TORCH_DTYPE[w.act_dtype]
        self.w_uk = w_uk.to(self.device).contiguous()
        self.w_uv = w_uv.to(self.device).contiguous()
        self.block_table = block_table.to(self.device, torch.int32).contiguous()
        self.seq_lens = seq_lens.to(self.device, torch.int32).contiguous()
        self.num_pages = w.num_pages
        ct = CACHE_TORCH[w.cache_dtype]
        self.cache = torch.empty(self.num_pages, self.P, ROW, dtype=ct, device=self.device)
        self.scales = (torch.empty(self.num_pages, self.P, 5, dtype=torch.float32, device=self.device)
                       if w.cache_dtype == E4M3 else None)
        if poison:
            self.poison()
        cos, sin = capi.mla_rope_table(max(w.max_pos, 1), 64, w.rope_base)
        self.rope_cos = cos.to(self.device)
        self.rope_sin = sin.to(self.device)
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.num_splits = w.num_splits if num_splits is None else num_splits
        B, Lq = w.batch, w.q_len
        self.splits = capi.mla_decode_num_splits(B, Lq, w.max_pages_per_seq, self.P, self.num_splits, self.H,
                                                 self.cache_dtype)
        need = capi.mla_decode_workspace_size(B, Lq, w.max_pages_per_seq, self.P, self.num_splits, self.H,
                                              self.cache_dtype)
        self.workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=self.device)
        self.q_lat = torch.empty(B, Lq, self.H, 512, dtype=self.act, device=self.device)
        self.u = torch.empty(B, Lq, self.H, 512, dtype=self.act, device=self.device)
        self.lse = torch.empty(B, Lq, self.H, dtype=torch.float32, device=self.device)
        self.o = torch.empty(B, Lq, self.H, 128, dtype=self.act, device=self.device)
        self.softmax_scale = 1.0 / math.sqrt(128 + 64)

    def poison(self):
        """Fill the pool with NaN (values and scales) so unwritten rows are visible."""
        if self.cache_dtype == E4M3:
            self.cache.fill_(0x7F)
            self.scales.fill_(float("nan"))
        else:
            self.cache.fill_(float("nan"))

    def append(self, c_kv, k_r, positions, slots, stream=None):
        capi.mla_cache_append(c_kv, k_r, positions, slots, self.rope_cos, self.rope_sin, self.cache, self.scales,
                              self.P, self.cache_dtype, self.dev_error, stream)

    def append_chunked(self, c_kv, k_r, positions, slots, chunk: int = 1 << 18):
        """Fill a long context from host or device tensors, chunk by chunk."""
        n = c_kv.shape[0]
        for i in range(0, n, chunk):
            sl = slice(i, min(n, i + chunk))
            self.append(c_kv[sl].to(self.device, non_blocking=True).contiguous(),
                        k_r[sl].to(self.device, non_blocking=True).contiguous(),
                        positions[sl].to(self.device, non_blocking=True).contiguous(),
                        slots[sl].to(self.device, non_blocking=True).contiguous())

    def absorb(self, q_nope, stream=None):
        return capi.mla_absorb_q(q_nope, self.w_uk, self.q_lat, stream)

    def decode(self, q_lat, q_rope, stream=None):
        return capi.mla_decode_paged(q_lat, q_rope, self.cache, self.scales, self.block_table, self.seq_lens, self.P,
                                     self.cache_dtype, self.softmax_scale, self.num_splits, self.workspace, self.u,
                                     self.lse, self.dev_error, stream)

    def out_proj(self, u, stream=None):
        return capi.mla_out_proj(u, self.w_uv, self.o, stream)

    def decode_out_proj(self, q_lat, q_rope, stream=None):
        """decode then out_proj as one call (the KV splits merged inside the
        projection kernel where the library can); fills u, lse and o."""
        capi.mla_decode_out_proj(q_lat, q_rope, self.cache, self.scales, self.block_table, self.seq_lens, self.P,
                                 self.cache_dtype, self.w_uv, self.softmax_scale, self.num_splits, self.workspace,
                                 self.u, self.lse, self.o, self.dev_error, stream)
        return self.o

    def step(self, q_nope, q_rope, new_c_kv, new_k_r, new_positions, new_slots, stream=None):
        """One decode step: append the q_len new tokens, then attend. Returns o."""
        if new_c_kv is not None and new_c_kv.shape[0] > 0:
            self.append(new_c_kv, new_k_r, new_positions, new_slots, stream)
        q_lat = self.absorb(q_nope, stream)
        return self.decode_out_proj(q_lat, q_rope, stream)

    # ------------------------------------------------------------------ model-level weights

    def attach_front(self, w_dq, w_dkv, w_kr, g_q, g_kv, w_uq, w_qr, eps: float):
        """Front-end weights (nn.Linear layouts [out, in]) and RMSNorm gains. The
        three down-projections and the two query up-projections are stacked once
        here, as mla_decode_front takes them; its workspace and outputs are
        allocated for the layer's B*Lq tokens."""
        dev = self.device
        self.w_dqkv = torch.cat([w_dq, w_dkv, w_kr], 0).to(dev).contiguous()
        self.w_uqr = torch.cat([w_uq, w_qr], 0).to(dev).contiguous()
        self.g_q = g_q.to(dev).contiguous()
        self.g_kv = g_kv.to(dev).contiguous()
        self.rms_eps = float(eps)
        n = self.w.batch * self.w.q_len
        d_model, d_cq = w_dq.shape[1], w_dq.shape[0]
        act = self.w.act_dtype
        self.front_ws = torch.empty(max(16, capi.mla_decode_front_workspace_size(n, d_model, d_cq, self.H, act)),
                                    dtype=torch.uint8, device=dev)
        mk = lambda *shape: torch.empty(*shape, dtype=self.act, device=dev)
        self.q_nope_buf, self.q_rope_buf = mk(n, self.H, 128), mk(n, self.H, 64)
        self.c_kv_buf, self.k_r_buf = mk(n, 512), mk(n, 64)

    def attach_output(self, w_o, fused: bool = True):
        """The output projection W_O [d_model, H, 128]. fused=True folds W_UV
        into it once (mla_fuse_out_weights) and a step ends with one product over
        all heads; fused=False keeps W_UV per head and applies W_O to the
        concatenated head outputs."""
        dev = self.device
        n = self.w.batch * self.w.q_len
        d_model = w_o.shape[0]
        act = self.w.act_dtype
        self.out_fused = fused
        w_o = w_o.to(dev).contiguous()
        if fused:
            self.w_out = capi.mla_fuse_out_weights(w_o, self.w_uv)
            need = capi.mla_out_proj_fused_workspace_size(n, d_model, self.H, act)
        else:
            self.w_out = w_o.view(d_model, self.H * 128)
            need = capi.mla_linear_workspace_size(n, d_model, self.H * 128, act)
        self.out_ws = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
        self.y = torch.empty(self.w.batch, self.w.q_len, d_model, dtype=self.act, device=dev)

    def front(self, h, positions, stream=None):
        """decode_front: h [B*Lq, d_model] -> (q_nope, q_rope, c_kv, k_r) in the layer's buffers."""
        return capi.mla_decode_front(h, self.w_dqkv, self.g_q, self.g_kv, self.w_uqr, positions, self.rope_cos,
                                     self.rope_sin, self.rms_eps, self.H, self.q_nope_buf, self.q_rope_buf,
                                     self.c_kv_buf, self.k_r_buf, self.front_ws, self.dev_error, stream)

    def output(self, u, stream=None):
        """u [B, Lq, H, 512] -> y [B, Lq, d_model] through the attached output projection."""
        if self.out_fused:
            return capi.mla_out_proj_fused(u, self.w_out, self.y, self.out_ws, stream)
        o = self.out_proj(u, stream)
        capi.mla_linear(o.view(-1, self.H * 128), self.w_out, self.y.view(-1, self.y.shape[-1]), self.out_ws,
                        stream)
        return self.y

    def step_from_hidden(self, h, positions, slots, stream=None):
        """One whole layer step: front end on the new tokens' hidden states, their
        rows appended at `slots`, absorbed paged decode, output projection.
        Returns y [B, Lq, d_model]."""
        B, Lq = self.w.batch, self.w.q_len
        q_nope, q_rope, c_kv, k_r = self.front(h, positions, stream)
        self.append(c_kv, k_r, positions, slots, stream)
        q_lat = self.absorb(q_nope.view(B, Lq, self.H, 128), stream)
        if self.out_fused:
            u, _ = self.decode(q_lat, q_rope.view(B, Lq, self.H, 64), stream)
            return self.output(u, stream)
        # W_UV per head (with the KV split merge inside its kernel), then W_O
        o = self.decode_out_proj(q_lat, q_rope.view(B, Lq, self.H, 64), stream)
        capi.mla_linear(o.view(-1, self.H * 128), self.w_out, self.y.view(-1, self.y.shape[-1]), self.out_ws, stream)
        return self.y

    def device_error(self) -> int:
        return capi.mla_read_device_error(self.dev_error)

    def capture(self, fn, warmup: int = 2):
        """Capture fn() (a sequence of this layer's calls on the current stream)
        into a CUDA graph. Every buffer fn touches must already exist; the
        library itself never allocates. Returns the torch.cuda.CUDAGraph."""
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream(self.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g


def build_layer(w: Workload, d: dict, device="cuda", fill_context: bool = True, **kw) -> MLADecodeLayer:
    """A layer for workload w with the inputs d of workloads.make_inputs, its cache
    filled with every context token except the step's new ones (when fill_context)."""
    layer = MLADecodeLayer(w, d["w_uk"], d["w_uv"], d["block_table"], d["seq_lens"], device=device, **kw)
    if fill_context:
        n = d["ctx_c_kv"].shape[0]
        keep = torch.ones(n, dtype=torch.bool)
        keep[d["new_index"]] = False
        idx = torch.nonzero(keep)[:, 0]
        layer.append_chunked(d["ctx_c_kv"][idx], d["ctx_k_r"][idx], d["ctx_positions"][idx], d["ctx_slots"][idx])
    return layer


def step_inputs(d: dict, device="cuda"):
    """Device tensors of one step's inputs (queries and the new tokens)."""
    ni = d["new_index"]
    return dict(q_nope=d["q_nope"].to(device).contiguous(), q_rope=d["q_rope"].to(device).contiguous(),
                new_c_kv=d["ctx_c_kv"][ni].to(device).contiguous(), new_k_r=d["ctx_k_r"][ni].to(device).contiguous(),
                new_positions=d["ctx_positions"][ni].to(device).contiguous(),
                new_slots=d["ctx_slots"][ni].to(device).contiguous())
