"""Device-memory helper around the C ABI: one Gated DeltaNet layer with its slot pool.

Allocation of the weights, the state pool and the prefill workspace happens here (torch owns
device memory); every computation is a call into libgdn.so through ``gdn``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import gdn
from .synth import BF16, Geometry


def torch_act(geo: Geometry):
    return torch.bfloat16 if geo.act == BF16 else torch.float32


def to_device(x: np.ndarray, dtype, device="cuda") -> torch.Tensor:
    """float32 ndarray holding act-dtype values -> device tensor of that dtype (exact)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device=device, dtype=dtype)


def pack_weight(w: torch.Tensor, stream=None) -> torch.Tensor:
    """A bf16 linear weight [N][K] on the device -> its packed tile layout (uint8 tensor)."""
    nbytes = gdn.gdn_proj_packed_bytes(w.shape[0], w.shape[1])
    if nbytes == 0:
        raise ValueError(f"cannot pack a weight of shape {tuple(w.shape)} (K must be a multiple of 64)")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    gdn.gdn_proj_pack(w, packed, stream)
    return packed


class GatedDeltaNetLayer:
    """Weights, state pool (rec f32 [N][Hv][dk][dv], conv act [N][K-1][Cqkv]) and status word."""

    def __init__(self, geo: Geometry, weights: dict, num_slots: int, device="cuda"):
        self.geo = geo
        self.device = device
        self.act = torch_act(geo)
        self.dims = gdn.make_dims(geo.Hk, geo.Hv, geo.dk, geo.dv, geo.K, geo.q_scale, geo.l2_eps,
                                  geo.norm_eps)
        self.A_log = to_device(weights["A_log"], torch.float32, device)
        self.dt_bias = to_device(weights["dt_bias"], torch.float32, device)
        self.conv_w = to_device(weights["conv_w"], self.act, device)
        self.norm_w = to_device(weights["norm_w"], self.act, device)
        self.w = gdn.make_weights(self.A_log, self.dt_bias, self.conv_w, self.norm_w)
        self.rec_state = torch.zeros((num_slots, geo.Hv, geo.dk, geo.dv), dtype=torch.float32,
                                     device=device)
        self.conv_state = torch.zeros((num_slots, geo.K - 1, geo.cqkv), dtype=self.act,
                                      device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.pool = gdn.make_pool(self.rec_state, self.conv_state, self.status)
        self._ws = None
        self.ws_cap = None   # bytes: a smaller prefill workspace (windows of whole chunks)

    @property
    def num_slots(self) -> int:
        return self.rec_state.shape[0]

    def load_state(self, rec: np.ndarray, conv: np.ndarray):
        self.rec_state.copy_(torch.from_numpy(np.ascontiguousarray(rec, np.float32)))
        self.conv_state.copy_(torch.from_numpy(np.ascontiguousarray(conv, np.float32)).to(self.act))

    def inputs(self, xs: dict) -> dict:
        return {k: to_device(v, self.act, self.device) for k, v in xs.items()}

    def decode_step(self, slot_idx: torch.Tensor, qkv, z, a, b, out=None, stream=None):
        if out is None:
            out = torch.empty((slot_idx.shape[0], self.geo.zdim), dtype=self.act, device=self.device)
        gdn.gdn_decode_step(self.dims, self.w, self.pool, slot_idx, qkv, z, a, b, out, stream)
        return out

    def decode_multi(self, slot_idx: torch.Tensor, qkv, z, a, b, out=None, stream=None):
        """T consecutive tokens per row: qkv [B][T][Cqkv], z [B][T][Hv*dv], a/b [B][T][Hv]."""
        if out is None:
            out = torch.empty((qkv.shape[0], qkv.shape[1], self.geo.zdim), dtype=self.act,
                              device=self.device)
        gdn.gdn_decode_multi(self.dims, self.w, self.pool, slot_idx, qkv, z, a, b, out, stream)
        return out

    def in_proj(self, hidden: torch.Tensor, w_in_packed: torch.Tensor, stream=None) -> dict:
        """Input projection of bf16 hidden states [rows][H] through the packed stacked weight
        (pack_weight of [Cqkv + Hv*dv + 2*Hv][H]): returns the step inputs qkv, z, a, b."""
        rows, g = hidden.shape[0], self.geo
        dev = hidden.device
        t = {"qkv": torch.empty((rows, g.cqkv), dtype=torch.bfloat16, device=dev),
             "z": torch.empty((rows, g.zdim), dtype=torch.bfloat16, device=dev),
             "a": torch.empty((rows, g.Hv), dtype=torch.bfloat16, device=dev),
             "b": torch.empty((rows, g.Hv), dtype=torch.bfloat16, device=dev)}
        gdn.gdn_in_proj(self.dims, hidden, w_in_packed, t["qkv"], t["z"], t["b"], t["a"],
                        self.status, stream)
        return t

    def out_proj(self, out: torch.Tensor, w_out_packed: torch.Tensor, hidden_size: int, y=None,
                 stream=None):
        """Output projection of the step's bf16 output [rows][Hv*dv] through the packed
        out_proj weight (pack_weight of [hidden_size][Hv*dv])."""
        if y is None:
            y = torch.empty((out.shape[0], hidden_size), dtype=torch.bfloat16, device=out.device)
        gdn.gdn_out_proj(self.dims, out, w_out_packed, y, self.status, stream)
        return y

    def conv1d_update(self, slot_idx: torch.Tensor, qkv_in, out=None, stream=None):
        if out is None:
            out = torch.empty_like(qkv_in)
        gdn.gdn_conv1d_update(self.dims, self.w, self.pool, slot_idx, qkv_in, out, stream)
        return out

    def workspace(self, num_seqs: int, total_tokens: int) -> torch.Tensor:
        need = gdn.gdn_prefill_workspace_bytes(self.dims, num_seqs, total_tokens)
        if self.ws_cap is not None:
            # head dims 128: the prefill runs in windows of whole chunks that fit the workspace
            need = max(gdn.gdn_prefill_workspace_bytes(self.dims, 1, 1), min(need, self.ws_cap))
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self._ws[:max(need, 256)]

    def prefill(self, cu_seqlens, slot_idx, has_init, qkv, z, a, b, out=None, stream=None):
        """cu_seqlens/slot_idx/has_init: device tensors (int32, int32, uint8 or None)."""
        total = qkv.shape[0]
        n = slot_idx.shape[0]
        if out is None:
            out = torch.empty((total, self.geo.zdim), dtype=self.act, device=self.device)
        ws = self.workspace(n, total)
        gdn.gdn_prefill_chunked(self.dims, self.w, self.pool, cu_seqlens, slot_idx, has_init, n,
                                total, qkv, z, a, b, out, ws, stream)
        return out

    def compact(self, src, dst, stream=None):
        gdn.gdn_state_compact(self.dims, gdn.act_code(self.act), self.pool, list(src), list(dst),
                              stream)


class _DeviceView:
    """A raw device buffer seen through __cuda_array_interface__ (no copy, no ownership)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 2}


class DecodeGraphs:
    """Bucketed CUDA-graph decode over a layer (gdn_decode_graphs_*): write rows [0, B) of the
    static input tensors, call step(B), read rows [0, B) of `out`."""

    def __init__(self, layer: GatedDeltaNetLayer, buckets):
        self.layer = layer
        self.handle = gdn.gdn_decode_graphs_create(layer.dims, layer.w, layer.pool, buckets)
        buf = gdn.gdn_decode_graphs_buffers(self.handle)
        self.max_batch = buf["max_batch"]
        geo, mb = layer.geo, buf["max_batch"]
        ts = "<f2" if layer.act == torch.bfloat16 else "<f4"

        def view(key, shape, typestr, dtype):
            t = torch.as_tensor(_DeviceView(buf[key], shape, typestr), device=layer.device)
            return t.view(dtype) if dtype is not None else t
        act = layer.act if layer.act == torch.bfloat16 else None
        self.slot_idx = view("slot_idx", (mb,), "<i4", None)
        self.qkv = view("qkv", (mb, geo.cqkv), ts, act)
        self.z = view("z", (mb, geo.zdim), ts, act)
        self.a = view("a", (mb, geo.Hv), ts, act)
        self.b = view("b", (mb, geo.Hv), ts, act)
        self.out = view("out", (mb, geo.zdim), ts, act)

    def step(self, B: int, stream=None):
        gdn.gdn_decode_graphs_launch(self.handle, B, stream)
        return self.out[:B]

    def close(self):
        if self.handle:
            torch.cuda.synchronize()
            gdn.gdn_decode_graphs_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
