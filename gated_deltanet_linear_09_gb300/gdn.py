"""Thin ctypes binding of libgdn.so (the C ABI declared in include/gdn.h).

Argument marshalling only: every function passes device pointers (``tensor.data_ptr()``),
sizes and the current CUDA stream to the C entry point of the same name and raises on a
non-zero return code.  Every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library has not been built, or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

GDN_F32 = 0
GDN_BF16 = 1
GDN_MAX_COMPACT_PAIRS = 2048
GDN_STATUS_SLOT_RANGE = 1
GDN_STATUS_BAD_SEQLENS = 2

_CODES = {
    0: "GDN_OK", -1: "GDN_ERR_INVALID_ARG", -2: "GDN_ERR_UNSUPPORTED_SHAPE",
    -3: "GDN_ERR_HEAD_DIVISIBILITY", -4: "GDN_ERR_SLOT_RANGE", -5: "GDN_ERR_WORKSPACE_TOO_SMALL",
    -6: "GDN_ERR_OVERLAP", -7: "GDN_ERR_MISALIGNED", -8: "GDN_ERR_CUDA", -9: "GDN_ERR_TOO_LARGE",
}

# Every symbol include/gdn.h declares.
EXPORTED = ("gdn_state_slot_bytes", "gdn_conv1d_update", "gdn_decode_step", "gdn_decode_multi",
            "gdn_prefill_workspace_bytes", "gdn_prefill_chunked", "gdn_state_compact",
            "gdn_status_string", "gdn_prefill_chunked_noalloc", "gdn_decode_graphs_create",
            "gdn_decode_graphs_buffers", "gdn_decode_graphs_launch", "gdn_decode_graphs_destroy",
            "gdn_proj_packed_bytes", "gdn_proj_pack", "gdn_linear_bf16", "gdn_in_proj",
            "gdn_out_proj")
GDN_MAX_DECODE_TOKENS = 8
GDN_MAX_GRAPH_BUCKETS = 16
GDN_NOALLOC_PREFILL_SCRATCH_BYTES = 64 << 20
GDN_MAX_PROJ_SEGMENTS = 4
GDN_PROJ_BLOCK_BYTES = 16384


class GdnError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {_CODES.get(code, code)} ({msg})")
        self.code = code


class gdn_dims(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_kernel", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float)]


class gdn_weights(ctypes.Structure):
    _fields_ = [("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("conv_weight", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p),
                ("act", ctypes.c_int)]


class gdn_proj_route(ctypes.Structure):
    _fields_ = [("nseg", ctypes.c_int32), ("start", ctypes.c_int32 * GDN_MAX_PROJ_SEGMENTS),
                ("ld", ctypes.c_int32 * GDN_MAX_PROJ_SEGMENTS),
                ("dst", ctypes.c_void_p * GDN_MAX_PROJ_SEGMENTS)]


class gdn_pool(ctypes.Structure):
    _fields_ = [("rec_state", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
                ("num_slots", ctypes.c_int32), ("status", ctypes.c_void_p)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libgdn.so (optionally building it first).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libgdn.so is not built ({path}); run __graft_entry__.build() or "
                           "python -m gated_deltanet_linear_09_gb300.build")
    lib = ctypes.CDLL(path)
    lib.gdn_state_slot_bytes.restype = ctypes.c_size_t
    lib.gdn_state_slot_bytes.argtypes = [_P, ctypes.c_int]
    lib.gdn_conv1d_update.restype = ctypes.c_int
    lib.gdn_conv1d_update.argtypes = [_P, _P, _P, _P, _I32, _P, _P, _P]
    lib.gdn_decode_step.restype = ctypes.c_int
    lib.gdn_decode_step.argtypes = [_P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P]
    lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_decode_multi.argtypes = [_P, _P, _P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P]
    lib.gdn_decode_multi.restype = ctypes.c_int
    lib.gdn_decode_graphs_create.argtypes = [_P, _P, _P, _P, _I32, _P]
    lib.gdn_decode_graphs_create.restype = ctypes.c_int
    lib.gdn_decode_graphs_buffers.argtypes = [_P] + [_P] * 7
    lib.gdn_decode_graphs_buffers.restype = ctypes.c_int
    lib.gdn_decode_graphs_launch.argtypes = [_P, _I32, _P]
    lib.gdn_decode_graphs_launch.restype = ctypes.c_int
    lib.gdn_decode_graphs_destroy.argtypes = [_P]
    lib.gdn_decode_graphs_destroy.restype = None
    lib.gdn_prefill_workspace_bytes.argtypes = [_P, _I32, _I32]
    lib.gdn_prefill_chunked.restype = ctypes.c_int
    lib.gdn_prefill_chunked.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I32, _P, _P, _P, _P, _P,
                                        _P, ctypes.c_size_t, _P]
    lib.gdn_prefill_chunked_noalloc.restype = ctypes.c_int
    lib.gdn_prefill_chunked_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I32, _P, _P, _P, _P,
                                                _P, _P]
    lib.gdn_state_compact.restype = ctypes.c_int
    lib.gdn_state_compact.argtypes = [_P, ctypes.c_int, _P, _P, _P, _I32, _P]
    lib.gdn_proj_packed_bytes.restype = ctypes.c_size_t
    lib.gdn_proj_packed_bytes.argtypes = [_I32, _I32]
    lib.gdn_proj_pack.restype = ctypes.c_int
    lib.gdn_proj_pack.argtypes = [_P, _I32, _I32, _P, ctypes.c_size_t, _P]
    lib.gdn_linear_bf16.restype = ctypes.c_int
    lib.gdn_linear_bf16.argtypes = [_P, _P, _I32, _I32, _I32, _P, _I32, _P, _P]
    lib.gdn_in_proj.restype = ctypes.c_int
    lib.gdn_in_proj.argtypes = [_P, _P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P]
    lib.gdn_out_proj.restype = ctypes.c_int
    lib.gdn_out_proj.argtypes = [_P, _P, _P, _I32, _I32, _P, _P, _P]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise GdnError(fn, rc, load().gdn_status_string(rc).decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def act_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return GDN_BF16
    if dtype == torch.float32:
        return GDN_F32
    raise ValueError(f"unsupported activation dtype {dtype}")


def make_dims(Hk, Hv, dk, dv, K=4, q_scale=0.0, l2_eps=1e-6, norm_eps=1e-6) -> gdn_dims:
    return gdn_dims(Hk, Hv, dk, dv, K, q_scale, l2_eps, norm_eps)


def make_weights(A_log, dt_bias, conv_weight, norm_weight) -> gdn_weights:
    return gdn_weights(_ptr(A_log), _ptr(dt_bias), _ptr(conv_weight), _ptr(norm_weight),
                       act_code(conv_weight.dtype))


def make_pool(rec_state, conv_state, status=None) -> gdn_pool:
    return gdn_pool(_ptr(rec_state), _ptr(conv_state), rec_state.shape[0], _ptr(status))


# ---------------------------------------------------------------- the C entry points

def gdn_state_slot_bytes(dims: gdn_dims, act: int) -> int:
    return int(load().gdn_state_slot_bytes(ctypes.byref(dims), act))


def gdn_conv1d_update(dims, weights, pool, slot_idx, qkv_in, qkv_out, stream=None):
    B = qkv_in.shape[0] if qkv_in is not None else 0
    _check("gdn_conv1d_update", load().gdn_conv1d_update(
        ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(pool), _ptr(slot_idx), B,
        _ptr(qkv_in), _ptr(qkv_out), _stream(stream)))


def gdn_decode_step(dims, weights, pool, slot_idx, qkv, z, a, b, out, stream=None):
    B = slot_idx.shape[0]
    _check("gdn_decode_step", load().gdn_decode_step(
        ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(pool), _ptr(slot_idx), B,
        _ptr(qkv), _ptr(z), _ptr(a), _ptr(b), _ptr(out), _stream(stream)))


def gdn_decode_multi(dims, weights, pool, slot_idx, qkv, z, a, b, out, stream=None):
    """T tokens per row: qkv [B][T][Cqkv], z/out [B][T][Hv*dv], a/b [B][T][Hv]."""
    B, T = int(qkv.shape[0]), int(qkv.shape[1])
    _check("gdn_decode_multi", load().gdn_decode_multi(
        ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(pool), _ptr(slot_idx), B, T,
        _ptr(qkv), _ptr(z), _ptr(a), _ptr(b), _ptr(out), _stream(stream)))


def gdn_decode_graphs_create(dims, weights, pool, buckets) -> int:
    """Returns the object handle (an address)."""
    arr = (ctypes.c_int32 * len(buckets))(*[int(x) for x in buckets])
    h = ctypes.c_void_p()
    _check("gdn_decode_graphs_create", load().gdn_decode_graphs_create(
        ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(pool), arr, len(buckets),
        ctypes.byref(h)))
    return h.value


def gdn_decode_graphs_buffers(handle) -> dict:
    """Device addresses of the static buffers and the largest bucket."""
    ptrs = [ctypes.c_void_p() for _ in range(6)]
    mb = ctypes.c_int32()
    _check("gdn_decode_graphs_buffers", load().gdn_decode_graphs_buffers(
        handle, *[ctypes.byref(p) for p in ptrs], ctypes.byref(mb)))
    d = dict(zip(("slot_idx", "qkv", "z", "a", "b", "out"), (p.value for p in ptrs)))
    d["max_batch"] = mb.value
    return d


def gdn_decode_graphs_launch(handle, B: int, stream=None):
    _check("gdn_decode_graphs_launch", load().gdn_decode_graphs_launch(handle, B, _stream(stream)))


def gdn_decode_graphs_destroy(handle):
    load().gdn_decode_graphs_destroy(handle)


def gdn_prefill_workspace_bytes(dims, num_seqs: int, total_tokens: int) -> int:
    return int(load().gdn_prefill_workspace_bytes(ctypes.byref(dims), num_seqs, total_tokens))


def gdn_prefill_chunked(dims, weights, pool, cu_seqlens, slot_idx, has_initial_state, num_seqs,
                        total_tokens, qkv, z, a, b, out, workspace, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("gdn_prefill_chunked", load().gdn_prefill_chunked(
        ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(pool), _ptr(cu_seqlens),
        _ptr(slot_idx), _ptr(has_initial_state), num_seqs, total_tokens, _ptr(qkv), _ptr(z),
        _ptr(a), _ptr(b), _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))


def gdn_prefill_chunked_noalloc(dims, weights, pool, cu_seqlens, slot_idx, has_initial_state,
                                num_seqs, total_tokens, qkv, z, a, b, out, stream=None):
    """Prefill whose scratch is the library's fixed device array: allocates nothing."""
    _check("gdn_prefill_chunked_noalloc", load().gdn_prefill_chunked_noalloc(
        ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(pool), _ptr(cu_seqlens),
        _ptr(slot_idx), _ptr(has_initial_state), num_seqs, total_tokens, _ptr(qkv), _ptr(z),
        _ptr(a), _ptr(b), _ptr(out), _stream(stream)))


def gdn_state_compact(dims, act: int, pool, src_slots, dst_slots, stream=None):
    src = (ctypes.c_int32 * len(src_slots))(*[int(x) for x in src_slots])
    dst = (ctypes.c_int32 * len(dst_slots))(*[int(x) for x in dst_slots])
    if len(src_slots) != len(dst_slots):
        raise ValueError("src_slots and dst_slots differ in length")
    _check("gdn_state_compact", load().gdn_state_compact(
        ctypes.byref(dims), act, ctypes.byref(pool), src, dst, len(src_slots), _stream(stream)))


def make_route(segments) -> gdn_proj_route:
    """segments: [(start, ld, dst tensor or address), ...] in increasing start order."""
    r = gdn_proj_route()
    r.nseg = len(segments)
    for i, (start, ld, dst) in enumerate(segments):
        r.start[i] = int(start)
        r.ld[i] = int(ld)
        r.dst[i] = _ptr(dst)
    return r


def gdn_proj_packed_bytes(N: int, K: int) -> int:
    return int(load().gdn_proj_packed_bytes(int(N), int(K)))


def gdn_proj_pack(w, packed, stream=None):
    """Packs a bf16 linear weight w [N][K] into the tile layout (packed: a uint8 device tensor)."""
    N, K = int(w.shape[0]), int(w.shape[1])
    _check("gdn_proj_pack", load().gdn_proj_pack(
        _ptr(w), N, K, _ptr(packed), packed.numel() * packed.element_size(), _stream(stream)))


def gdn_linear_bf16(x, w_packed, N: int, route: gdn_proj_route, k_split: int = 0, status=None,
                    stream=None):
    """y = x w^T (bf16, f32 sums): x [M][K], w packed from [N][K]; outputs go where route says."""
    M, K = int(x.shape[0]), int(x.shape[1])
    _check("gdn_linear_bf16", load().gdn_linear_bf16(
        _ptr(x), _ptr(w_packed), M, int(N), K, ctypes.byref(route), int(k_split), _ptr(status),
        _stream(stream)))


def gdn_in_proj(dims, hidden, w_in_packed, qkv, z, b, a, status=None, stream=None):
    """hidden [rows][H], packed w_in [Cqkv + Hv*dv + 2*Hv][H] -> qkv, z, b, a (step layouts)."""
    rows, H = int(hidden.shape[0]), int(hidden.shape[1])
    _check("gdn_in_proj", load().gdn_in_proj(
        ctypes.byref(dims), _ptr(hidden), _ptr(w_in_packed), rows, H, _ptr(qkv), _ptr(z),
        _ptr(b), _ptr(a), _ptr(status), _stream(stream)))


def gdn_out_proj(dims, out, w_out_packed, y, status=None, stream=None):
    """out [rows][Hv*dv], packed w_out [H][Hv*dv] -> y [rows][H] (bf16)."""
    rows, H = int(out.shape[0]), int(y.shape[1])
    _check("gdn_out_proj", load().gdn_out_proj(
        ctypes.byref(dims), _ptr(out), _ptr(w_out_packed), rows, H, _ptr(y), _ptr(status),
        _stream(stream)))


def gdn_status_string(code: int) -> str:
    return load().gdn_status_string(code).decode()
