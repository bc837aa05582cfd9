"""float64 CPU oracle for the Gated DeltaNet layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product library (``gated_deltanet_linear_09_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, IEEE double, built with FMA
contraction off so results are identical on x86-64 and aarch64).  This module
builds it with gcc and wraps each entry point with numpy marshalling only.
Every wrapped function cites, in the C source, the passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def compile_to(src: str, out: str) -> None:
    """Compile an oracle source file into a shared library (gcc, -O2, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so.  GDN_ORACLE_LIB, when set, names an
    already built library to load instead (the mutation tests point it at deliberately broken
    copies of the oracle)."""
    override = os.environ.get("GDN_ORACLE_LIB")
    if override:
        return override
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        compile_to(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_D = ctypes.c_double
_I = ctypes.c_int
_P = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        for name in ("oracle_softplus", "oracle_sigmoid", "oracle_silu"):
            getattr(lib, name).restype = _D
            getattr(lib, name).argtypes = [_D]
        lib.oracle_gates.argtypes = [_D, _D, _D, _D, _P, _P]
        lib.oracle_conv_step.argtypes = [_I, _I, _P, _P, _P, _P]
        lib.oracle_l2norm.argtypes = [_I, _P, _D, _D, _P]
        lib.oracle_core_step.argtypes = [_I, _I, _P, _P, _P, _P, _D, _D, _P]
        lib.oracle_gated_rmsnorm.argtypes = [_I, _P, _P, _P, _D, _P]
        lib.oracle_decode_step.restype = _I
        lib.oracle_decode_step.argtypes = [_I] * 5 + [_D] * 3 + [_P] * 6 + [_I, _P, _I] + [_P] * 5
        lib.oracle_conv1d_update.restype = _I
        lib.oracle_conv1d_update.argtypes = [_I, _I, _P, _P, _I, _P, _I, _P, _P]
        lib.oracle_prefill.restype = _I
        lib.oracle_prefill.argtypes = [_I] * 5 + [_D] * 3 + [_P] * 6 + [_I, _P, _P, _P, _I] + [_P] * 5
        lib.oracle_prefill_chunkwise.restype = _I
        lib.oracle_prefill_chunkwise.argtypes = lib.oracle_prefill.argtypes + [_I]
        lib.oracle_state_compact.restype = _I
        lib.oracle_state_compact.argtypes = [_P, _P, _I, ctypes.c_int64, ctypes.c_int64, _P, _P, _I]
        lib.oracle_linear.argtypes = [_I, _I, _I, _P, _P, _P]
        lib.oracle_in_proj.argtypes = [_I] * 6 + [_P] * 6
        _lib = lib
    return _lib


def _f64(x, writable=False):
    a = np.ascontiguousarray(x, dtype=np.float64)
    if writable and a is x:
        return a
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_c_f64(a, name):
    if not (isinstance(a, np.ndarray) and a.dtype == np.float64 and a.flags.c_contiguous):
        raise TypeError(f"{name} must be a C-contiguous float64 ndarray (updated in place)")


def _check_i32(a, name):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


# ---------------------------------------------------------------- scalars

def softplus(x: float) -> float:
    return _load().oracle_softplus(float(x))


def sigmoid(x: float) -> float:
    return _load().oracle_sigmoid(float(x))


def silu(x: float) -> float:
    return _load().oracle_silu(float(x))


def gates(A_log: float, dt_bias: float, a: float, b: float):
    """(g, beta) of one V-head for one token."""
    g = ctypes.c_double()
    beta = ctypes.c_double()
    _load().oracle_gates(float(A_log), float(dt_bias), float(a), float(b), ctypes.byref(g),
                         ctypes.byref(beta))
    return g.value, beta.value


def conv_step(state: np.ndarray, w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """One conv token. state [K-1][C] f64 (updated in place), w [C][K], x [C] -> y [C]."""
    _check_c_f64(state, "state")
    C = x.shape[0]
    K = w.shape[1]
    w = _f64(w)
    x = _f64(x)
    y = np.zeros(C)
    _load().oracle_conv_step(C, K, _ptr(state), _ptr(w), _ptr(x), _ptr(y))
    return y


def l2norm(x: np.ndarray, eps: float, scale: float = 1.0) -> np.ndarray:
    x = _f64(x)
    y = np.zeros_like(x)
    _load().oracle_l2norm(x.shape[0], _ptr(x), float(eps), float(scale), _ptr(y))
    return y


def core_step(S: np.ndarray, k, v, q, g: float, beta: float) -> np.ndarray:
    """One delta-rule token on S [dk][dv] (updated in place); returns o = S_new^T q."""
    _check_c_f64(S, "S")
    dk, dv = S.shape
    k = _f64(k)
    v = _f64(v)
    q = _f64(q)
    o = np.zeros(dv)
    _load().oracle_core_step(dk, dv, _ptr(S), _ptr(k), _ptr(v), _ptr(q), float(g), float(beta),
                             _ptr(o))
    return o


def gated_rmsnorm(o, z, w, eps: float) -> np.ndarray:
    o = _f64(o)
    z = _f64(z)
    w = _f64(w)
    out = np.zeros_like(o)
    _load().oracle_gated_rmsnorm(o.shape[0], _ptr(o), _ptr(z), _ptr(w), float(eps), _ptr(out))
    return out


# ---------------------------------------------------------------- layer calls

def _dims_args(dims):
    return (int(dims["Hk"]), int(dims["Hv"]), int(dims["dk"]), int(dims["dv"]), int(dims["K"]),
            float(dims["q_scale"]), float(dims["l2_eps"]), float(dims["norm_eps"]))


def decode_step(dims, weights, rec_state, conv_state, slot_idx, qkv, z, a, b):
    """Batched decode step; rec_state [N][Hv][dk][dv] and conv_state [N][K-1][Cqkv] (f64) are
    updated in place.  Returns (rc, out [B][Hv*dv])."""
    _check_c_f64(rec_state, "rec_state")
    _check_c_f64(conv_state, "conv_state")
    slot_idx = _check_i32(slot_idx, "slot_idx")
    B = slot_idx.shape[0]
    qkv, z, a, b = (_f64(t) for t in (qkv, z, a, b))
    A_log, dt_bias, conv_w, norm_w = (_f64(weights[k]) for k in ("A_log", "dt_bias", "conv_w",
                                                                  "norm_w"))
    out = np.zeros((B, int(dims["Hv"]) * int(dims["dv"])))
    rc = _load().oracle_decode_step(*_dims_args(dims), _ptr(A_log), _ptr(dt_bias), _ptr(conv_w),
                                    _ptr(norm_w), _ptr(rec_state), _ptr(conv_state),
                                    rec_state.shape[0], _ptr(slot_idx), B, _ptr(qkv), _ptr(z),
                                    _ptr(a), _ptr(b), _ptr(out))
    return rc, out


def conv1d_update(conv_w, conv_state, slot_idx, qkv_in):
    _check_c_f64(conv_state, "conv_state")
    slot_idx = _check_i32(slot_idx, "slot_idx")
    conv_w = _f64(conv_w)
    qkv_in = _f64(qkv_in)
    B, C = qkv_in.shape
    out = np.zeros((B, C))
    rc = _load().oracle_conv1d_update(C, conv_w.shape[1], _ptr(conv_w), _ptr(conv_state),
                                      conv_state.shape[0], _ptr(slot_idx), B, _ptr(qkv_in),
                                      _ptr(out))
    return rc, out


def _prefill_common(fn, dims, weights, rec_state, conv_state, cu_seqlens, slot_idx, has_init,
                    qkv, z, a, b, extra=()):
    _check_c_f64(rec_state, "rec_state")
    _check_c_f64(conv_state, "conv_state")
    cu = _check_i32(cu_seqlens, "cu_seqlens")
    slot_idx = _check_i32(slot_idx, "slot_idx")
    n = slot_idx.shape[0]
    hi = np.ascontiguousarray(has_init if has_init is not None else np.zeros(n), dtype=np.uint8)
    qkv, z, a, b = (_f64(t) for t in (qkv, z, a, b))
    A_log, dt_bias, conv_w, norm_w = (_f64(weights[k]) for k in ("A_log", "dt_bias", "conv_w",
                                                                  "norm_w"))
    T = int(cu[-1]) if n > 0 else 0
    out = np.zeros((T, int(dims["Hv"]) * int(dims["dv"])))
    rc = fn(*_dims_args(dims), _ptr(A_log), _ptr(dt_bias), _ptr(conv_w), _ptr(norm_w),
            _ptr(rec_state), _ptr(conv_state), rec_state.shape[0], _ptr(cu), _ptr(slot_idx),
            _ptr(hi), n, _ptr(qkv), _ptr(z), _ptr(a), _ptr(b), _ptr(out), *extra)
    return rc, out


def prefill(dims, weights, rec_state, conv_state, cu_seqlens, slot_idx, has_init, qkv, z, a, b):
    """Token-by-token prefill of packed sequences (the definition).  Returns (rc, out [T][Hv*dv])."""
    return _prefill_common(_load().oracle_prefill, dims, weights, rec_state, conv_state,
                           cu_seqlens, slot_idx, has_init, qkv, z, a, b)


def prefill_chunkwise(dims, weights, rec_state, conv_state, cu_seqlens, slot_idx, has_init, qkv,
                      z, a, b, chunk):
    """The chunkwise WY/UT form of the same prefill (pins the GPU prefill's algebra)."""
    return _prefill_common(_load().oracle_prefill_chunkwise, dims, weights, rec_state, conv_state,
                           cu_seqlens, slot_idx, has_init, qkv, z, a, b, extra=(int(chunk),))


def state_compact(rec_state, conv_state, src, dst):
    _check_c_f64(rec_state, "rec_state")
    _check_c_f64(conv_state, "conv_state")
    src = _check_i32(src, "src")
    dst = _check_i32(dst, "dst")
    N = rec_state.shape[0]
    return _load().oracle_state_compact(_ptr(rec_state), _ptr(conv_state), N,
                                        rec_state[0].size if N else 0,
                                        conv_state[0].size if N else 0, _ptr(src), _ptr(dst),
                                        src.shape[0])


# ---------------------------------------------------------------- projections

def linear(x, w) -> np.ndarray:
    """y = x w^T for x [M][K] and w [N][K] (weight row n = output feature n)."""
    x = _f64(x)
    w = _f64(w)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("x and w disagree on K")
    y = np.zeros((M, N))
    _load().oracle_linear(M, N, K, _ptr(x), _ptr(w), _ptr(y))
    return y


def in_proj(dims, x, w_in):
    """The stacked input projection; returns dict(qkv, z, b, a) of [rows][...] float64."""
    Hk, Hv, dk, dv = (int(dims[k]) for k in ("Hk", "Hv", "dk", "dv"))
    x = _f64(x)
    w_in = _f64(w_in)
    rows, hidden = x.shape
    cqkv = 2 * Hk * dk + Hv * dv
    if w_in.shape != (cqkv + Hv * dv + 2 * Hv, hidden):
        raise ValueError("w_in must be [Cqkv + Hv*dv + 2*Hv][hidden]")
    out = {"qkv": np.zeros((rows, cqkv)), "z": np.zeros((rows, Hv * dv)),
           "b": np.zeros((rows, Hv)), "a": np.zeros((rows, Hv))}
    _load().oracle_in_proj(Hk, Hv, dk, dv, rows, hidden, _ptr(x), _ptr(w_in), _ptr(out["qkv"]),
                           _ptr(out["z"]), _ptr(out["b"]), _ptr(out["a"]))
    return out


def out_proj(o, w_out) -> np.ndarray:
    """y [rows][hidden] = o [rows][Hv*dv] w_out^T."""
    return linear(o, w_out)
