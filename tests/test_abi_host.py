"""CPU-side checks of the C ABI: the library loads, exports every symbol include/gdn.h declares,
and every host-side argument check returns its documented code without touching a GPU."""
import ctypes
import os
import re

import pytest

from gated_deltanet_linear_09_gb300 import build as gbuild
from gated_deltanet_linear_09_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load()


def _declared_functions():
    txt = open(os.path.join(ROOT, "include", "gdn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(gdn_\w+)\s*\(", txt, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 7
    assert set(declared) == set(gdn.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name
    # and they are exported with C linkage from the shared object itself
    handle = ctypes.CDLL(gdn.lib_path())
    for name in declared:
        getattr(handle, name)


def D(**kw):
    base = dict(Hk=16, Hv=32, dk=128, dv=128, K=4)
    base.update(kw)
    return gdn.make_dims(base["Hk"], base["Hv"], base["dk"], base["dv"], base["K"])


def test_slot_and_workspace_bytes(lib):
    d = D(Hv=48)
    # 48 V-heads x 128 x 128 f32 + 3 rows x 10240 channels bf16
    assert gdn.gdn_state_slot_bytes(d, gdn.GDN_BF16) == 48 * 128 * 128 * 4 + 3 * 10240 * 2
    assert gdn.gdn_state_slot_bytes(d, gdn.GDN_F32) == 48 * 128 * 128 * 4 + 3 * 10240 * 4
    assert gdn.gdn_state_slot_bytes(D(Hv=33), gdn.GDN_BF16) == 0       # not divisible
    assert gdn.gdn_state_slot_bytes(D(dk=96), gdn.GDN_BF16) == 0       # unsupported
    w1 = gdn.gdn_prefill_workspace_bytes(D(), 1, 4096)
    w2 = gdn.gdn_prefill_workspace_bytes(D(), 1, 8192)
    assert 0 < w1 < w2
    assert w1 % 256 == 0
    assert gdn.gdn_prefill_workspace_bytes(D(), -1, 10) == 0


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9):
        assert gdn.gdn_status_string(code)
    assert "unknown" in gdn.gdn_status_string(12345)


def _call_decode(lib, dims, B=1, aligned=True, null_w=False):
    # host pointers that are never dereferenced: every case below fails the host checks first
    fake = 0x10000 if aligned else 0x10008 + 2
    w = gdn.gdn_weights(0 if null_w else 0x20000, 0x20000, 0x20000, 0x20000, gdn.GDN_BF16)
    p = gdn.gdn_pool(0x30000, 0x30000, 4, None)
    return lib.gdn_decode_step(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(p), 0x40000, B,
                               fake, fake, fake, fake, fake, None)


def test_decode_host_checks(lib):
    assert _call_decode(lib, D(Hv=33)) == -3          # fail closed on head divisibility
    assert _call_decode(lib, D(dk=96)) == -2
    assert _call_decode(lib, D(K=3)) == -2
    assert _call_decode(lib, D(Hk=0)) == -1
    assert _call_decode(lib, D(), B=-1) == -1
    assert _call_decode(lib, D(), B=70000) == -9
    assert _call_decode(lib, D(), B=0) == 0           # empty batch: no-op
    assert _call_decode(lib, D(), null_w=True) == -1
    assert _call_decode(lib, D(), aligned=False) == -7


def test_decode_multi_host_checks(lib):
    d = D()
    w = gdn.gdn_weights(0x20000, 0x20000, 0x20000, 0x20000, gdn.GDN_BF16)
    p = gdn.gdn_pool(0x30000, 0x30000, 4, None)

    def call(B, T, fake=0x10000):
        return lib.gdn_decode_multi(ctypes.byref(d), ctypes.byref(w), ctypes.byref(p), 0x40000, B,
                                    T, fake, fake, fake, fake, fake, None)
    assert call(1, 0) == -1                           # T outside [1, GDN_MAX_DECODE_TOKENS]
    assert call(1, gdn.GDN_MAX_DECODE_TOKENS + 1) == -1
    assert call(-1, 2) == -1
    assert call(70000, 2) == -9
    assert call(0, 2) == 0                            # empty batch: no-op
    assert call(1, 2, fake=0x10008 + 2) == -7


def test_decode_graphs_host_checks(lib):
    d = D()
    w = gdn.gdn_weights(0x20000, 0x20000, 0x20000, 0x20000, gdn.GDN_BF16)
    p = gdn.gdn_pool(0x30000, 0x30000, 4, None)
    h = ctypes.c_void_p(0x1234)

    def create(buckets, dims=d):
        arr = (ctypes.c_int32 * max(1, len(buckets)))(*buckets)
        return lib.gdn_decode_graphs_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(p),
                                            arr, len(buckets), ctypes.byref(h))
    # all rejected before any allocation or CUDA call, with *out cleared
    assert create([]) == -1 and h.value is None
    assert create([4, 2]) == -1
    assert create([1, 1]) == -1
    assert create([0, 4]) == -1
    assert create(list(range(1, gdn.GDN_MAX_GRAPH_BUCKETS + 2))) == -1
    assert create([1, 70000]) == -9
    assert create([1, 2], dims=D(Hv=33)) == -3
    assert lib.gdn_decode_graphs_launch(None, 1, None) == -1
    lib.gdn_decode_graphs_destroy(None)                # no-op


def test_projection_host_checks(lib):
    """gdn_linear_bf16 / gdn_in_proj / gdn_out_proj: every bad argument is refused before any
    CUDA call (the fake addresses are never dereferenced); M = 0 is a no-op."""
    X, W, Y = 0x10000, 0x20000, 0x30000

    def route(starts=(0,), lds=(64,), dsts=(Y,)):
        return gdn.make_route(list(zip(starts, lds, dsts)))

    def lin(M=4, N=64, K=128, r=None, ks=0, x=X, w=W):
        r = route() if r is None else r
        return lib.gdn_linear_bf16(x, w, M, N, K, ctypes.byref(r), ks, None, None)
    assert lin(x=0) == -1
    assert lin(N=0) == -1
    assert lin(M=-1) == -1
    assert lin(K=100) == -2                               # K not a multiple of 64
    assert lin(M=65535 * 64 + 1) == -9
    assert lin(x=X + 8) == -7                             # 16-byte alignment of x and w
    assert lin(r=route((), (), ())) == -1                  # no segment
    assert lin(r=route((1,))) == -1                        # start[0] != 0
    assert lin(N=64, r=route((0, 32, 32), (32, 32, 32), (Y, Y, Y))) == -1   # empty segment
    assert lin(N=64, r=route((0, 70), (70, 70), (Y, Y))) == -1              # start beyond N
    assert lin(r=route((0,), (63,))) == -1                 # ld below the segment's width
    assert lin(r=route(dsts=(Y + 1,))) == -7               # bf16 destination alignment
    assert lin(ks=9) == -1 and lin(ks=-1) == -1
    assert lin(K=128, ks=3) == -1                         # more parts than the 2 chunks of K / 64
    assert lin(K=128, ks=4) == -1                         # every part takes at least one chunk
    assert lin(M=0, ks=5, x=0) == 0                       # empty: nothing read or launched
    d = D()
    assert lib.gdn_in_proj(ctypes.byref(D(Hv=33)), X, W, 4, 256, Y, Y, Y, Y, None, None) == -3
    assert lib.gdn_in_proj(ctypes.byref(d), X, W, 4, 100, Y, Y, Y, Y, None, None) == -2
    assert lib.gdn_in_proj(ctypes.byref(d), X, W, 4, 256, Y, None, Y, Y, None, None) == -1
    assert lib.gdn_in_proj(ctypes.byref(d), X, W, 0, 256, Y, Y, Y, Y, None, None) == 0
    assert lib.gdn_out_proj(ctypes.byref(d), X, W, 4, 256, None, None, None) == -1
    assert lib.gdn_out_proj(ctypes.byref(d), X + 4, W, 4, 256, Y, None, None) == -7
    assert lib.gdn_out_proj(ctypes.byref(d), X, W, 0, 256, Y, None, None) == 0
    assert lib.gdn_proj_packed_bytes(300, 192) == 3 * 128 * 192 * 2
    assert lib.gdn_proj_packed_bytes(300, 100) == 0 and lib.gdn_proj_packed_bytes(0, 64) == 0
    assert lib.gdn_proj_pack(W, 300, 192, Y, 3 * 128 * 192 * 2 - 1, None) == -5
    assert lib.gdn_proj_pack(W, 300, 100, Y, 1 << 20, None) == -2
    assert lib.gdn_proj_pack(W + 8, 300, 192, Y, 1 << 20, None) == -7
    assert lib.gdn_proj_pack(None, 300, 192, Y, 1 << 20, None) == -1


def test_prefill_and_compact_host_checks(lib):
    d = D()
    w = gdn.gdn_weights(0x20000, 0x20000, 0x20000, 0x20000, gdn.GDN_BF16)
    p = gdn.gdn_pool(0x30000, 0x30000, 4, None)
    need = lib.gdn_prefill_workspace_bytes(ctypes.byref(d), 2, 100)
    # head dims 128 run in windows of whole chunks: the smallest workspace is one chunk's records
    # (the size quoted for one token), a byte less is refused
    least = lib.gdn_prefill_workspace_bytes(ctypes.byref(d), 1, 1)
    assert 0 < least < need and least == lib.gdn_prefill_workspace_bytes(ctypes.byref(d), 1, 63)
    f = 0x10000
    rc = lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(w), ctypes.byref(p), f, f, None, 2,
                                 100, f, f, f, f, f, 0x50000, least - 1, None)
    assert rc == -5
    # head dims 64 take the same path (one chunk's records at least)
    d64 = D(dk=64, dv=64)
    least64 = lib.gdn_prefill_workspace_bytes(ctypes.byref(d64), 1, 1)
    rc = lib.gdn_prefill_chunked(ctypes.byref(d64), ctypes.byref(w), ctypes.byref(p), f, f, None, 2,
                                 100, f, f, f, f, f, 0x50000, least64 - 1, None)
    assert rc == -5
    # more than four V-heads per K-head take the CUDA-core path, which needs the full size
    d8 = D(Hk=1, Hv=8)
    need8 = lib.gdn_prefill_workspace_bytes(ctypes.byref(d8), 2, 100)
    rc = lib.gdn_prefill_chunked(ctypes.byref(d8), ctypes.byref(w), ctypes.byref(p), f, f, None, 2,
                                 100, f, f, f, f, f, 0x50000, need8 - 1, None)
    assert rc == -5
    rc = lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(w), ctypes.byref(p), f, f, None, 2,
                                 100, f, f, f, f, f, 0x50000 + 16, need, None)
    assert rc == -7                                   # workspace must be 256-byte aligned
    rc = lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(w), ctypes.byref(p), f, f, None, 0,
                                 0, None, None, None, None, None, None, 0, None)
    assert rc == 0
    assert lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(w), ctypes.byref(p), f, f, None,
                                   0, 5, f, f, f, f, f, None, 0, None) == -1

    def compact(src, dst, slots=4):
        pp = gdn.gdn_pool(0x30000, 0x30000, slots, None)
        s = (ctypes.c_int32 * len(src))(*src)
        t = (ctypes.c_int32 * len(dst))(*dst)
        return lib.gdn_state_compact(ctypes.byref(d), gdn.GDN_BF16, ctypes.byref(pp), s, t,
                                     len(src), None)
    assert compact([0, 1], [1, 1]) == -6              # duplicate destination
    assert compact([0, 4], [1, 2]) == -4              # source out of range
    assert compact([0, 1], [1, -1]) == -4
    assert compact([], []) == 0
    big = list(range(2049))
    assert compact(big, big, slots=4096) == -9


def test_product_path_has_no_oracle_or_fallback():
    """The library and its binding never reach the CPU oracle."""
    pkg = os.path.join(ROOT, "gated_deltanet_linear_09_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), fn
                assert "liboracle" not in src and "gdn_oracle" not in src, fn


def test_header_is_c_and_links(lib, tmp_path):
    """A C99 program compiled against include/gdn.h (gcc, not nvcc) links with libgdn.so and
    runs the host-side entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    cuda_inc = None
    for cand in ("/usr/local/cuda/include", "/usr/local/cuda/targets/x86_64-linux/include",
                 "/usr/local/cuda/targets/sbsa-linux/include"):
        if os.path.exists(os.path.join(cand, "cuda_runtime_api.h")):
            cuda_inc = cand
            break
    if cuda_inc is None:
        pytest.skip("CUDA headers not found")
    libpath = gdn.lib_path()
    exe = tmp_path / "abi_c_check"
    src = os.path.join(ROOT, "tests", "csrc", "abi_c_check.c")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, src, "-o", str(exe), libpath,
                    "-Wl,-rpath," + os.path.dirname(libpath)], check=True)
    env = dict(os.environ)
    res = subprocess.run([str(exe)], capture_output=True, text=True, env=env)
    assert res.returncode == 0, (res.returncode, res.stdout, res.stderr)
    assert res.stdout.startswith("ok")
