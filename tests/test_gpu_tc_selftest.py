"""The tcgen05 / TMEM / shared-memory-descriptor / cluster primitives the prefill kernels use,
checked in isolation: a 128 x N x K GEMM with bf16 operands (one pass) and with split-bf16
operands (hi*hi + hi*lo + lo*hi, three passes) against float64 products on the CPU, with dense
and padded (144-byte) B layouts and with the A operand copied into TMEM; the st.async exchange
among the CTAs of a cluster; and a bounded mbarrier wait that gives up."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_09_gb300 import build as gbuild
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libtcselftest.so")
    cmd = [gbuild.nvcc()] + gbuild.flags() + ["-shared", "-o", so,
                                              os.path.join(HERE, "csrc", "tc_selftest.cu")]
    subprocess.run(cmd, check=True)
    l = ctypes.CDLL(so)
    l.tc_gemm.restype = ctypes.c_int
    l.tc_gemm.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    l.tc_gemm_p.restype = ctypes.c_int
    l.tc_gemm_p.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    l.tc_gemm_ta.restype = ctypes.c_int
    l.tc_gemm_ta.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    l.tc_gemm_tast.restype = ctypes.c_int
    l.tc_gemm_tast.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    l.tc_gemm_mnb.restype = ctypes.c_int
    l.tc_gemm_mnb.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    l.tc_mma_cost.restype = ctypes.c_int
    l.tc_mma_cost.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    l.tc_cluster_xchg.restype = ctypes.c_int
    l.tc_cluster_xchg.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return l


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("N,K", [(64, 128), (128, 128), (192, 64), (256, 64), (16, 16)])
def test_tc_gemm(lib, N, K):
    rng = np.random.default_rng(N * 1000 + K)
    A = rng.standard_normal((128, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    # one pass: exactly the product of the bf16-rounded operands (f32 accumulation)
    D = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    assert lib.tc_gemm(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 1, err.data_ptr()) == 0
    assert int(err.item()) == 0
    ref1 = _bf16(A) @ _bf16(B).T
    np.testing.assert_allclose(D.cpu().numpy(), ref1, rtol=0, atol=2e-4 * np.sqrt(K))
    # three passes: close to the float32 operands' product
    D.zero_()
    assert lib.tc_gemm(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 3, err.data_ptr()) == 0
    assert int(err.item()) == 0
    e3 = np.max(np.abs(D.cpu().numpy() - ref)) / np.max(np.abs(ref))
    e1 = np.max(np.abs(ref1 - ref)) / np.max(np.abs(ref))
    assert e3 < 2e-5, e3
    assert e3 < e1 / 20


@pytest.mark.parametrize("N,K", [(32, 128), (32, 64), (64, 64)])
def test_tc_gemm_padded_b(lib, N, K):
    """B operand with its K-direction core matrices 144 bytes apart (a padded layout in which a
    warp stores 2-byte elements without bank conflicts)."""
    rng = np.random.default_rng(N * 7 + K)
    A = rng.standard_normal((128, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    D = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    assert lib.tc_gemm_p(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 3, 144, err.data_ptr()) == 0
    assert int(err.item()) == 0
    e3 = np.max(np.abs(D.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert e3 < 2e-5, e3


@pytest.mark.parametrize("N,K", [(32, 128), (32, 64), (64, 128)])
def test_tc_gemm_tmem_a(lib, N, K):
    """A operand copied into TMEM with tcgen05.cp and read from there by the MMAs."""
    rng = np.random.default_rng(N * 11 + K)
    A = rng.standard_normal((128, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    D = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    assert lib.tc_gemm_ta(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 1, err.data_ptr()) == 0
    assert int(err.item()) == 0
    ref1 = _bf16(A) @ _bf16(B).T
    np.testing.assert_allclose(D.cpu().numpy(), ref1, rtol=0, atol=2e-4 * np.sqrt(K))
    D.zero_()
    assert lib.tc_gemm_ta(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 3, err.data_ptr()) == 0
    assert int(err.item()) == 0
    e3 = np.max(np.abs(D.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert e3 < 2e-5, e3


@pytest.mark.parametrize("N,K", [(128, 128), (128, 64), (64, 64), (256, 64)])
def test_tc_gemm_tmem_a_from_registers(lib, N, K):
    """A operand written into TMEM from registers with tcgen05.st (bf16 pairs, element 2c in the
    low half of column c) and read from there by the MMAs: one pass equals the product of the
    bf16 operands, three passes are close to the float32 product."""
    rng = np.random.default_rng(N * 17 + K)
    A = rng.standard_normal((128, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    D = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    assert lib.tc_gemm_tast(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 1, err.data_ptr()) == 0
    assert int(err.item()) == 0
    ref1 = _bf16(A) @ _bf16(B).T
    np.testing.assert_allclose(D.cpu().numpy(), ref1, rtol=0, atol=2e-4 * np.sqrt(K))
    D.zero_()
    assert lib.tc_gemm_tast(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), N, K, 3, err.data_ptr()) == 0
    assert int(err.item()) == 0
    e3 = np.max(np.abs(D.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert e3 < 2e-5, e3


@pytest.mark.parametrize("N,K", [(128, 64), (64, 64), (128, 128), (256, 64)])
def test_tc_gemm_mn_major_b(lib, N, K):
    """B operand read MN-major out of a tile stored with k as its row index (the prefill reads
    K^T and V^T this way from its token-row tiles): one pass equals the product of the bf16
    operands, three passes are close to the float32 product."""
    rng = np.random.default_rng(N * 13 + K)
    A = rng.standard_normal((128, K)).astype(np.float32)
    Bt = rng.standard_normal((K, N)).astype(np.float32)
    dA, dBt = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = A.astype(np.float64) @ Bt.astype(np.float64)
    D = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    assert lib.tc_gemm_mnb(dA.data_ptr(), dBt.data_ptr(), D.data_ptr(), N, K, 1, err.data_ptr()) == 0
    assert int(err.item()) == 0
    ref1 = _bf16(A) @ _bf16(Bt)
    np.testing.assert_allclose(D.cpu().numpy(), ref1, rtol=0, atol=2e-4 * np.sqrt(K))
    D.zero_()
    assert lib.tc_gemm_mnb(dA.data_ptr(), dBt.data_ptr(), D.data_ptr(), N, K, 3, err.data_ptr()) == 0
    assert int(err.item()) == 0
    e3 = np.max(np.abs(D.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert e3 < 2e-5, e3


def test_mma_issue_cost(lib):
    """Cycles per MMA (M = 128, K = 16, bf16) over 24 back-to-back MMAs, A in shared memory or
    in TMEM, N = 64 / 128 / 192 / 256 (printed with -s; the prefill chain kernel keeps its A operands in
    TMEM because of this).  Checked: every run completes and the figures are sane."""
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = []
    for tmem_a in (0, 1):
        for N in (64, 128, 192, 256):
            spans = []
            for nmma in (8, 24):
                assert lib.tc_mma_cost(N, tmem_a, nmma, out.data_ptr(), err.data_ptr()) == 0
                assert int(err.item()) == 0
                spans.append(int(out.item()))
            per = (spans[1] - spans[0]) / 16.0   # the marginal cost of one more MMA
            rows.append(("tmem" if tmem_a else "smem", N, per))
            assert 10.0 < per < 2000.0, (tmem_a, N, per)
    for where, N, per in rows:
        print(f"A in {where}: N = {N:3d}: {per:6.1f} cycles per MMA")


def test_cluster_exchange(lib):
    """st.async exchange among the 4 CTAs of a cluster, double-buffered over rounds: every CTA
    sees the sum of the four ranks' values of each round."""
    ncl, rounds = 6, 9
    out = torch.zeros((4 * ncl, rounds, 64), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.tc_cluster_xchg(ncl, rounds, out.data_ptr(), err.data_ptr()) == 0
    assert int(err.item()) == 0
    t = np.arange(64)[None, :]
    c = np.arange(rounds)[:, None]
    want = (0 + 1000 + 2000 + 3000) + 4 * t + 4 * 0.25 * c
    got = out.cpu().numpy()
    for blk in range(4 * ncl):
        np.testing.assert_array_equal(got[blk], want.astype(np.float32))


def test_bounded_wait_gives_up_and_reports(lib):
    """A wait on an mbarrier phase that never completes returns after its limit with the
    timeout status; the GPU context stays usable (a GEMM runs right after)."""
    lib.tc_timeout_probe.restype = ctypes.c_int
    lib.tc_timeout_probe.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_void_p]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 2_000_000  # 2 ms
    assert lib.tc_timeout_probe(limit, status.data_ptr(), waited.data_ptr()) == 0
    assert int(status.item()) == 4
    assert limit <= int(waited.item()) < 1_000_000_000
    test_tc_gemm(lib, 64, 128)
