"""Parity of the "wgmma_gemm.cu" layout, D[M,N] = A[M,K] . B[K,N] with B
stored row-major [K, N] and an fp32 result, against the CPU oracle.

Integer-valued operands give exact fp32 sums in any order, so those cases
must match bit for bit; real-valued ones must meet
|d_gpu - d_ref| <= 1e-3 * sum|a*b| + ulp32(d_ref) element by element.
"""
import numpy as np
import pytest

from gpu_helpers import require_gpu, to_dev, torch

import oracle
from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _nn_variants():
    return [v for v in range(G.gemm_f16_variant_count()) if G.gemm_f16_variant_info(v)["layout"] == 1]


def run_nn(A, B_kn, variant=None, stream_k=0, use_ws=False):
    M, K = A.shape
    N = B_kn.shape[1]
    a, b = to_dev(A), to_dev(B_kn)
    d = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    if variant is None and not use_ws:
        G.gemm_f16_nn_f32(a, b, d)
    elif variant is None:
        p = G.gemm_f16_nn_f32_plan_ex(M, N, K, -1, 0, -1)
        ws = torch.empty(max(256, int(p.workspace_bytes)), dtype=torch.uint8, device="cuda")
        G.gemm_f16_nn_f32_ws(a, b, d, ws)
    else:
        p = G.gemm_f16_nn_f32_plan_ex(M, N, K, variant, 0, stream_k)
        G.gemm_f16_nt_run(p, a, b, d, G.workspace_for(p))
    st, code = G.gemm_f16_take_device_error()
    assert st == G.GEMM_OK, "device error word 0x%x" % code
    return d.cpu().numpy()


def check(D, A, B_kn, exact=False):
    ref, absum = oracle.gemm_nn_f32(A, B_kn)
    if exact:
        bad = np.argwhere(D != ref)
        assert bad.size == 0, "first mismatch %s: gpu %r oracle %r (%d)" % (
            tuple(bad[0]), D[tuple(bad[0])], ref[tuple(bad[0])], len(bad))
    rep = oracle.check_parity_f32(D, ref, absum, index_shape=ref.shape)
    assert rep.ok, repr(rep)


def test_day78_problem_256():
    """The page's own problem: 256^3, its LCG operands (A then B, B as [K, N]),
    fp32 D; its gate is |d - ref| / max(|ref|, 1) <= 1e-3, here bit-exact."""
    A, B_flat = inputs.lcg_eighths(256, 256, 256)
    B_kn = np.ascontiguousarray(B_flat).reshape(256, 256)
    D = run_nn(A, B_kn)
    ref, _ = oracle.gemm_nn_f32(A, B_kn)
    assert np.max(np.abs(D - ref) / np.maximum(np.abs(ref), 1.0)) <= 1e-3
    check(D, A, B_kn, exact=True)


@pytest.mark.parametrize("shape", [(1, 8, 8), (129, 264, 72), (128, 256, 64), (300, 520, 136), (640, 1032, 520),
                                   (1000, 1000, 1000), (96, 2056, 264)])
@pytest.mark.parametrize("stream_k", [0, 1])
def test_nn_ragged_exact(shape, stream_k):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "eighths", seed=11 * M + N + K)
    B_kn = np.ascontiguousarray(B.T)
    for v in _nn_variants():
        check(run_nn(A, B_kn, variant=v, stream_k=stream_k), A, B_kn, exact=True)


@pytest.mark.parametrize("shape", [(777, 1000, 1536), (1024, 1024, 4096), (128, 2048, 4096)])
def test_nn_real_valued_tolerance(shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "normal", seed=M + K)
    B_kn = np.ascontiguousarray(B.T)
    for v in _nn_variants():
        for sk in (0, 1):
            check(run_nn(A, B_kn, variant=v, stream_k=sk), A, B_kn)


def test_nn_identity_operands():
    rng = np.random.Generator(np.random.PCG64(4))
    B = rng.standard_normal((256, 200)).astype(np.float16)
    D = run_nn(inputs.identity(256), B)                 # A = I: D = B exactly
    assert np.array_equal(D, B.astype(np.float32))
    A = rng.standard_normal((136, 256)).astype(np.float16)
    D = run_nn(A, inputs.identity(256))                 # B = I: D = A exactly
    assert np.array_equal(D, A.astype(np.float32))


def test_nn_zero_k_and_guard_bands():
    a = torch.zeros((40, 0), dtype=torch.float16, device="cuda")
    b = torch.zeros((0, 24), dtype=torch.float16, device="cuda")
    d = torch.full((40, 24), 7.0, dtype=torch.float32, device="cuda")
    G.gemm_f16_nn_f32(a, b, d)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d).item() == 0
    M, N, K = 300, 520, 136
    A, B = inputs.make_operands(M, N, K, "eighths", seed=2)
    B_kn = np.ascontiguousarray(B.T)
    guard = 2048
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.float32, device="cuda")
    d = buf[guard:guard + M * N].view(M, N)
    G.gemm_f16_nn_f32(to_dev(A), to_dev(B_kn), d)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + M * N:]).all()
    check(d.cpu().numpy(), A, B_kn, exact=True)


@pytest.mark.parametrize("use_ws", [False, True])
def test_nn_square_4096_full(use_ws):
    A, B = inputs.workload_operands(inputs.BY_NAME["square_4096"])
    B_kn = np.ascontiguousarray(B.T)
    check(run_nn(A, B_kn, use_ws=use_ws), A, B_kn)
