"""Parity at the size extremes, through the automatic plan: a C of 2^32
elements (8 GiB; element offsets past 32 bits), 2^20 rows of one 8-column
strip (4096 tile rows), and K = 2^20 on one output tile (16384 K blocks, so
split-K cuts that tile's K into parts over every cluster).  Operands in
{-8..8}/8 make every product a multiple of 2^-6, so fp32 sums are exact while
their partial sums stay below 2^18 in magnitude: always for K = 64, and for
K = 2^20 because these zero-mean draws keep them in the hundreds.  So the
sampled entries must match the oracle bit for bit; the samples always include
the first and last rows and columns.  Entries are gathered on the device, C
never leaves it.
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


def _sample(M, N, n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = np.concatenate([rng.integers(0, M, size=n), [0, 0, M - 1, M - 1], np.full(64, M - 1)])
    cols = np.concatenate([rng.integers(0, N, size=n), [0, N - 1, 0, N - 1], np.arange(N - 64, N) % N])
    return rows, cols


def _check_sampled(M, N, K, n_samples, seed, ws=False):
    A, B = inputs.make_operands(M, N, K, "eighths", seed=seed)
    a, b = to_dev(A), to_dev(B)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    if ws:
        need = G.gemm_f16_nt_workspace_size(M, N, K)
        w = torch.empty(max(256, need), dtype=torch.uint8, device="cuda")
        G.gemm_f16_nt_ws(a, b, c, w)
    else:
        G.gemm_f16_nt(a, b, c)
    st, code = G.gemm_f16_take_device_error()
    assert st == G.GEMM_OK, "device error word 0x%x" % code
    rows, cols = _sample(M, N, n_samples, seed)
    r_d = torch.from_numpy(rows).cuda()
    c_d = torch.from_numpy(cols).cuda()
    got = c[r_d, c_d].cpu().view(torch.int16).numpy().view(np.uint16)
    ref, _ = oracle.gemm_nt_entries(A, B, rows, cols)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, "entry (%d, %d): gpu 0x%04x oracle 0x%04x (%d of %d differ)" % (
        rows[bad[0]], cols[bad[0]], got[bad[0]], ref[bad[0]], bad.size, got.size)
    del c
    torch.cuda.empty_cache()


def test_c_of_2_pow_32_elements():
    _check_sampled(65536, 65536, 64, 20000, seed=41)


def test_one_strip_of_2_pow_20_rows():
    _check_sampled(1 << 20, 8, 64, 20000, seed=42)


@pytest.mark.parametrize("ws", [False, True])
def test_k_of_2_pow_20_on_one_tile(ws):
    p = G.gemm_f16_nt_plan(256, 256, 1 << 20)
    if ws:
        assert p.split_k > 1                    # the one tile's K is split over all clusters
    _check_sampled(256, 256, 1 << 20, 300, seed=43, ws=ws)
