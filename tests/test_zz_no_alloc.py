"""The allocation-free entry point, gemm_f16_nt_noalloc.

It exists for callers that may not allocate device memory (code inside a
host that owns every allocation through its own pool, paths that must not
call cudaMalloc/cudaFree because those can synchronize the device).  It runs
plans that need scratch (a stream-K tail, split K) with that scratch taken
from an array built into the library, so its results must agree with the
workspace entry point
(gemm_f16_nt_ws with a caller-allocated workspace) within the parity bound
the other tests use, on consecutive calls that reuse that one array -- and,
like every other entry point, with the CPU oracle.

This file is collected last on purpose: a failure here leaves every other
test already run.
"""
import numpy as np
import pytest

from gpu_helpers import from_dev_bits, require_gpu, to_dev, torch

import oracle
from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu


def _within_bound(got_bits, ref_bits, absum):
    rep = oracle.check_parity(got_bits, ref_bits, absum, index_shape=ref_bits.shape)
    assert rep.ok, repr(rep)


# 100 x 20000 x 4104: one strip of B rows a little past one wave of tiles, a stream-K tail;
# 1024 x 2048 x 4096: few tiles, split K
@pytest.mark.parametrize("shape,dist", [((100, 20000, 4104), "eighths"), ((1024, 2048, 4096), "normal")])
def test_noalloc_matches_workspace_entry_point_twice(shape, dist):
    require_gpu()
    M, N, K = shape
    need = G.gemm_f16_nt_workspace_size(M, N, K)
    assert 0 < need <= G.STATIC_SCRATCH_BYTES     # a plan with scratch: the built-in array serves it
    A, B = inputs.make_operands(M, N, K, dist, seed=M + N)
    a, b = to_dev(A), to_dev(B)

    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    c_ws = torch.empty((M, N), dtype=torch.float16, device="cuda")
    G.gemm_f16_nt_ws(a, b, c_ws, ws)
    ws_bits = from_dev_bits(c_ws)
    oracle_bits, absum = oracle.gemm_nt(A, B)

    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        G.gemm_f16_nt_noalloc(a, b, c)
        st, code = G.gemm_f16_take_device_error()
        assert st == G.GEMM_OK, "call %d: device error word 0x%x" % (call, code)
        got_bits = from_dev_bits(c)
        _within_bound(got_bits, ws_bits, absum)       # against the workspace entry point
        _within_bound(got_bits, oracle_bits, absum)   # against the oracle
        if dist == "eighths":              # integer-valued sums are exact in any order
            assert np.array_equal(got_bits, ws_bits)
            assert np.array_equal(got_bits, oracle_bits)
