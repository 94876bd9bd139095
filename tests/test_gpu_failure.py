"""Failure detection on the GPU without a fault: a stage fill that never
happens makes the kernel's bounded waits expire; the kernel records the
failure in its device error word, frees its tensor memory and returns, and
the host reads GEMM_ERR_TIMEOUT.  The context stays usable: the next product
is correct and the error word is clear again."""
import numpy as np
import pytest

from gpu_helpers import assert_parity, num_sms, require_gpu, run_gpu, to_dev, torch

from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu

WAIT_LIMIT_CYCLES = 1 << 24   # about 10 ms at GB300 clocks


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("variant,skip", [(0, 3), (2, 3), (4, 3), (11, 3), (13, 3), (15, 3), (16, 3), (17, 3),
                                          (19, 1), (20, 3), (21, 3)])
def test_starved_wait_reports_timeout_and_recovers(variant, skip):
    """The skipped fill starves the first CTA's MMA (or, for the clusters that share a tile by
    multicast, every MMA that waits for that CTA's slice; for a K-split cluster, the partners wait
    for its partial slices in vain).  Before the CTAs exit, the owners of the ring's barriers wait
    for every load still in flight, and a K-split CTA for partner slices it never waited for (the
    abort drain), so no copy lands after teardown; the error word names the first wait that gave
    up.  `skip` is a fill the first CTA does issue (a K-split CTA walks only its share of K)."""
    M, N, K = 256, 512, 640
    A, B = inputs.make_operands(M, N, K, "eighths", seed=77)
    a, b = to_dev(A), to_dev(B)
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    plan = G.gemm_f16_nt_plan_ex(M, N, K, variant, 0, 0)
    assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
    st = G.gemm_f16_nt_run_stall_test(plan, a, b, c, skip, WAIT_LIMIT_CYCLES)
    assert st == G.GEMM_OK                       # the launch itself is fine
    st, code = G.gemm_f16_take_device_error()
    assert st == G.GEMM_ERR_TIMEOUT
    assert (code & 0xFF) in (1, 2, 3, 4, 8, 9)   # one of the pipeline (or partner-slice) waits gave up
    # the error word is cleared by reading it, and the context still works
    assert G.gemm_f16_take_device_error() == (G.GEMM_OK, 0)
    assert_parity(run_gpu(A, B, variant=variant), A, B, exact=True)
