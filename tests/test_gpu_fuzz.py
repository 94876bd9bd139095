"""Seeded random shapes through every way a plan can be made, bit for bit.

Operands in {-8..8}/8 make every product a multiple of 2^-6 and every partial
sum exact in fp32 (|sum| <= K <= 2^18 units), whatever the order, split or
tile; so every configuration must reproduce the oracle's bits exactly.  Each
seeded case draws M from 1, N and K as multiples of 8 from 8 (the only shape
rule), then runs the automatic plans of both entry points, the allocation-free
entry point and a few forced plans: a random variant of the fp16 layout, a
random raster width and, where the variant has them, a forced stream-K tail
or split K.  The fp32-output layout (B stored [K, N]) gets its own cases.
"""
import numpy as np
import pytest

from gpu_helpers import assert_parity, from_dev_bits, require_gpu, to_dev, torch

import oracle
from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = 160


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _shape(rng):
    kind = rng.integers(0, 4)
    if kind == 0:                                    # tiny: single partial tiles, K below one block
        return int(rng.integers(1, 80)), 8 * int(rng.integers(1, 20)), 8 * int(rng.integers(1, 12))
    if kind == 1:                                    # one strip of rows (the few-rows plans)
        return int(rng.integers(1, 129)), 8 * int(rng.integers(16, 600)), 8 * int(rng.integers(8, 400))
    if kind == 2:                                    # long K over few tiles (split K, stream-K)
        return int(rng.integers(100, 600)), 8 * int(rng.integers(16, 80)), 8 * int(rng.integers(400, 1500))
    return int(rng.integers(200, 1800)), 8 * int(rng.integers(30, 220)), 8 * int(rng.integers(8, 160))


def _run(plan, a, b, M, N, ws_fill=None):
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    ws = None
    if plan.workspace_bytes:
        ws = torch.full((int(plan.workspace_bytes),), 0xA5 if ws_fill is None else ws_fill, dtype=torch.uint8,
                        device="cuda")
    G.gemm_f16_nt_run(plan, a, b, c, ws)
    st, code = G.gemm_f16_take_device_error()
    assert st == G.GEMM_OK, "device error word 0x%x for %r" % (code, plan)
    return from_dev_bits(c)


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_nt_exact(case):
    rng = np.random.Generator(np.random.PCG64(90000 + case))
    M, N, K = _shape(rng)
    A, B = inputs.make_operands(M, N, K, "eighths", seed=int(rng.integers(1 << 30)))
    ref, _ = oracle.gemm_nt(A, B)
    a, b = to_dev(A), to_dev(B)

    def check(bits, what):
        bad = np.argwhere(bits != ref)
        assert bad.size == 0, "%s on %dx%dx%d: first mismatch at %s (%d differ)" % (
            what, M, N, K, tuple(bad[0]), len(bad))

    # the automatic plans of the three device entry points
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    G.gemm_f16_nt(a, b, c)
    check(from_dev_bits(c), "gemm_f16_nt")
    ws = torch.empty(max(256, G.gemm_f16_nt_workspace_size(M, N, K)), dtype=torch.uint8, device="cuda")
    G.gemm_f16_nt_ws(a, b, c, ws)
    check(from_dev_bits(c), "gemm_f16_nt_ws")
    if G.gemm_f16_nt_workspace_size(M, N, K) <= G.STATIC_SCRATCH_BYTES:
        G.gemm_f16_nt_noalloc(a, b, c)
        check(from_dev_bits(c), "gemm_f16_nt_noalloc")
    assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK

    # forced plans: random variants, raster widths, and each variant's splits
    nt = [v for v in range(G.gemm_f16_variant_count()) if G.gemm_f16_variant_info(v)["layout"] == 0]
    for v in rng.choice(nt, size=3, replace=False):
        v = int(v)
        width = int(rng.integers(1, 9))
        for stream_k in (0, 1, 2):
            try:
                plan = G.gemm_f16_nt_plan_ex(M, N, K, v, width, stream_k)
            except G.GemmError as e:               # no split K (or, K-split clusters, no tail) for this variant
                k_split = G.gemm_f16_variant_info(v)["k_split"] > 1
                assert e.status == G.GEMM_ERR_INVALID_ARG and (stream_k == 2 or (stream_k == 1 and k_split))
                continue
            check(_run(plan, a, b, M, N), "variant %d raster %d stream_k %d (plan %r)" % (v, width, stream_k, plan))


@pytest.mark.parametrize("case", range(40))
def test_fuzz_nn_f32_exact(case):
    """D = A . B with B stored [K, N] and an fp32 result: integer-valued sums are exact in fp32 too."""
    rng = np.random.Generator(np.random.PCG64(91000 + case))
    M, N, K = _shape(rng)
    A, B = inputs.make_operands(M, N, K, "eighths", seed=int(rng.integers(1 << 30)))
    B_kn = np.ascontiguousarray(B.T)
    ref, _ = oracle.gemm_nn_f32(A, B_kn)
    a, b = to_dev(A), to_dev(B_kn)
    d = G.gemm_f16_nn_f32(a, b)
    assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
    got = d.cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, "%dx%dx%d: first mismatch at %s" % (M, N, K, tuple(bad[0]))
