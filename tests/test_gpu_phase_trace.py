"""The phase-trace build (GEMM_F16_PHASE_TRACE) computes what the product build computes, and its
stamps are a consistent timeline: every CTA reaches its phases in order, and a launch is released
from its dependency wait only after the previous launch's last CTA has exited."""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,variant", [((64, 64, 64), -1), ((256, 256, 256), -1), ((300, 520, 136), -1),
                                           ((256, 512, 2048), 19), ((1000, 1000, 1088), 21)])
def test_phase_trace_matches_product_and_is_ordered(shape, variant):
    from dense_fp16_gemm_03_gb300 import phase_trace

    out = phase_trace.trace_shape(*shape, launches=12, traced_at=5, variant=variant)
    assert out["same_c"]
    assert out["phases_in_order"]
    assert len(out["launches"]) == 3
    names = phase_trace.PHASES if variant in (19, 21) else phase_trace.COMMON
    for row in out["launches"]:
        for name in names:
            assert name in row, name
    # the dependency wait of launch i + 1 returns after launch i's last exit stamp
    assert all(h > 0 for h in out["handover_us"]), out["handover_us"]
