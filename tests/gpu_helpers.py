"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on numpy operands and compare with the CPU oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from dense_fp16_gemm_03_gb300 import gemm as G  # noqa: E402


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.lib()


def num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.float16).to("cuda")


def from_dev_bits(c):
    return c.cpu().view(torch.int16).numpy().view(np.uint16)


def run_gpu(A, B, variant=None, raster_width=0, stream=None, stream_k=0, use_ws_entry=False):
    """C bits (uint16 [M,N]) from the CUDA path.

    variant None and raster 0 with stream_k 0: gemm_f16_nt (automatic, no workspace);
    use_ws_entry: gemm_f16_nt_ws with the workspace it asks for;
    otherwise an explicit plan (stream_k 1 forces a stream-K tail) through gemm_f16_nt_run."""
    M, K = A.shape
    N = B.shape[0]
    a, b = to_dev(A), to_dev(B)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    if use_ws_entry:
        ws = torch.empty(max(1, G.gemm_f16_nt_workspace_size(M, N, K)), dtype=torch.uint8, device="cuda")
        G.gemm_f16_nt_ws(a, b, c, ws, stream=stream)
    elif variant is None and raster_width == 0 and stream_k == 0:
        G.gemm_f16_nt(a, b, c, stream=stream)
    else:
        plan = G.gemm_f16_nt_plan_ex(M, N, K, -1 if variant is None else variant, raster_width, stream_k)
        ws = G.workspace_for(plan)
        G.gemm_f16_nt_run(plan, a, b, c, ws, stream=stream)
    st, code = G.gemm_f16_take_device_error(stream)
    assert st == G.GEMM_OK, "device error word 0x%x" % code
    return from_dev_bits(c)


def assert_parity(c_bits, A, B, exact=False):
    ref, absum = oracle.gemm_nt(A, B)
    if exact:
        bad = np.argwhere(c_bits != ref)
        assert bad.size == 0, "first mismatch at %s: gpu 0x%04x oracle 0x%04x (%d mismatches)" % (
            tuple(bad[0]), c_bits[tuple(bad[0])], ref[tuple(bad[0])], len(bad))
    rep = oracle.check_parity(c_bits, ref, absum, index_shape=ref.shape)
    assert rep.ok, repr(rep)
    return rep
