"""The Python binding passes only addresses to the C ABI, so it checks the
shape, dtype, layout and device of every tensor it is given -- outputs
included -- before a call: a too-small output must be refused, not written
past its end.  No GPU is needed: the checks run before the library is
called (CPU tensors stand in where the check is about the device)."""
import pytest

torch = pytest.importorskip("torch")

from dense_fp16_gemm_03_gb300 import gemm as G  # noqa: E402


def test_check_matrix_rejects_wrong_shape_dtype_layout_device():
    t = torch.zeros((4, 8), dtype=torch.float16)
    with pytest.raises(ValueError):
        G._check_matrix(t, 4, 8, "float16", "c")               # host tensor where a device one is needed
    with pytest.raises(ValueError):
        G._check_matrix(torch.zeros((4, 8), dtype=torch.float32), 4, 8, "float16", "c")
    with pytest.raises(ValueError):
        G._check_matrix(torch.zeros((8, 4), dtype=torch.float16).t(), 4, 8, "float16", "c")   # not contiguous
    with pytest.raises(ValueError):
        G._check_matrix(torch.zeros((4, 7), dtype=torch.float16), 4, 8, "float16", "c")
    G._check_matrix(None, 4, 8, "float16", "c")                 # raw addresses and absent buffers pass through
    G._check_matrix(1 << 20, 4, 8, "float16", "c")


def test_host_entry_point_checks_host_tensors():
    a = torch.zeros((16, 8), dtype=torch.float16)
    b = torch.zeros((24, 8), dtype=torch.float16)
    c_small = torch.zeros((16, 23), dtype=torch.float16)
    with pytest.raises(ValueError):
        G.gemm_f16_nt_host(a, b, c_small, 1 << 20, 1 << 21, 1 << 22)
    with pytest.raises(ValueError):
        G.gemm_f16_nt_host(a, b.float(), torch.zeros((16, 24), dtype=torch.float16), 1 << 20, 1 << 21, 1 << 22)


def test_run_checks_operands_against_the_plan():
    p = G.gemm_f16_nt_plan_for(64, 128, 64, 152)
    with pytest.raises(ValueError):
        G.gemm_f16_nt_run(p, torch.zeros((64, 64), dtype=torch.float16), 1 << 20, 1 << 21)   # a on the host
    with pytest.raises(ValueError):
        G.gemm_f16_nt_run(p, 1 << 20, 1 << 21, torch.zeros((64, 127), dtype=torch.float16))
