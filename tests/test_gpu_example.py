"""The usage example of the Python binding (volumetric_ultrasound_delay_gb300/example.py)
runs as written."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)


def test_python_usage_example():
    from volumetric_ultrasound_delay_gb300.example import example
    y = example()
    torch.cuda.synchronize()
    assert tuple(y.shape) == (32, 64 * 64 * 64) and bool(torch.isfinite(y).all())
