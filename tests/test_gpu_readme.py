"""The Python usage example in README.md runs as written."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example():
    with open(os.path.join(ROOT, "README.md")) as f:
        blocks = re.findall(r"```python\n(.*?)```", f.read(), flags=re.S)
    assert blocks
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    y = scope["y"]
    torch.cuda.synchronize()
    assert tuple(y.shape) == (32, 64 * 64 * 64) and bool(torch.isfinite(y).all())
