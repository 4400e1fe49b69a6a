"""The oracle and the CUDA path share no code and neither imports the other:
the product package (Python binding and CUDA sources) never imports, includes
or loads the oracle, and the oracle never reaches into the package; the one
module both sides use, synth.py, only makes inputs."""
import re
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent
PKG = ROOT / "volumetric_ultrasound_delay_gb300"
ORACLE = ROOT / "oracle"


def _sources(folder, patterns):
    for pattern in patterns:
        for path in folder.rglob(pattern):
            if "_lib" in path.parts or "_build" in path.parts or "__pycache__" in path.parts:
                continue
            yield path


def test_product_never_imports_the_oracle():
    pattern = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|#\s*include\s*[<\"].*oracle)", re.M)
    for path in _sources(PKG, ("*.py", "*.cu", "*.cuh", "*.h")):
        assert not pattern.search(path.read_text()), path


def test_oracle_never_imports_the_product():
    pattern = re.compile(r"^\s*(import\s+volumetric_ultrasound_delay_gb300|from\s+volumetric_ultrasound_delay_gb300"
                         r"|#\s*include\s*[<\"].*(das|csrc))", re.M)
    for path in _sources(ORACLE, ("*.py", "*.c", "*.h")):
        assert not pattern.search(path.read_text()), path


def test_importing_the_package_does_not_load_the_oracle():
    code = ("import sys; sys.path.insert(0, %r); import volumetric_ultrasound_delay_gb300 as p; "
            "from volumetric_ultrasound_delay_gb300 import das, synth; "
            "print('oracle' in sys.modules)" % str(ROOT))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120, cwd="/")
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "False"


def test_synth_holds_no_beamforming_arithmetic():
    """The input module does not interpolate a record (no floor of a sample
    index) and does not import the library; its echo synthesis is a forward
    model of its own."""
    text = (PKG / "synth.py").read_text()
    assert "floor(" not in text
    assert "das" not in re.findall(r"^\s*(?:from|import)\s+(\S+)", text, re.M)
