"""The product path has no fallback (CPU only): without the CUDA library every
call raises, and importing and loading the package never loads the oracle."""
import os
import subprocess
import sys

import pytest

import io_aware_attention_gb300 as fa
from io_aware_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        fa.library()
    with pytest.raises(RuntimeError, match="missing"):
        fa.version()
    with pytest.raises(RuntimeError, match="missing"):
        fa.set_wait_limit_ns(1)


def test_package_does_not_load_the_oracle():
    code = ("import os, sys\n"
            "import io_aware_attention_gb300 as fa\n"
            "from io_aware_attention_gb300 import workloads\n"
            "if os.path.exists(fa.library_path()):\n"
            "    fa.library()\n"
            "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "[]"
