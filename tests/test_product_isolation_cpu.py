"""The product path stands apart from the oracle: the package and its CUDA
sources never import, include or name it, the package import does not load
it, and the two share no source file.  (The oracle is test infrastructure;
only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs use it.)"""

import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sink_short_window_sinkwin_b300")


def _sources(top, exts):
    for d, _, files in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_package_sources_do_not_reference_the_oracle():
    pat = re.compile(r"\b(import\s+oracle|from\s+oracle|oracle[/.])")
    for path in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        txt = open(path, encoding="utf-8").read()
        assert not pat.search(txt), f"{path} references the oracle"


def test_importing_the_package_does_not_load_the_oracle():
    code = ("import sys; import sink_short_window_sinkwin_b300 as m; "
            "bad = [k for k in sys.modules if k == 'oracle' or k.startswith('oracle.')]; "
            "print(bad); sys.exit(1 if bad else 0)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr


def test_oracle_does_not_use_the_library():
    pat = re.compile(r"sink_short_window_sinkwin_b300|libsinkwin|ctypes")
    for path in _sources(os.path.join(ROOT, "oracle"), (".py",)):
        assert not pat.search(open(path, encoding="utf-8").read()), f"{path} touches the library"


def test_missing_library_fails_loudly(tmp_path):
    """Without libsinkwin.so the binding refuses to load: there is no fallback."""
    import pytest
    from sink_short_window_sinkwin_b300 import _abi
    with pytest.raises(ImportError, match="missing"):
        _abi.load(str(tmp_path / "libsinkwin.so"))
