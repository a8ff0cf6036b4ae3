"""The product path has no fallback: without the built libmhc every entry
point raises instead of computing anything another way (checked in a fresh
interpreter whose library path points at nothing)."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
import sys
sys.path.insert(0, sys.argv[1])
import hyper_connection_residual_mhc_gb300 as m
m.LIB_PATH = "/nonexistent/libmhc.so"
for call in (lambda: m.lib(), lambda: m.default_params(), lambda: m.mhc_pre_workspace_bytes(16)):
    try:
        call()
    except RuntimeError as e:
        assert "not built" in str(e), e
    else:
        raise SystemExit("an entry point ran without libmhc")
print("raised")
"""


def test_every_entry_raises_without_the_library():
    out = subprocess.run([sys.executable, "-c", PROBE, ROOT], capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == "raised"
