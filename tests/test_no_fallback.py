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


def test_cpu_tensors_are_refused():
    # host tensors are never computed on: every entry point refuses them
    # before reaching the library
    import pytest
    import torch
    import hyper_connection_residual_mhc_gb300 as m
    rows = 4
    R = torch.zeros((rows, 4, 5120), dtype=torch.bfloat16)
    y = torch.zeros((rows, 5120), dtype=torch.bfloat16)
    fn = torch.zeros((24, 20480), dtype=torch.float32)
    sc, bs = torch.zeros(3), torch.zeros(24)
    w = torch.zeros(5120, dtype=torch.bfloat16)
    post, comb = torch.zeros((rows, 4)), torch.zeros((rows, 4, 4))
    calls = [
        lambda: m.mhc_pre(R, fn, sc, bs, w),
        lambda: m.mhc_post(R, y, post, comb),
        lambda: m.mhc_fused_post_pre(R, y, post, comb, fn, sc, bs, w),
        lambda: m.mhc_combine_norm(R, post, w),
        lambda: m.mhc_hc_head(R, torch.zeros((4, 20480)), torch.zeros(1), torch.zeros(4)),
        lambda: m.mhc_prepare_weights(fn),
        lambda: m.mhc_quantize_mxfp8(y),
        lambda: m.mhc_swizzle_scales_128x4(torch.zeros((rows, 160), dtype=torch.uint8)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
