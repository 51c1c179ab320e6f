"""The product path has no fallback: without its CUDA library every entry point raises
instead of computing anything another way (run in a fresh process pointed at a missing
library file)."""

import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CODE = r"""
import sys
sys.path.insert(0, ROOT)
import torch
from quantized_attention_mean_gb300 import _lib
_lib.LIB_PATH = "/nonexistent/libsageattn.so"
_lib._lib = None
import quantized_attention_mean_gb300 as qa
q = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
for call in (lambda: qa.sage_attn(q, q, q), lambda: qa.workspace_bytes(1, 2, 2, 8, 8, 64),
             lambda: qa.merge_partials([q], [torch.zeros(1, 2, 8)])):
    try:
        call()
    except ImportError as e:
        assert "no CPU fallback" in str(e)
    else:
        raise SystemExit("an entry point ran without the library")
print("ok")
""".replace("ROOT", repr(ROOT))


def test_entry_points_raise_without_the_library():
    r = subprocess.run([sys.executable, "-c", CODE], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().endswith("ok")
