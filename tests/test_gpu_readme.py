"""The README's Python quick start runs as written on the GPU (its own asserts
check the round trip)."""
from __future__ import annotations

import re
from pathlib import Path

import pytest
import torch

import weight_compression_codec_gb300 as sz

pytestmark = pytest.mark.gpu

README = Path(__file__).resolve().parent.parent / "README.md"


def test_readme_quick_start_runs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sz.build()
    blocks = re.findall(r"```python\n(.*?)```", README.read_text(), flags=re.S)
    assert blocks, "README has no python block"
    for code in blocks:
        exec(compile(code, str(README), "exec"), {})
    torch.cuda.synchronize()
