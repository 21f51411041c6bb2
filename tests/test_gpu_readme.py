"""The README's Python quick start runs as written (on the tiny DiT stack
instead of DiT-XL, to keep the test short)."""
import os
import re

import pytest

pytest.importorskip("layerwise_weight_offload_slot_gb300")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_quick_start_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python block in README.md"
    code = blocks[0].replace("synth.CFG_DITXL", "synth.CFG_TINY")
    assert "synth.CFG_TINY" in code
    scope = {}
    exec(compile(code, "README.md", "exec"), scope)
    st = scope["st"]
    assert st.ctx == 0   # closed by the snippet
