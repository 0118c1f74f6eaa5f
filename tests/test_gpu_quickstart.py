"""The README's Python example runs as written (sizes shrunk, checkpoint
directory moved into a temporary one), so the documented calls stay the
library's calls."""
import os
import re

import pytest

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs(lib, tmp_path):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    for big, small in (("110_418_432", "65_600"), ("24_576_000", "30_000")):
        assert big in code
        code = code.replace(big, small)
    code = code.replace('"ckpt/', repr(str(tmp_path)).strip("'\"").join(['"', '/']))
    scope = {}
    exec(compile(code, "README.md", "exec"), scope)
    assert os.path.exists(tmp_path / "step_000200.bin")
    assert osr.ckpt_probe(str(tmp_path / "step_000200.bin")) == (200, 65_600)
    assert scope["step"] == 200
