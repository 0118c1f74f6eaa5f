"""The quick-start example (examples/quickstart.py) runs as written, at a
small size with its checkpoints in a temporary directory, so the documented
calls stay the library's calls."""
import importlib.util
import os

import pytest

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_quickstart_example_runs(lib, tmp_path):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    spec = importlib.util.spec_from_file_location(
        "quickstart", os.path.join(ROOT, "examples", "quickstart.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    step, norm, factor = mod.main(n=65_600, first=30_000, directory=str(tmp_path))
    assert step == 200 and norm > 0 and 0 < factor <= 1
    path = tmp_path / "step_000200.bin"
    assert osr.ckpt_probe(str(path)) == (200, 65_600)
    assert os.path.exists(tmp_path / "step_000100.bin")
