"""The Python usage example (examples/readme_step.py), run as a script, so
the documented calls stay the library's real API."""
import os
import runpy

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EXAMPLE = os.path.join(ROOT, "examples", "readme_step.py")


def test_example_is_valid_python():
    with open(EXAMPLE, encoding="utf-8") as f:
        compile(f.read(), EXAMPLE, "exec")


@pytest.mark.gpu
def test_example_runs():
    runpy.run_path(EXAMPLE, run_name="__main__")
