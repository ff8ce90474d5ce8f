"""The README's Python example, run as written (the block between its
example markers), so the documented calls stay the library's real API."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example() -> str:
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    m = re.search(r"<!-- example:begin -->\s*```python\n(.*?)```\s*<!-- example:end -->", text,
                  re.S)
    assert m, "README example block not found"
    return m.group(1)


def test_example_is_valid_python():
    compile(_example(), "README.md example", "exec")


@pytest.mark.gpu
def test_example_runs():
    exec(compile(_example(), "README.md example", "exec"), {})
