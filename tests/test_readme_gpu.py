"""The README's usage example runs as written."""

import os
import re

import pytest

from _gpu import lib

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    lib()
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in the README"
    for code in blocks:
        exec(compile(code, "README.md", "exec"), {})
