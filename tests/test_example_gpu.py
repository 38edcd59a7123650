"""The usage example (tests/example_usage.py) runs and gives the shapes it states."""

import pytest

from _gpu import lib

pytestmark = pytest.mark.gpu


def test_example_runs():
    lib()
    import example_usage
    out, grad_res, grad_pre, streams = example_usage.main()
    assert tuple(out.shape) == (4096, 7168)
    assert tuple(grad_res.shape) == (4096, 4, 7168) and tuple(grad_pre.shape) == (4096, 4)
    assert tuple(streams.shape) == (4096, 4, 7168)
