"""The CPU oracle against values and laws fixed outside it (no GPU needed)."""

import os
import subprocess

import pytest

import oracle
import _pins


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(o, check):
    check(o)


def test_oracle_compiled_without_contraction():
    """The oracle's float arithmetic must not be fused into FMAs (GCC fuses by
    default on aarch64) nor built with fast math."""
    assert "-ffp-contract=off" in oracle.CFLAGS
    assert not any("fast-math" in f and not f.startswith("-fno") for f in oracle.CFLAGS)
    assert not any(f.startswith("-Ofast") for f in oracle.CFLAGS)


def test_oracle_source_has_no_fma_calls():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mhc_oracle.c")).read()
    assert "fma" not in src.replace("fast math", "")


def test_oracle_rebuilds_from_source(tmp_path):
    out = tmp_path / "liboracle.so"
    oracle.compile_library(os.path.join(os.path.dirname(oracle.__file__), "mhc_oracle.c"),
                           str(out))
    o2 = oracle.Oracle(str(out))
    _pins.check_fwd_golden(o2)
    _pins.check_gp_golden(o2)


def test_gcc_present():
    assert subprocess.run(["gcc", "--version"], capture_output=True).returncode == 0
