"""The autotuner's cache file and gate, on the host (no GPU): lines are read back by key,
malformed lines are ignored, and the environment gate is read when asked to."""
import os

import pytest

import block_scaled_precision_mma_gb300 as bs


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    yield
    bs.autotune_configure(0, None)


def test_cache_file_round_trip(tmp_path):
    path = tmp_path / "autotune.txt"
    path.write_text("grouped 16384 16384 6656 8 256\n"
                    "dense 8192 8192 8192 0 0 0 2\n"
                    "not a valid line\n"
                    "\n"
                    "grouped 128 2048 7168 8 128\n")
    bs.autotune_configure(1, str(path))
    assert bs.autotune_lookup("grouped 16384 16384 6656 8") == 256
    assert bs.autotune_lookup("dense 8192 8192 8192 0 0 0") == 2
    assert bs.autotune_lookup("grouped 128 2048 7168 8") == 128
    assert bs.autotune_lookup("grouped 1 2 3 4") == -1
    assert bs.autotune_lookup("not a valid") == -1


def test_later_lines_win(tmp_path):
    path = tmp_path / "autotune.txt"
    path.write_text("dense 256 256 256 0 0 0 1\ndense 256 256 256 0 0 0 3\n")
    bs.autotune_configure(1, str(path))
    assert bs.autotune_lookup("dense 256 256 256 0 0 0") == 3


def test_missing_file_is_an_empty_cache(tmp_path):
    bs.autotune_configure(1, str(tmp_path / "none" / "autotune.txt"))
    assert bs.autotune_lookup("dense 256 256 256 0 0 0") == -1


def test_environment_gate_and_path(tmp_path, monkeypatch):
    path = tmp_path / "env.txt"
    path.write_text("grouped 1024 2048 7168 8 256\n")
    monkeypatch.setenv("BSMMA_AUTOTUNE_CACHE", str(path))
    monkeypatch.setenv("BSMMA_AUTOTUNE", "1")
    bs.autotune_configure(-1, None)
    assert bs.autotune_lookup("grouped 1024 2048 7168 8") == 256


def test_bad_enable_value():
    assert bs.load().bsmma_autotune_configure(2, None) == 1
