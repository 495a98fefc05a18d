"""The driver's smoke entry point, run as a test: one small GEMM on cuda:0 against the oracle."""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def test_graft_entry_smoke(gpu_lib, capsys):
    import __graft_entry__

    __graft_entry__.smoke()
    assert "smoke ok" in capsys.readouterr().out
