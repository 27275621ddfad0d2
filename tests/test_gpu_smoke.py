"""The entry point's smoke run (schedule, verify at T = 1 and T = 0, calibration, Markov
drafting, each checked against the oracle) as part of the GPU suite."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_smoke():
    import __graft_entry__ as g

    g.smoke()
