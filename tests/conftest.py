import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def tiny_weights():
    import synth
    return synth.make_weights(synth.model_config("tiny"), seed=0)


@pytest.fixture(scope="session")
def tiny_oracle(tiny_weights):
    from oracle import Oracle
    return Oracle(tiny_weights, np.float32)


@pytest.fixture(scope="session")
def tiny_oracle64(tiny_weights):
    from oracle import Oracle
    return Oracle(tiny_weights, np.float64)


@pytest.fixture(scope="session")
def request1():
    import synth
    return synth.make_request(1)
