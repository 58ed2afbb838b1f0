import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libwq.so")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu but no CUDA device is visible")
    return torch.device("cuda:0")


@pytest.fixture
def tune():
    """Set launch-shape knobs (wq_set_tuning) for one test; every knob it touched is
    restored to the library's own choice afterwards."""
    import weight_only_quantized_linear_gb300 as wq
    touched = []

    def set_knob(knob, value):
        wq.wq_set_tuning(knob, value)
        touched.append(knob)

    yield set_knob
    for k in touched:
        wq.wq_set_tuning(k, 0)
