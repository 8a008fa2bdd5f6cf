import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def has_gpu() -> bool:
    return torch.cuda.is_available()


def np_logits(t: torch.Tensor) -> np.ndarray:
    """Host copy of logits for the oracle: fp32 as float32, bf16 as uint16 bits."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.float().numpy()


def bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of exactly representable values."""
    return np_logits(torch.tensor(values, dtype=torch.float32).to(torch.bfloat16))


def pytest_terminal_summary(terminalreporter):
    """The flag rate of every GPU-oracle comparison of the session."""
    try:
        from tests.compare import TALLY
    except ImportError:
        return
    if TALLY["decisions"]:
        terminalreporter.write_line(
            "oracle flags: {flagged} of {decisions} decisions ({rate:.2e}) inside their margins; "
            "{flagged_requests} of {requests} requests flagged".format(
                rate=TALLY["flagged"] / TALLY["decisions"], **TALLY))
