import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: '[section]' headers, 'key = values'
    lines, '#' comments.  Returns {section: {key: str}} (section '' for keys
    before the first header)."""
    out, cur = {"": {}}, ""
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = line[1:-1]
                out[cur] = {}
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[cur][key] = val
    return out


def ints(s):
    return np.array([int(x) for x in s.split()], dtype=np.int64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().float().numpy()


def i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().to(torch.int32).numpy()


def bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
