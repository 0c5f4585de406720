import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def read_golden(name):
    """Parse a golden fixture: 'bytes', 'values' and 'at <index> <value>' lines."""
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split(None, 1)
            if key == "bytes":
                cur = {"bytes": bytes.fromhex(rest), "values": None, "at": {}}
                blocks.append(cur)
            elif key == "values":
                cur["values"] = [float(v) for v in rest.split()]
            elif key == "at":
                idx, val = rest.split()
                cur["at"][int(idx)] = float(val)
            else:
                blocks.append((int(key), float(rest)))
    return blocks


@pytest.fixture(scope="session")
def h():
    """One qmm handle on cuda:0 for the GPU tests (fails, never skips, without a GPU)."""
    import torch

    import gemv_dequant_gemm_gb300 as q
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    handle = q.qmm_create(0)
    yield handle
    torch.cuda.synchronize()
    q.qmm_destroy(handle)
