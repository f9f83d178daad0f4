import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (full-size shapes)")


GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


# ----------------------------------------------------------------------------- GPU helpers


@pytest.fixture(scope="session")
def bm():
    """The CUDA library, built in place; GPU tests fail (never fall back) without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    from f16_weight_gemv_gb300 import _build
    import f16_weight_gemv_gb300 as lib
    _build.build()
    lib.lib()
    return lib


def to_dev(a, device="cuda"):
    """numpy uint16 (f16 bits) -> torch.float16 on the GPU; float32 stays float32."""
    import numpy as np
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return torch.from_numpy(a).to(device)


def bits32(t):
    """A float32 tensor or array as its uint32 bit patterns (numpy)."""
    import numpy as np
    a = t.detach().cpu().numpy() if hasattr(t, "detach") else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
