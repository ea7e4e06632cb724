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
    config.addinivalue_line("markers", "slow: long-running")


def pytest_collection_modifyitems(config, items):
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor (any device) -> uint16 numpy bit patterns, same shape."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode BF16 bit patterns through torch's own BF16 type (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def to_bf16_bits(x) -> np.ndarray:
    """Values exactly representable in BF16 -> bit patterns (raises if not exact)."""
    xd = torch.as_tensor(np.asarray(x, dtype=np.float64))
    b = xd.to(torch.bfloat16)
    if not torch.equal(b.double(), xd):
        raise ValueError("value not exact in BF16")
    return b.view(torch.int16).numpy().view(np.uint16)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (nb if nb > 0 else 1.0))


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def whole_and_head_rel_l2(got, ref):
    """Relative L2 over the whole [H, N, D] result and the largest per-head relative L2.
    got: torch tensor (any device, any float dtype, H*N*D elements in head-major order);
    ref: FP64 numpy array or tensor of the same elements.  Computed on got's device."""
    r = torch.as_tensor(ref).to(got.device, torch.float64)
    H = r.shape[0]
    g = got.reshape(r.shape).to(torch.float64)
    d = (g - r).reshape(H, -1)
    r = r.reshape(H, -1)
    rn = torch.linalg.vector_norm(r, dim=1)
    whole = (torch.linalg.vector_norm(d) / torch.linalg.vector_norm(r)).item()
    per_head = (torch.linalg.vector_norm(d, dim=1) / torch.where(rn > 0, rn, torch.ones_like(rn))).max().item()
    return whole, per_head
