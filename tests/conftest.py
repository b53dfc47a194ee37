import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle._load()
    return oracle


def cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


# Every kernel choice of the sampling calls (ls_set_split_policy): per-call
# choice from the shape, the one-CTA row kernel, and the streaming sampler
# with 1, 2, 4 and 8 CTAs per row.
SPLIT_POLICIES = [0, -1, 1, 2, 4, 8]


@pytest.fixture(params=SPLIT_POLICIES, ids=lambda c: f"split{c}")
def split_policy(request):
    import logits_sampling_gb300 as ls
    ls.load_library()
    ls.set_split_policy(request.param)
    yield request.param
    ls.set_split_policy(0)


@pytest.fixture(params=[1, -1, 0], ids=["tiled-write", "row-write", "no-workspace"])
def lp_write(request):
    """Log-prob calls with a workspace and the tiled write kernel forced, with
    a workspace and the row kernel's write forced, and without a workspace."""
    import logits_sampling_gb300 as ls
    from logits_sampling_gb300 import _binding
    ls.load_library()
    ls.set_log_prob_write_policy(request.param if request.param != 0 else -1)
    _binding.LOG_PROBS_WORKSPACE = request.param != 0
    yield request.param
    ls.set_log_prob_write_policy(0)
    _binding.LOG_PROBS_WORKSPACE = True
