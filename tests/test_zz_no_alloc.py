"""GPU check of ls_sample_log_probs_noalloc (the fixed-scratch variant of the
fused call) against ls_sample_log_probs with a workspace: two calls in a row,
on different inputs and steps, give identical ids, log-prob rows and
selected log-probs; a batch above the fixed scratch is refused with nothing
launched.  Collected last, and independent of every other test."""
import numpy as np
import pytest

from logits_sampling_gb300 import workloads as W

from gpu_util import params_of, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()
    ls.set_split_policy(0)
    ls.set_log_prob_write_policy(1)  # the tiled write, which uses the scratch, on every batch
    yield
    ls.set_log_prob_write_policy(0)


def _both(w, x, step):
    import torch
    import logits_sampling_gb300 as ls
    prm = params_of(w)
    ids_a, lp_a, sel_a = ls.sample_log_probs(x, w.n, prm, step, w.no_top_k, w.no_top_p, workspace=True)
    ids_b, lp_b, sel_b = ls.sample_log_probs_noalloc(x, w.n, prm, step, w.no_top_k, w.no_top_p)
    torch.cuda.synchronize()
    return (ids_a.cpu().numpy(), lp_a.cpu().numpy(), sel_a.cpu().numpy()), \
           (ids_b.cpu().numpy(), lp_b.cpu().numpy(), sel_b.cpu().numpy())


def test_noalloc_matches_the_workspace_call_twice_in_a_row():
    cases = [(W.make_decode(), 3), (W.make_tiny(), 11)]
    for w, step in cases:
        x = to_device(w)
        ref, got = _both(w, x, step)
        for a, b, what in zip(ref, got, ("ids", "log-probs", "selected")):
            assert np.array_equal(a, b, equal_nan=True), (w.name, what)


def test_noalloc_refuses_more_rows_than_its_scratch():
    import torch
    import logits_sampling_gb300 as ls
    n = ls.NOALLOC_MAX_ROWS + 1
    x = torch.zeros((n, 64), dtype=torch.float32, device="cuda")
    prm = ls.SamplingParams.from_host(np.ones(n, np.float32), np.zeros(n, np.int32), np.ones(n, np.float32),
                                      np.arange(n, dtype=np.uint64))
    with pytest.raises(ls.LSError) as e:
        ls.sample_log_probs_noalloc(x, n, prm, 0, False, False)
    assert e.value.args and "at most" in str(e.value)
