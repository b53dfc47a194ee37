"""GPU parity of every kernel choice of the sampling calls (ls_set_split_policy):
the one-CTA row kernel and the streaming sampler with 1, 2, 4 and 8 CTAs per
row (a thread-block cluster), against the oracle on the five workloads at full
size (ids and the speculative mapping), through the C ABI.  The oracle runs
once per workload."""
import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import workloads as W

from conftest import SPLIT_POLICIES
from gpu_util import check_ids, gpu_sample, oracle_sample, to_device

pytestmark = pytest.mark.gpu

_REF = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()
    yield
    ls.set_split_policy(0)


def _case(name):
    if name not in _REF:
        w = W.MAKERS[name]()
        _REF[name] = (w, oracle_sample(w), to_device(w))
    return _REF[name]


@pytest.mark.parametrize("policy", SPLIT_POLICIES, ids=lambda c: f"split{c}")
@pytest.mark.parametrize("name", ["tiny", "decode", "top_p", "speculative", "large"])
def test_workload_ids_every_kernel(name, policy):
    import logits_sampling_gb300 as ls
    w, ref, x = _case(name)
    ls.set_split_policy(policy)
    ids, err, mp = gpu_sample(w, logits_dev=x)
    assert err == 0
    if mp is not None:
        assert np.array_equal(mp, oracle.speculative_mapping(*w.spec))
    nflag = check_ids(ids, ref, f"{name} split {policy}")
    assert nflag <= max(2, w.n // 50)


@pytest.mark.parametrize("policy", [1, 2, 4, 8], ids=lambda c: f"split{c}")
def test_routes_and_steps_every_kernel(policy):
    import logits_sampling_gb300 as ls
    ls.set_split_policy(policy)
    w = W.make_decode(rows=24, vocab=20000)
    for route in [(False, False), (True, False), (False, True), (True, True)]:
        for step in (0, 9, (1 << 40) + 5):
            ids, err, _ = gpu_sample(w, route=route, step=step)
            assert err == 0
            check_ids(ids, oracle_sample(w, step=step, route=route), f"split {policy} route {route} step {step}")


@pytest.mark.parametrize("policy", [1, 2, 4, 8], ids=lambda c: f"split{c}")
def test_flat_rows_overflow_the_lists(policy):
    """Flat rows with top-p near 1 and large top-k keep most of the row: the
    lists overflow and the slices are re-read from global memory."""
    import logits_sampling_gb300 as ls
    ls.set_split_policy(policy)
    rng = np.random.default_rng(31)
    rows, V = 8, 40000
    x = (rng.standard_normal((rows, V)) * 0.3).astype(np.float32)
    for dt in (W.F32, W.BF16):
        logits = W.to_bf16_bits(x) if dt == W.BF16 else x
        w = W.Workload("flat", dt, logits, rows, temperature=np.full(rows, 1.3, np.float32),
                       top_k=np.array([0, 0, 0, 0, 30000, 30000, 5000, 0], np.int32),
                       top_p=np.array([0.999, 0.99, 0.9, 0.5, 1.0, 0.995, 0.97, 1.0], np.float32),
                       seed=np.arange(rows, dtype=np.uint64), no_top_k=False, no_top_p=False)
        ids, err, _ = gpu_sample(w)
        assert err == 0
        check_ids(ids, oracle_sample(w), f"flat {dt} split {policy}")


def _probe_case(dt):
    key = ("probe", dt)
    if key not in _REF:
        rng = np.random.default_rng(47)
        rows, V = 16, 32000
        x = (rng.standard_normal((rows, V)) * 3.0).astype(np.float32)
        logits = W.to_bf16_bits(x) if dt == W.BF16 else x
        w = W.Workload("probe", dt, logits, rows, temperature=np.full(rows, 2.0, np.float32),
                       top_k=np.zeros(rows, np.int32),
                       top_p=np.array([0.001, 0.01, 0.05, 0.2, 0.5, 0.8, 0.9, 0.95] * 2, np.float32),
                       seed=np.arange(rows, dtype=np.uint64) + 7, no_top_k=True, no_top_p=False)
        _REF[key] = (w, oracle_sample(w))
    return _REF[key]


@pytest.mark.parametrize("dt", [W.BF16, W.F32])
@pytest.mark.parametrize("policy", [1, 2, 4, 8], ids=lambda c: f"split{c}")
def test_topp_probe_rounds(policy, dt):
    """Flat rows under top-p alone keep thousands of candidates.  With a small
    p the kept set is the top few entries while the best Gumbel scores lie
    anywhere among the candidates: the streaming sampler's probe rounds reject
    the best-scoring candidate round after round and, after the last round,
    fall back to the select; larger p answers within the first rounds."""
    import logits_sampling_gb300 as ls
    ls.set_split_policy(policy)
    w, ref = _probe_case(dt)
    ids, err, _ = gpu_sample(w)
    assert err == 0
    check_ids(ids, ref, f"probe {dt} split {policy}")


@pytest.mark.parametrize("dt", [W.BF16, W.F32])
def test_topp_flat_rows_row_kernel_log_probs(dt):
    """The same flat top-p rows through the one-CTA row kernel: its first
    select level bins values over [lc, M] (a key-range binning put thousands of
    candidates into a few bins) -- ids and log-prob rows against the oracle."""
    import logits_sampling_gb300 as ls
    from gpu_util import check_log_probs, gpu_log_probs
    ls.set_split_policy(-1)
    w, ref = _probe_case(dt)
    ids, err, _ = gpu_sample(w)
    assert err == 0
    check_ids(ids, ref, f"flat {dt} row kernel")
    lp, err = gpu_log_probs(w)
    assert err == 0
    rlp = oracle.log_probs(w.logits, 1 if dt == W.BF16 else 0, w.n, w.temperature, w.top_k, w.top_p)
    check_log_probs(lp, rlp, f"flat {dt} row kernel lp")
