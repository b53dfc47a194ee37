"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every workload runs at its full size for the sampled ids (the oracle computes
them row by row); log-probs are compared on full rows, on all rows for the
small workloads and on a sample of rows for the large ones.
"""
import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import workloads as W

from gpu_util import (check_ids, check_log_probs, gpu_log_probs, gpu_sample, odt, oracle_sample, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()


def _lp_oracle(w, rows=None):
    gather = w.gather_indices if rows is None else (
        w.gather_indices[rows] if w.gather_indices is not None else np.asarray(rows, np.int32))
    t2r = None
    if w.spec is not None:
        mp = oracle.speculative_mapping(*w.spec)
        t2r = mp if rows is None else mp[rows]
    n = w.n if rows is None else len(rows)
    r = oracle.log_probs(w.logits, odt(w), n, w.temperature, w.top_k, w.top_p, gather_indices=gather,
                         token_to_request_index=t2r)
    return r, gather, t2r, n


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------
@pytest.mark.usefixtures("lp_write")
def test_tiny_ids_and_log_probs():
    w = W.make_tiny()
    ids, err, _ = gpu_sample(w)
    ref = oracle_sample(w)
    assert err == 0
    check_ids(ids, ref, "tiny")
    r, g, t, n = _lp_oracle(w)
    lp, err = gpu_log_probs(w, gather=g, t2r=t, num_rows=n)
    assert err == 0
    check_log_probs(lp, r, "tiny lp")


@pytest.mark.usefixtures("lp_write")
def test_decode_ids_and_log_probs():
    w = W.make_decode()
    ids, err, _ = gpu_sample(w)
    assert err == 0
    check_ids(ids, oracle_sample(w), "decode")
    r, g, t, n = _lp_oracle(w)
    lp, _ = gpu_log_probs(w, gather=g, t2r=t, num_rows=n)
    check_log_probs(lp, r, "decode lp")


def test_top_p_full_size_ids():
    w = W.make_top_p()
    ids, err, _ = gpu_sample(w)
    assert err == 0
    check_ids(ids, oracle_sample(w), "top_p")


@pytest.mark.usefixtures("lp_write")
def test_top_p_log_probs_sampled_rows():
    w = W.make_top_p(rows=24)
    r, g, t, n = _lp_oracle(w)
    lp, _ = gpu_log_probs(w, gather=g, t2r=t, num_rows=n)
    check_log_probs(lp, r, "top_p lp")


def test_speculative_full_size_ids_and_mapping():
    w = W.make_speculative()
    ids, err, mp = gpu_sample(w)
    assert err == 0
    assert np.array_equal(mp, oracle.speculative_mapping(*w.spec))
    check_ids(ids, oracle_sample(w), "speculative")


@pytest.mark.usefixtures("lp_write")
def test_speculative_log_probs_sampled_rows():
    w = W.make_speculative()
    rows = np.r_[0:5, 317:322, 638:642, 667:672]
    r, g, t, n = _lp_oracle(w, rows)
    x = to_device(w)
    lp, _ = gpu_log_probs(w, logits_dev=x, gather=g, t2r=t, num_rows=n)
    check_log_probs(lp, r, "speculative lp")


def test_large_full_size_ids():
    w = W.make_large()
    ids, err, _ = gpu_sample(w)
    assert err == 0
    nflag = check_ids(ids, oracle_sample(w), "large")
    assert nflag < 20


@pytest.mark.usefixtures("lp_write")
def test_large_log_probs_sampled_rows():
    w = W.make_large(rows=64, vocab=262144)
    r, g, t, n = _lp_oracle(w)
    lp, _ = gpu_log_probs(w, gather=g, t2r=t, num_rows=n)
    check_log_probs(lp, r, "large lp")


# ---------------------------------------------------------------------------
# routes, steps, determinism
# ---------------------------------------------------------------------------
def test_routes_agree_where_flags_hold():
    """The route is a performance choice only: on batches where a flag holds,
    every route that the flag allows returns the joint route's ids."""
    w = W.make_top_p(rows=32)  # no request uses top-k
    joint, _, _ = gpu_sample(w, route=(False, False))
    tp, _, _ = gpu_sample(w, route=(True, False))
    assert np.array_equal(joint, tp)
    w2 = W.make_decode(rows=48, vocab=5000)
    w2.top_p[:] = 1.0  # no request uses top-p
    a, _, _ = gpu_sample(w2, route=(False, False))
    b, _, _ = gpu_sample(w2, route=(False, True))
    assert np.array_equal(a, b)
    w2.top_k[:] = 0  # no filter at all
    c = [gpu_sample(w2, route=r)[0] for r in [(False, False), (True, False), (False, True), (True, True)]]
    assert all(np.array_equal(c[0], x) for x in c[1:])
    check_ids(c[0], oracle_sample(w2, route=(True, True)), "no-filter")


def test_route_flags_switch_filters_off():
    w = W.make_decode(rows=32, vocab=4000)
    for route in [(True, False), (False, True), (True, True)]:
        ids, _, _ = gpu_sample(w, route=route)
        check_ids(ids, oracle_sample(w, route=route), f"route {route}")


def test_steps_reproducible_and_fresh():
    w = W.make_decode(rows=64, vocab=8000)
    a, _, _ = gpu_sample(w, step=11)
    b, _, _ = gpu_sample(w, step=11)
    c, _, _ = gpu_sample(w, step=12)
    assert np.array_equal(a, b)
    assert np.mean(a != c) > 0.2
    check_ids(c, oracle_sample(w, step=12), "step 12")
    big = (1 << 40) + 5
    d, _, _ = gpu_sample(w, step=big)
    check_ids(d, oracle_sample(w, step=big), "step 2^40+5")


@pytest.mark.usefixtures("lp_write")
def test_log_probs_deterministic():
    w = W.make_decode(rows=16, vocab=6000)
    a, _ = gpu_log_probs(w)
    b, _ = gpu_log_probs(w)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
