"""GPU parity of the top-p re-select: when the candidates above the top-p
bound weigh less than the target, the cut is selected again over every finite
entry of the row.  With the shipped slack that happens only when rounding beats
it, so no ordinary input reaches it.  A test-only build of the same sources
(build.VARIANTS["reselect"]: LS_TOPP_SLACK = -64) puts the bound above every
cut, and every top-p row takes that path: in the row kernel (ids, log-prob rows,
fused call) and in the streaming sampler (the leader finishing the row alone),
checked against the oracle like the shipped build."""
import ctypes
import os

import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import _binding
from logits_sampling_gb300 import build as cuda_build
from logits_sampling_gb300 import workloads as W

from gpu_util import check_ids, check_log_probs, gpu_log_probs, gpu_sample, odt, oracle_sample, params_of, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def reselect_lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    path = cuda_build.variant_path("reselect")
    if not os.path.exists(path):
        pytest.fail(f"{path} is missing: __graft_entry__.build() builds it")
    lib = _binding.configure(ctypes.CDLL(path))
    saved = _binding._lib
    _binding._lib = lib  # every binding call of this module goes to the variant
    yield lib
    lib.ls_set_split_policy(0)
    _binding._lib = saved


@pytest.mark.parametrize("policy", [-1, 1, 2, 8], ids=lambda c: f"split{c}")
def test_top_p_rows_reselect(reselect_lib, policy):
    assert reselect_lib.ls_set_split_policy(policy) == 0
    w = W.make_top_p(rows=24)
    ids, err, _ = gpu_sample(w)
    assert err == 0
    check_ids(ids, oracle_sample(w), f"top_p reselect split {policy}")
    w2 = W.make_decode(rows=24, vocab=20000)
    ids2, err2, _ = gpu_sample(w2)
    assert err2 == 0
    check_ids(ids2, oracle_sample(w2), f"decode reselect split {policy}")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_near_one_and_log_probs_reselect(reselect_lib, dtype):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, 20000)) * np.array([1, 1, 3, 3, 0.2, 6], np.float32)[:, None]).astype(np.float32)
    logits = W.to_bf16_bits(x) if dtype == W.BF16 else x
    for (p, T) in [(0.99, 1.0), (0.9999, 0.7), (0.5, 1.5), (0.0, 1.0)]:
        w = W.Workload("near_one", dtype, logits, 6, temperature=np.full(6, T, np.float32),
                       top_k=np.zeros(6, np.int32), top_p=np.full(6, p, np.float32),
                       seed=np.arange(6, dtype=np.uint64), no_top_k=True, no_top_p=False)
        for policy in (-1, 1, 4):
            assert reselect_lib.ls_set_split_policy(policy) == 0
            ids, err, _ = gpu_sample(w)
            assert err == 0
            check_ids(ids, oracle_sample(w), f"{dtype} p={p} T={T} split {policy}")
        lp, err = gpu_log_probs(w)
        assert err == 0
        r = oracle.log_probs(w.logits, odt(w), w.n, w.temperature, w.top_k, w.top_p)
        check_log_probs(lp, r, f"{dtype} p={p} T={T} lp")


def test_fused_reselect(reselect_lib):
    import torch
    import logits_sampling_gb300 as ls
    assert reselect_lib.ls_set_split_policy(0) == 0
    for w in (W.make_top_p(rows=16), W.make_large(rows=12, vocab=262144)):
        x = to_device(w)
        ids, lp, sel = ls.sample_log_probs(x, w.n, params_of(w), 3, w.no_top_k, w.no_top_p)
        torch.cuda.synchronize()
        ref = oracle.sample(w.logits, odt(w), w.n, w.temperature, w.top_k, w.top_p, w.seed, step=3,
                            no_top_k=w.no_top_k, no_top_p=w.no_top_p, want_lp=True)
        check_ids(ids.cpu().numpy(), ref, f"{w.name} fused reselect")
        check_log_probs(lp.cpu().numpy(), ref, f"{w.name} fused reselect lp")
