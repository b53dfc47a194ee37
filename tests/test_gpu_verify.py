"""GPU parity of speculative chain verification (ls_verify_chain) and of
sampling the verify rows followed by verification (ls_sample_verify) with the
oracle."""
import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import workloads as W

from gpu_util import check_ids, odt, params_of, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()


def _check_verify(cand, tgt, pred, ai, an, where=""):
    rpred, rai, ran = oracle.verify_chain(cand, tgt)
    assert np.array_equal(an, ran), (where, an, ran)
    assert np.array_equal(ai, rai), where
    acc = rai.reshape(-1) >= 0
    assert np.array_equal(pred[acc], rpred[acc]), where


def test_verify_chain_random():
    import torch
    import logits_sampling_gb300 as ls
    rng = np.random.default_rng(4)
    for bs, n in [(1, 1), (5, 2), (64, 5), (300, 4), (1000, 8)]:
        tgt = rng.integers(0, 4, bs * n).astype(np.int32)
        cand = rng.integers(0, 4, (bs, n)).astype(np.int32)
        # plant long accepted prefixes in half the requests
        for b in range(0, bs, 2):
            k = rng.integers(0, n)
            cand[b, 1:k + 1] = tgt[b * n:b * n + k]
        c, t = torch.from_numpy(cand).cuda(), torch.from_numpy(tgt).cuda()
        pred, ai, an = ls.verify_chain(c, t)
        torch.cuda.synchronize()
        _check_verify(cand, tgt, pred.cpu().numpy(), ai.cpu().numpy(), an.cpu().numpy(), f"bs={bs} n={n}")


def test_sample_verify_against_oracle():
    import torch
    import logits_sampling_gb300 as ls
    bs, n, V = 48, 5, 12000
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((bs * n + 7, V)) * 3).astype(np.float32)
    w = W.Workload("verify", W.BF16, W.to_bf16_bits(x), bs * n,
                   temperature=rng.uniform(0.5, 1.2, bs).astype(np.float32),
                   top_k=rng.choice([0, 20, 50], bs).astype(np.int32),
                   top_p=rng.choice([1.0, 0.9], bs).astype(np.float32),
                   seed=np.arange(bs, dtype=np.uint64), no_top_k=False, no_top_p=False)
    gather = rng.permutation(bs * n + 7)[:bs * n].astype(np.int32)
    t2r = np.repeat(np.arange(bs, dtype=np.int32), n)
    step = 9
    ref = oracle.sample(w.logits, odt(w), bs * n, w.temperature, w.top_k, w.top_p, w.seed, step=step,
                        gather_indices=gather, token_to_request_index=t2r)
    # drafts: the oracle's target tokens for a random prefix of each chain, then a miss
    cand = np.full((bs, n), -5, np.int32)
    for b in range(bs):
        k = rng.integers(0, n)
        cand[b, 1:k + 1] = ref["ids"][b * n:b * n + k]
    x_dev = to_device(w)
    out = ls.sample_verify(x_dev, torch.from_numpy(cand).cuda(), params_of(w), step, False, False,
                           gather_indices=torch.from_numpy(gather).cuda())
    torch.cuda.synchronize()
    target, pred, ai, an = (t.cpu().numpy() for t in out)
    check_ids(target, ref, "verify rows")
    if not np.any(ref["flags"]):
        assert np.array_equal(target, ref["ids"])
    _check_verify(cand, target, pred, ai, an, "sample_verify")
    assert np.array_equal(an, [min(np.argmax(np.r_[cand[b, 1:] != target[b * n:b * n + n - 1], True]), n - 1)
                               for b in range(bs)])
