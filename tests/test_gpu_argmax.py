"""GPU parity of the all-greedy fast path (ls_argmax) with the oracle's greedy
rows: random rows of both dtypes and several vocabularies, misaligned rows,
special values and ties, gather indices and bad rows."""
import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()


def _greedy_ref(x, dtype, n, gather=None):
    nreq = n
    r = oracle.sample(x, oracle.DTYPE_BF16 if dtype == W.BF16 else oracle.DTYPE_F32, n,
                      np.zeros(nreq, np.float32), np.zeros(nreq, np.int32), np.ones(nreq, np.float32),
                      np.arange(nreq, dtype=np.uint64), gather_indices=gather, want_kept=False)
    return r["ids"], r["error_word"]


def _run(x, dtype, col_off=0, pad=0, gather=None, n=None):
    import torch
    import logits_sampling_gb300 as ls
    rows, V = x.shape
    if dtype == W.BF16:
        host = W.to_bf16_bits(x)
        big = np.zeros((rows, col_off + V + pad), np.uint16)
        big[:, col_off:col_off + V] = host
        dev = torch.from_numpy(big.view(np.int16)).view(torch.bfloat16).cuda()[:, col_off:col_off + V]
    else:
        host = np.ascontiguousarray(x, np.float32)
        big = np.zeros((rows, col_off + V + pad), np.float32)
        big[:, col_off:col_off + V] = host
        dev = torch.from_numpy(big).cuda()[:, col_off:col_off + V]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = None if gather is None else torch.from_numpy(np.asarray(gather, np.int32)).cuda()
    ids = ls.argmax(dev, n=n, gather_indices=g, error_word=err)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), int(err.item()), host


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("V", [1, 5, 16, 17, 1000, 32000, 128256, 262144])
def test_random_rows(dtype, V):
    rng = np.random.default_rng(V)
    x = (rng.standard_normal((6, V)) * 3).astype(np.float32)
    ids, err, host = _run(x, dtype)
    ref, rerr = _greedy_ref(host, dtype, 6)
    assert err == rerr == 0
    assert np.array_equal(ids, ref), (ids, ref)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("col_off,pad", [(1, 0), (3, 5), (7, 1)])
def test_misaligned_rows(dtype, col_off, pad):
    rng = np.random.default_rng(col_off + 10 * pad)
    x = np.round(rng.standard_normal((9, 3001)) * 2).astype(np.float32)  # many ties
    ids, err, host = _run(x, dtype, col_off=col_off, pad=pad)
    ref, _ = _greedy_ref(host, dtype, 9)
    assert np.array_equal(ids, ref)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_special_values(dtype):
    V = 777
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((8, V)) * 2).astype(np.float32)
    x[0, ::5] = np.nan
    x[1, [40, 100, 700]] = np.inf
    x[2, :] = -np.inf
    x[3, :] = np.nan
    x[4, :] = 1.5
    x[5, 10:20] = 9.0
    x[6, :] = -np.inf
    x[6, 776] = -3.0
    x[7, :] = 0.0
    x[7, 5::7] = -0.0
    ids, err, host = _run(x, dtype)
    ref, rerr = _greedy_ref(host, dtype, 8)
    assert np.array_equal(ids, ref), (ids, ref)
    assert err == rerr == oracle.ERR_NO_FINITE
    assert list(ids[[1, 2, 3, 4, 5, 6]]) == [40, -1, -1, 0, 10, 776]


def test_gather_and_bad_rows():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((20, 5000)) * 3).astype(np.float32)
    gather = np.array([3, 19, 0, 25, -1, 7, 7, 12], np.int32)
    ids, err, host = _run(x, W.BF16, gather=gather)
    ref, rerr = _greedy_ref(host, W.BF16, 8, gather=gather)
    assert np.array_equal(ids, ref)
    assert err == rerr == oracle.ERR_BAD_GATHER
    assert list(np.nonzero(ids < 0)[0]) == [3, 4]


def test_matches_greedy_sampling():
    """ls_argmax gives the ids ls_sample gives a batch of greedy rows."""
    import torch
    import logits_sampling_gb300 as ls
    w = W.make_top_p(rows=32)
    x = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).cuda()
    prm = ls.SamplingParams.from_host(np.zeros(32), w.top_k, w.top_p, w.seed)
    a = ls.argmax(x)
    b = ls.sample(x, 32, prm, 0, True, False)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
