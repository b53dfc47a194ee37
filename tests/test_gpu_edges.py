"""GPU edge cases against the oracle: tiny and ragged vocabularies, misaligned
rows, special values, degenerate filters, bad indices and host-side argument
errors."""
import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import workloads as W

from gpu_util import check_ids, check_log_probs

# every test runs under each kernel choice of the sampling calls
pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("split_policy", "lp_write")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()


def _run(x, dtype, T, k, p, seed=None, step=0, no_top_k=False, no_top_p=False, col_off=0, pad=0, gather=None,
         t2r=None, nreq=None, n=None):
    """x: float32 [rows, V] host values (bf16 rounding applied here when dtype
    is bf16).  The device copy is placed at column col_off of rows padded by
    `pad` entries, so rows start at arbitrary (misaligned) addresses."""
    import torch
    import logits_sampling_gb300 as ls
    rows, V = x.shape
    n = (rows if gather is None else len(gather)) if n is None else n
    nreq = (n if t2r is None else int(np.max(t2r)) + 1) if nreq is None else nreq
    T = np.broadcast_to(np.float32(T), (nreq,)).copy() if np.ndim(T) == 0 else np.asarray(T, np.float32)
    k = np.broadcast_to(np.int32(k), (nreq,)).copy() if np.ndim(k) == 0 else np.asarray(k, np.int32)
    p = np.broadcast_to(np.float32(p), (nreq,)).copy() if np.ndim(p) == 0 else np.asarray(p, np.float32)
    seed = np.arange(nreq, dtype=np.uint64) if seed is None else seed
    if dtype == W.BF16:
        host = W.to_bf16_bits(x)
        big = np.zeros((rows, col_off + V + pad), np.uint16)
        big[:, col_off:col_off + V] = host
        dev = torch.from_numpy(big.view(np.int16)).view(torch.bfloat16).cuda()[:, col_off:col_off + V]
        odtype = oracle.DTYPE_BF16
    else:
        host = np.ascontiguousarray(x, np.float32)
        big = np.zeros((rows, col_off + V + pad), np.float32)
        big[:, col_off:col_off + V] = host
        dev = torch.from_numpy(big).cuda()[:, col_off:col_off + V]
        odtype = oracle.DTYPE_F32
    prm = ls.SamplingParams.from_host(T, k, p, seed)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gd = None if gather is None else torch.from_numpy(np.asarray(gather, np.int32)).cuda()
    td = None if t2r is None else torch.from_numpy(np.asarray(t2r, np.int32)).cuda()
    ids = ls.sample(dev, n, prm, step, no_top_k, no_top_p, gather_indices=gd, token_to_request_index=td,
                    error_word=err)
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lp = ls.log_probs(dev, prm, num_rows=n, gather_indices=gd, token_to_request_index=td, error_word=err2)
    torch.cuda.synchronize()
    ref = oracle.sample(host, odtype, n, T, k, p, seed, step=step, no_top_k=no_top_k, no_top_p=no_top_p,
                        gather_indices=gather, token_to_request_index=t2r)
    rlp = oracle.log_probs(host, odtype, n, T, k, p, gather_indices=gather, token_to_request_index=t2r)
    return ids.cpu().numpy(), int(err.item()), lp.cpu().numpy(), int(err2.item()), ref, rlp


def _check(out, where):
    ids, err, lp, err2, ref, rlp = out
    check_ids(ids, ref, where)
    assert err == ref["error_word"], (where, err, ref["error_word"])
    assert err2 == rlp["error_word"], (where, err2, rlp["error_word"])
    check_log_probs(lp, rlp, where)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("V", [1, 2, 3, 15, 16, 17, 31, 33, 1000, 4099])
def test_small_and_ragged_vocab(dtype, V):
    rng = np.random.default_rng(V)
    x = (rng.standard_normal((6, V)) * 2).astype(np.float32)
    for (k, p, T) in [(0, 1.0, 1.0), (3, 1.0, 0.8), (0, 0.7, 1.1), (5, 0.9, 0.6), (1, 0.5, 1.0)]:
        _check(_run(x, dtype, T, k, p), f"V={V} {dtype} k={k} p={p}")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("col_off,pad", [(1, 0), (3, 5), (7, 1), (0, 9)])
def test_misaligned_rows(dtype, col_off, pad):
    rng = np.random.default_rng(col_off * 10 + pad)
    x = (rng.standard_normal((9, 3001)) * 3).astype(np.float32)
    k = rng.choice([0, 7, 40], 9).astype(np.int32)
    p = rng.choice([1.0, 0.8, 0.95], 9).astype(np.float32)
    T = rng.uniform(0.4, 1.4, 9).astype(np.float32)
    _check(_run(x, dtype, T, k, p, col_off=col_off, pad=pad), f"misaligned {dtype} {col_off} {pad}")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_special_values(dtype):
    V = 777
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((10, V)) * 2).astype(np.float32)
    x[0, ::5] = np.nan                      # NaN entries read as -inf
    x[1, ::3] = -np.inf                     # -inf entries never kept
    x[2, [4, 100, 700]] = np.inf            # uniform over the +inf entries
    x[3, :] = -np.inf                       # no finite entry: error row
    x[4, :] = np.nan                        # idem
    x[5, :] = 1.5                           # all equal
    x[6, :] = -np.inf
    x[6, 123] = 0.0                         # a single finite entry
    x[7, :] = np.nan
    x[7, 9] = -3.0
    x[8, 10:20] = 9.0                       # ties at the maximum
    x[9, :] = 0.0
    x[9, 5::7] = -0.0                       # signed zeros compare equal
    for (k, p, T) in [(0, 1.0, 1.0), (4, 1.0, 1.0), (0, 0.5, 0.7), (12, 0.9, 1.3), (0, 1.0, 0.0), (2, 0.3, 0.0)]:
        _check(_run(x, dtype, T, k, p), f"special {dtype} k={k} p={p} T={T}")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_degenerate_filters(dtype):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((12, 2000)) * 3).astype(np.float32)
    x[:, 100] = x.max() + 1  # unique maximum in every row
    V = x.shape[1]
    cases = [(1, 1.0, 1.0), (V, 1.0, 1.0), (V + 5, 0.5, 1.0), (-3, 0.5, 1.0), (0, 0.0, 1.0), (0, -2.0, 0.9),
             (0, 0.99999, 1.0), (0, 0.9999, 1.0), (50, 1e-6, 1.0), (V - 1, 0.999, 2.0), (0, 1.0, 1e-5),
             (0, 1.0, 9e-6), (0, 1.0, 1e4)]
    for (k, p, T) in cases:
        out = _run(x, dtype, T, k, p)
        _check(out, f"degenerate {dtype} k={k} p={p} T={T}")
        if k == 1 or T < 1e-5 or p <= 0:
            assert np.all(out[0] == 100)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_top_p_near_one(dtype):
    # p just under the point where the filter switches off: the kept set is
    # most of a wide row, the candidate bound sits deep in the tail and the
    # candidates overflow the shared-memory list
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, 50000)) * np.array([1, 1, 3, 3, 0.2, 6], np.float32)[:, None]).astype(np.float32)
    for (p, T) in [(0.99, 1.0), (0.9999, 0.7), (0.99998, 1.5), (0.99998, 0.3)]:
        _check(_run(x, dtype, T, 0, p), f"near one {dtype} p={p} T={T}")


def test_ties_at_the_cut():
    x = np.tile(np.array([5, 5, 5, 3, 3, 3, 3, 1, 1, 0], np.float32), (4, 1))
    for (k, p) in [(2, 1.0), (4, 1.0), (0, 0.3), (0, 0.97), (5, 0.5)]:
        _check(_run(x, W.F32, 1.0, k, p), f"ties k={k} p={p}")


def test_gather_and_mapping_with_bad_indices():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((20, 3000)) * 3).astype(np.float32)
    gather = np.array([3, 19, 0, 25, -1, 7, 7, 12], np.int32)
    t2r = np.array([0, 1, 2, 3, 4, 5, 6, 9], np.int32)
    out = _run(x, W.BF16, 0.9, 10, 0.9, gather=gather, t2r=t2r, nreq=8)
    ids, err, lp, err2, ref, rlp = out
    assert err == oracle.ERR_BAD_GATHER | oracle.ERR_BAD_REQUEST
    assert list(np.nonzero(ids < 0)[0]) == [3, 4, 7]
    _check(out, "bad indices")


def test_no_finite_rows_error_bit():
    x = np.full((3, 100), -np.inf, np.float32)
    x[1, 50] = 2.0
    out = _run(x, W.F32, 1.0, 0, 1.0)
    assert out[1] == oracle.ERR_NO_FINITE and list(out[0]) == [-1, 50, -1]
    _check(out, "no finite")


def test_host_argument_errors():
    import torch
    import logits_sampling_gb300 as ls
    x = torch.zeros((4, 10), dtype=torch.float32, device="cuda")
    prm = ls.SamplingParams.from_host(np.ones(4), np.zeros(4), np.ones(4), np.arange(4))
    out = torch.full((4,), -9, dtype=torch.int32, device="cuda")
    ls.sample(x, 0, prm, 0, False, False, out=out)  # n = 0: nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == -9)
    with pytest.raises(ls.LSError) as e:
        ls.sample(x, 5, prm, 0, False, False)  # n > rows without gather
    assert e.value.status == 1
    small = ls.SamplingParams.from_host(np.ones(2), np.zeros(2), np.ones(2), np.arange(2))
    with pytest.raises(ls.LSError):
        ls.sample(x, 4, small, 0, False, False)  # n > num_requests without a mapping
    with pytest.raises(ls.LSError):
        ls.sample_speculative(x, 2, 1, 1, prm, 0, False, False)  # 5 rows > 4 logits rows
    with pytest.raises(ls.LSError):
        ls.sample_speculative(x, 3, 2, 0, prm, 0, False, False)  # 5 requests > 4
    assert ls.max_vocab(ls.LS_DTYPE_BF16) >= 262144 and ls.max_vocab(ls.LS_DTYPE_F32) >= 262144


def test_speculative_without_gather():
    import torch
    import logits_sampling_gb300 as ls
    D, P, S, V = 5, 3, 2, 5000
    n = D * (1 + S) + P
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((n + 4, V)) * 3).astype(np.float32)
    nreq = D + P + 2
    T = rng.uniform(0.5, 1.5, nreq).astype(np.float32)
    k = rng.choice([0, 10, 30], nreq).astype(np.int32)
    p = rng.choice([1.0, 0.9], nreq).astype(np.float32)
    seed = rng.integers(0, 2 ** 63, nreq).astype(np.uint64)
    prm = ls.SamplingParams.from_host(T, k, p, seed)
    mp = torch.zeros(n, dtype=torch.int32, device="cuda")
    ids = ls.sample_speculative(torch.from_numpy(x).cuda(), D, P, S, prm, 3, False, False,
                                out_token_to_request_index=mp)
    torch.cuda.synchronize()
    omap = oracle.speculative_mapping(D, P, S)
    assert np.array_equal(mp.cpu().numpy(), omap)
    ref = oracle.sample(x, oracle.DTYPE_F32, n, T, k, p, seed, step=3, token_to_request_index=omap)
    check_ids(ids.cpu().numpy(), ref, "spec no gather")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_largest_vocab(dtype):
    """A vocabulary at the library's shared-memory limit (one CTA per SM, the
    smallest candidate list, candidates re-read from L2) and the first size
    beyond it, which the host rejects."""
    import logits_sampling_gb300 as ls
    V = int(ls.max_vocab(ls.LS_DTYPE_BF16 if dtype == W.BF16 else ls.LS_DTYPE_F32))
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((4, V)) * 3).astype(np.float32)
    x[:, rng.choice(V, 50, replace=False)] += 12.0
    for (k, p, T) in [(0, 1.0, 1.0), (40, 1.0, 0.7), (0, 0.9, 0.8), (100, 0.95, 1.2)]:
        _check(_run(x, dtype, T, k, p), f"V={V} {dtype} k={k} p={p}")
    import torch
    big = torch.zeros((1, V + 64), dtype=torch.float32 if dtype == W.F32 else torch.bfloat16, device="cuda")
    prm = ls.SamplingParams.from_host(np.ones(1), np.zeros(1), np.ones(1), np.arange(1))
    with pytest.raises(ls.LSError) as e:
        ls.sample(big, 1, prm, 0, False, False)
    assert e.value.status == 2  # LS_ERR_UNSUPPORTED


def test_explicit_side_stream():
    """Calls given a stream other than the current one allocate and fill their
    outputs on that stream: the results equal those of the same calls on the
    current stream, with nothing synchronised in between but that stream."""
    import torch
    import logits_sampling_gb300 as ls
    w = W.make_decode(rows=24, vocab=9000)
    x = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).cuda()
    prm = ls.SamplingParams.from_host(w.temperature, w.top_k, w.top_p, w.seed)
    ids0 = ls.sample(x, w.n, prm, 5, w.no_top_k, w.no_top_p)
    f0 = ls.sample_log_probs(x, w.n, prm, 5, w.no_top_k, w.no_top_p)
    cand = torch.from_numpy(np.random.default_rng(1).integers(0, 9000, (6, 4)).astype(np.int32)).cuda()
    v0 = ls.verify_chain(cand, ids0[:24])
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(torch.cuda.Stream()):  # a third stream is current meanwhile
        ids1 = ls.sample(x, w.n, prm, 5, w.no_top_k, w.no_top_p, stream=side)
        f1 = ls.sample_log_probs(x, w.n, prm, 5, w.no_top_k, w.no_top_p, stream=side)
        v1 = ls.verify_chain(cand, ids1[:24], stream=side)
    side.synchronize()
    assert torch.equal(ids0, ids1)
    assert torch.equal(f0[0], f1[0]) and torch.equal(f0[1], f1[1]) and torch.equal(f0[2], f1[2])
    assert all(torch.equal(a, b) for a, b in zip(v0, v1))
