"""GPU parity of the fused call (ls_sample_log_probs): the ids equal ls_sample's
for the same arguments (outside the exemption rows); the log-prob rows and the selected token's raw
log-prob match the oracle; error rows; optional outputs."""
import numpy as np
import pytest

import oracle
from logits_sampling_gb300 import workloads as W

from gpu_util import check_ids, check_log_probs, odt, params_of, selected_tolerance, to_device

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("lp_write")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()


def _run(w, route=None, step=None, want_lp=True, want_sel=True, gather=None, t2r=None, n=None):
    import torch
    import logits_sampling_gb300 as ls
    x = to_device(w)
    nk, np_ = (w.no_top_k, w.no_top_p) if route is None else route
    step = w.step if step is None else step
    n = w.n if n is None else n
    g = None if gather is None else torch.from_numpy(np.ascontiguousarray(gather, np.int32)).cuda()
    t = None if t2r is None else torch.from_numpy(np.ascontiguousarray(t2r, np.int32)).cuda()
    prm = params_of(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids, lp, sel = ls.sample_log_probs(x, n, prm, step, nk, np_, gather_indices=g, token_to_request_index=t,
                                       want_log_probs=want_lp, want_selected=want_sel, error_word=err)
    ids_s = ls.sample(x, n, prm, step, nk, np_, gather_indices=g, token_to_request_index=t)
    torch.cuda.synchronize()
    return (ids.cpu().numpy(), None if lp is None else lp.cpu().numpy(), None if sel is None else sel.cpu().numpy(),
            ids_s.cpu().numpy(), int(err.item()))


def _check(w, out, route=None, step=None, gather=None, t2r=None, where=""):
    ids, lp, sel, ids_s, err = out
    nk, np_ = (w.no_top_k, w.no_top_p) if route is None else route
    n = len(ids)
    ref = oracle.sample(w.logits, odt(w), n, w.temperature, w.top_k, w.top_p, w.seed,
                        step=w.step if step is None else step, no_top_k=nk, no_top_p=np_, gather_indices=gather,
                        token_to_request_index=t2r, want_lp=lp is not None)
    # the same ids as ls_sample (which may run another kernel, summing the
    # row's mass in another order) on every row outside the exemption
    clear = ref["flags"] == 0
    assert np.array_equal(ids[clear], ids_s[clear]), (where, np.nonzero((ids != ids_s) & clear)[0][:10])
    check_ids(ids_s, ref, where + " ls_sample")
    assert err == ref["error_word"], (where, err, ref["error_word"])
    check_ids(ids, ref, where)
    if lp is not None:
        check_log_probs(lp, ref, where + " lp")
    if sel is not None:
        want = oracle.selected_log_probs(w.logits, odt(w), np.where(ids >= 0, ids, 0), gather_indices=gather)
        for i in range(n):
            if ids[i] < 0:
                assert np.isnan(sel[i]), (where, i)
                continue
            tol = float(selected_tolerance(want[i]))
            assert abs(float(sel[i]) - want[i]) <= tol or (np.isinf(want[i]) and sel[i] == want[i]), \
                (where, i, float(sel[i]), want[i])


def test_tiny_and_decode():
    for w in (W.make_tiny(), W.make_decode(rows=48, vocab=12000)):
        _check(w, _run(w), where=w.name)


def test_top_p_rows():
    w = W.make_top_p(rows=24)
    _check(w, _run(w), where="top_p")


def test_large_fp32_rows():
    w = W.make_large(rows=40, vocab=262144)
    _check(w, _run(w), where="large")


def test_routes_and_steps():
    w = W.make_decode(rows=32, vocab=5000)
    for route in [(False, False), (True, False), (False, True), (True, True)]:
        _check(w, _run(w, route=route, step=7), route=route, step=7, where=f"route {route}")


def test_gather_mapping_and_bad_rows():
    rng = np.random.default_rng(21)
    w = W.make_decode(rows=20, vocab=3000)
    gather = np.array([3, 19, 0, 25, -1, 7, 7, 12], np.int32)
    t2r = np.array([0, 1, 2, 3, 4, 5, 6, 9], np.int32)
    w.temperature, w.top_k, w.top_p = w.temperature[:8], w.top_k[:8], w.top_p[:8]
    w.seed = w.seed[:8]
    out = _run(w, gather=gather, t2r=t2r, n=8)
    ids = out[0]
    assert list(np.nonzero(ids < 0)[0]) == [3, 4, 7]
    assert np.all(np.isnan(out[1][[3, 4, 7]])) and np.all(np.isnan(out[2][[3, 4, 7]]))
    _check(w, out, gather=gather, t2r=t2r, where="bad rows")


def test_optional_outputs():
    w = W.make_decode(rows=16, vocab=4000)
    a = _run(w, want_lp=False)
    b = _run(w, want_sel=False)
    assert a[1] is None and b[2] is None
    assert np.array_equal(a[0], b[0])
    _check(w, a, where="selected only")
    _check(w, b, where="log-probs only")


def test_special_rows():
    V = 777
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((8, V)) * 2).astype(np.float32)
    x[0, ::5] = np.nan
    x[1, [4, 100, 700]] = np.inf
    x[2, :] = 1.5
    x[3, 10:20] = 9.0
    x[4, :] = -np.inf
    x[4, 123] = 0.0
    w = W.Workload("special", W.F32, x, 8, temperature=np.array([1, 0.7, 1, 1e-6, 1, 2, 0.5, 1], np.float32),
                   top_k=np.array([0, 0, 3, 0, 5, 0, 40, 2], np.int32),
                   top_p=np.array([1, 0.9, 1, 0.5, 1, 0.8, 0.9, 1], np.float32),
                   seed=np.arange(8, dtype=np.uint64), no_top_k=False, no_top_p=False)
    _check(w, _run(w), where="special")
