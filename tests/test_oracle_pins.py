"""Pins for the CPU oracle: each test ties it to something other than itself.

* Philox4x32-10 against libcurand's host-side generator (NVIDIA's library,
  called through its C API).
* The uniform / Gumbel mapping against closed forms.
* Greedy, top_k=1 and near-zero temperature against the argmax.
* Kept sets against a brute-force enumeration of the subset definitions on
  vocabularies of at most 16 entries.
* Gumbel-max frequencies against the renormalised filtered softmax (chi-square).
* Log-probs against torch.log_softmax / scipy logsumexp in fp64.
* The speculative row layout against the counts the API page states.
* Special values (NaN, +-inf), bad indices, route flags and steps.
"""
import ctypes
import itertools
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
from logits_sampling_gb300 import workloads as W

F32 = oracle.DTYPE_F32
BF16 = oracle.DTYPE_BF16


def _sample(logits, T, k, p, seeds=None, **kw):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    n = logits.shape[0] if "gather_indices" not in kw or kw["gather_indices"] is None else len(kw["gather_indices"])
    nreq = n if kw.get("token_to_request_index") is None else int(np.max(kw["token_to_request_index"])) + 1
    nreq = kw.pop("nreq", nreq)
    T = np.broadcast_to(np.float32(T), (nreq,)) if np.ndim(T) == 0 else T
    k = np.broadcast_to(np.int32(k), (nreq,)) if np.ndim(k) == 0 else k
    p = np.broadcast_to(np.float32(p), (nreq,)) if np.ndim(p) == 0 else p
    seeds = np.arange(nreq, dtype=np.uint64) if seeds is None else seeds
    return oracle.sample(logits, F32, n, T, k, p, seeds, **kw)


# --------------------------------------------------------------------------
# Philox4x32-10 against libcurand's host generator
# --------------------------------------------------------------------------
def _curand_host():
    for name in ("libcurand.so", "libcurand.so.10"):
        for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
                  "/usr/local/cuda/targets/x86_64-linux/lib", ""):
            path = os.path.join(d, name) if d else name
            try:
                return ctypes.CDLL(path)
            except OSError:
                continue
    return None


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def _curand_words(lib, seed, n_words, offset_words):
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset_words)) == 0
        buf = (ctypes.c_uint32 * n_words)()
        assert lib.curandGenerate(gen, buf, ctypes.c_size_t(n_words)) == 0
        return np.frombuffer(buf, dtype=np.uint32).copy()
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed,offset_blocks", [
    (0, 0), (1, 0), (0xDEADBEEF01234567, 0), (0x0123456789ABCDEF, 65536 * 3 + 17),
    (0xFFFFFFFFFFFFFFFF, (1 << 40) + 12345), (42, ((1 << 33) + 7) * 65536 + 999),
])
def test_philox_matches_curand_host_generator(seed, offset_blocks):
    """libcurand's host Philox4x32-10 generator hands out 4-word blocks; block b
    of seed s is Philox(counter=(lo32(b>>16), hi32(b>>16), b & 0xffff, 0),
    key=(lo32(s), hi32(s))).  This exercises both key words, three counter
    words and all four output lanes of the oracle's Philox."""
    lib = _curand_host()
    if lib is None:
        pytest.skip("libcurand not loadable on this host")
    nblk = 96
    words = _curand_words(lib, seed, 4 * nblk, 4 * offset_blocks)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in range(nblk):
        b = offset_blocks + i
        hi = b >> 16
        ctr = [hi & 0xFFFFFFFF, hi >> 32, b & 0xFFFF, 0]
        assert list(oracle.philox4x32_10(ctr, key)) == list(words[4 * i:4 * i + 4]), (seed, b)


def test_philox_counter_words_all_matter():
    """Changing any counter or key word changes every output lane (avalanche),
    so no word is dropped from the round function."""
    base_c, base_k = [1, 2, 3, 4], [5, 6]
    ref = oracle.philox4x32_10(base_c, base_k)
    for w in range(4):
        c = list(base_c)
        c[w] ^= 1
        out = oracle.philox4x32_10(c, base_k)
        assert np.all(out != ref)
    for w in range(2):
        k = list(base_k)
        k[w] ^= 1
        assert np.all(oracle.philox4x32_10(base_c, k) != ref)


def test_noise_word_layout():
    """word(seed, step, row, j) = lane j%4 of Philox((j/4, row, lo32 step, hi32 step), (lo32 seed, hi32 seed))."""
    seed, step, row = 0x1122334455667788, (7 << 32) | 9, 13
    for j in [0, 1, 2, 3, 4, 5, 1001, 262143]:
        blk = oracle.philox4x32_10([j >> 2, row, step & 0xFFFFFFFF, step >> 32], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.noise_word(seed, step, row, j) == int(blk[j & 3])


# --------------------------------------------------------------------------
# uniform and Gumbel mapping
# --------------------------------------------------------------------------
def test_uniform_closed_forms():
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform(1 << 9) == 3.0 * 2.0 ** -24
    rng = np.random.default_rng(0)
    for x in rng.integers(0, 2 ** 32, 200, dtype=np.uint64):
        u = oracle.uniform(int(x))
        m = u * 2 ** 24
        assert m == int(m) and int(m) % 2 == 1 and 0 < u < 1


def test_gumbel_bounds_closed_form():
    g_lo = -math.log(24 * math.log(2.0))
    g_hi = -math.log(-math.log1p(-2.0 ** -24))
    assert oracle.gumbel(0) == pytest.approx(g_lo, abs=1e-12)
    assert oracle.gumbel(0xFFFFFFFF) == pytest.approx(g_hi, rel=1e-9)
    assert g_lo == pytest.approx(-2.8116, abs=1e-4)
    assert g_hi == pytest.approx(16.6355, abs=1e-4)


def test_gumbel_distribution_ks():
    rng = np.random.default_rng(1)
    xs = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64)
    g = np.array([oracle.gumbel(int(x)) for x in xs])
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 1e-3


# --------------------------------------------------------------------------
# greedy / top_k=1 / near-zero temperature = argmax
# --------------------------------------------------------------------------
def _unique_max_rows(rng, n, V, scale=3.0):
    x = (rng.standard_normal((n, V)) * scale).astype(np.float32)
    for r in range(n):
        while np.sum(x[r] == x[r].max()) > 1:
            x[r] = (rng.standard_normal(V) * scale).astype(np.float32)
    return x


def test_greedy_below_eps_is_argmax():
    rng = np.random.default_rng(2)
    x = _unique_max_rows(rng, 64, 500)
    for T in [0.0, 1e-6, 9.9e-6, -1.0, float("nan")]:
        r = _sample(x, T, 0, 1.0)
        assert np.array_equal(r["ids"], np.argmax(x, axis=1)), T
        assert np.array_equal(r["kept"].sum(1), np.ones(64))


def test_greedy_ties_take_lowest_index():
    x = np.zeros((3, 10), np.float32)
    x[0, [3, 7]] = 5.0
    x[1, [9, 0, 4]] = 2.0
    x[2, :] = 1.0
    r = _sample(x, 0.0, 0, 1.0, want_lp=True)
    assert list(r["ids"]) == [3, 0, 0]
    assert np.allclose(r["lp"][0][[3, 7]], -math.log(2))
    assert np.allclose(r["lp"][2], -math.log(10))


def test_top_k_1_is_argmax():
    rng = np.random.default_rng(3)
    x = _unique_max_rows(rng, 128, 300)
    r = _sample(x, 1.3, 1, 0.7)
    assert np.array_equal(r["ids"], np.argmax(x, axis=1))


def test_small_temperature_with_gap_is_argmax():
    """With T = 1e-4 and a top gap d > 19.45 T, z_max - z_other > 19.45 exceeds
    the full span of the noise (g in [-2.8117, 16.6356]), so argmax is forced."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((200, 64)) * 0.1).astype(np.float32)
    am = rng.integers(0, 64, 200)
    for r in range(200):
        x[r, am[r]] = x[r].max() + np.float32(0.01)
    r = _sample(x, 1e-4, 0, 1.0)
    assert np.array_equal(r["ids"], am)


# --------------------------------------------------------------------------
# kept sets against brute force (V <= 16)
# --------------------------------------------------------------------------
def _brute_kept(l, T, k, p, allow_k=True, allow_p=True):
    V = len(l)
    l = [(-math.inf if math.isnan(v) else float(v)) for v in l]
    finite = [j for j in range(V) if l[j] > -math.inf]
    # top-k subset definition: j survives iff fewer than k entries are strictly larger
    if allow_k and 1 <= k < V:
        K = [j for j in finite if sum(1 for i in range(V) if l[i] > l[j]) < k]
    else:
        K = list(finite)
    if allow_p and np.float32(p) < np.float32(0.99999):
        z = {j: l[j] / float(np.float32(T)) for j in K}
        zm = max(z.values())
        w = {j: math.exp(z[j] - zm) for j in K}
        S = sum(w.values())
        best = None
        for mask in range(1, 1 << len(K)):
            A = [K[t] for t in range(len(K)) if mask >> t & 1]
            Aset = set(A)
            # upward closed in z (ties included)
            if any(z[i] >= z[j] and i not in Aset for j in A for i in K):
                continue
            if sum(w[j] for j in A) >= float(np.float32(p)) * S:
                if best is None or len(A) < len(best):
                    best = A
        K = sorted(best)
    return sorted(K)


def _tie_rows(rng, n, V):
    rows = []
    for _ in range(n):
        if rng.random() < 0.5:
            vals = rng.integers(-3, 4, V).astype(np.float32)  # many ties
        else:
            vals = (rng.standard_normal(V) * 2).astype(np.float32)
        rows.append(vals)
    return np.array(rows, np.float32)


def test_kept_set_brute_force_top_k():
    rng = np.random.default_rng(5)
    for V in [1, 2, 3, 7, 16]:
        x = _tie_rows(rng, 60, V)
        for k in [0, 1, 2, 3, 5, 16, 20]:
            r = _sample(x, 0.9, k, 1.0)
            for i in range(len(x)):
                assert list(np.nonzero(r["kept"][i])[0]) == _brute_kept(x[i], 0.9, k, 1.0), (V, k, i)


def test_kept_set_brute_force_top_p_and_joint():
    rng = np.random.default_rng(6)
    checked = 0
    for V in [1, 2, 5, 9, 12]:
        x = _tie_rows(rng, 40, V)
        for (k, p, T) in [(0, 0.5, 1.0), (0, 0.9, 0.7), (0, 0.0, 1.0), (0, -1.0, 2.0), (3, 0.8, 1.1),
                          (5, 0.3, 0.6), (0, 0.99, 1.0)]:
            r = _sample(x, T, k, p)
            for i in range(len(x)):
                if r["flags"][i] & oracle.FLAG_TOP_P_TIE:
                    continue
                assert list(np.nonzero(r["kept"][i])[0]) == _brute_kept(x[i], T, k, p), (V, k, p, i)
                checked += 1
    assert checked > 1000


def test_route_flags_disable_filters():
    """no_top_k / no_top_p switch the filter off for every row, whatever the
    per-request values say (the batch flags choose the route)."""
    rng = np.random.default_rng(7)
    x = _tie_rows(rng, 30, 9)
    for nk, np_ in [(True, False), (False, True), (True, True)]:
        r = _sample(x, 1.0, 3, 0.6, no_top_k=nk, no_top_p=np_)
        for i in range(len(x)):
            assert list(np.nonzero(r["kept"][i])[0]) == _brute_kept(x[i], 1.0, 3, 0.6, not nk, not np_)


# --------------------------------------------------------------------------
# sampling distribution (chi-square over seeds)
# --------------------------------------------------------------------------
def _chi2_pvalue(ids, probs):
    counts = np.bincount(ids, minlength=len(probs)).astype(float)
    n = counts.sum()
    exp = probs * n
    assert counts[probs == 0].sum() == 0, "sampled an entry outside the kept set"
    order = np.argsort(exp)
    # merge the smallest expected bins until each merged bin expects >= 5
    obs_m, exp_m, acc_o, acc_e = [], [], 0.0, 0.0
    for j in order:
        if exp[j] == 0:
            continue
        acc_o += counts[j]
        acc_e += exp[j]
        if acc_e >= 5:
            obs_m.append(acc_o)
            exp_m.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0:
        obs_m[-1] += acc_o
        exp_m[-1] += acc_e
    return stats.chisquare(obs_m, exp_m).pvalue


def _filtered_softmax(l, T, kept):
    z = np.where(kept, l.astype(np.float64) / T, -np.inf)
    return np.exp(z - special.logsumexp(z))


@pytest.mark.parametrize("V,k,p,T", [(8, 0, 1.0, 1.0), (16, 5, 1.0, 0.7), (16, 0, 0.8, 1.2), (12, 6, 0.7, 0.9),
                                     (1000, 50, 0.9, 1.0), (1000, 0, 1.0, 1.5)])
def test_gumbel_max_frequencies_chi_square(V, k, p, T):
    rng = np.random.default_rng(100 + V + k)
    row = (rng.standard_normal(V) * (1.5 if V <= 16 else 2.0)).astype(np.float32)
    nsamp = 100_000
    gather = np.zeros(nsamp, np.int32)
    r = _sample(row[None, :], T, k, p, gather_indices=gather, nreq=nsamp, want_kept=False)
    if V <= 16:
        kept = np.zeros(V, bool)
        kept[_brute_kept(row, T, k, p)] = True
    else:
        # kept set from sorting with numpy (independent of the oracle's code)
        kept = np.ones(V, bool)
        if 1 <= k < V:
            kept &= row >= np.sort(row)[::-1][k - 1]
        if p < 0.99999:
            z = row.astype(np.float64) / T
            order = np.argsort(-z, kind="stable")
            w = np.exp(z[order] - z.max())
            w[~kept[order]] = 0
            c = np.cumsum(w)
            cut = z[order][np.searchsorted(c, p * c[-1])]
            kept &= z >= cut
    probs = _filtered_softmax(row, T, kept)
    assert _chi2_pvalue(r["ids"], probs) > 1e-3


def test_inf_row_is_uniform_over_inf_entries():
    V = 12
    row = np.linspace(-5, 5, V).astype(np.float32)
    row[[2, 5, 11]] = np.inf
    nsamp = 30000
    r = _sample(row[None, :], 0.7, 4, 0.5, gather_indices=np.zeros(nsamp, np.int32), nreq=nsamp, want_kept=False)
    probs = np.zeros(V)
    probs[[2, 5, 11]] = 1 / 3
    assert _chi2_pvalue(r["ids"], probs) > 1e-3
    g = _sample(row[None, :], 0.0, 0, 1.0, want_lp=True)
    assert g["ids"][0] == 2
    assert np.allclose(g["lp"][0][[2, 5, 11]], -math.log(3))


# --------------------------------------------------------------------------
# log-probs
# --------------------------------------------------------------------------
def test_log_probs_unfiltered_equal_log_softmax():
    import torch
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((16, 777)) * 3).astype(np.float32)
    T = rng.uniform(0.3, 1.5, 16).astype(np.float32)
    r = oracle.log_probs(x, F32, 16, T, np.zeros(16, np.int32), np.ones(16, np.float32))
    ref = torch.log_softmax(torch.from_numpy(x).double() / torch.from_numpy(T).double()[:, None], dim=1).numpy()
    assert np.max(np.abs(r["lp"] - ref)) < 1e-6


def test_log_probs_filtered_logsumexp_zero():
    w = W.make_tiny()
    r = oracle.log_probs(w.logits, F32, w.n, w.temperature, w.top_k, w.top_p)
    for i in range(w.n):
        kept = r["kept"][i]
        assert abs(special.logsumexp(r["lp"][i][kept])) < 1e-5
        assert np.all(np.isneginf(r["lp"][i][~kept]))
        z = w.logits[i].astype(np.float64) / w.temperature[i]
        ref = z[kept] - special.logsumexp(z[kept])
        assert np.max(np.abs(r["lp"][i][kept] - ref)) < 1e-9


def test_sample_and_log_probs_agree_on_kept_set():
    w = W.make_decode(rows=16, vocab=3000)
    s = oracle.sample(w.logits, BF16, w.n, w.temperature, w.top_k, w.top_p, w.seed, want_lp=True)
    lp = oracle.log_probs(w.logits, BF16, w.n, w.temperature, w.top_k, w.top_p)
    assert np.array_equal(s["kept"], lp["kept"])
    assert np.array_equal(s["lp"], lp["lp"])
    for i in range(w.n):
        assert s["kept"][i][s["ids"][i]]


# --------------------------------------------------------------------------
# bf16 input, special values, indices, steps
# --------------------------------------------------------------------------
def test_bf16_reads_widen_exactly():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((8, 257)) * 3).astype(np.float32)
    bits = W.to_bf16_bits(x)
    widened = W.bf16_bits_to_f32(bits)
    T, k, p = np.full(8, 0.9, np.float32), np.full(8, 7, np.int32), np.full(8, 0.8, np.float32)
    seed = np.arange(8, dtype=np.uint64)
    a = oracle.sample(bits, BF16, 8, T, k, p, seed, want_lp=True)
    b = oracle.sample(widened, F32, 8, T, k, p, seed, want_lp=True)
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["lp"], b["lp"])
    assert np.all(np.abs(widened - x) <= np.abs(x) * 2.0 ** -8)


def test_nan_reads_as_minus_inf_and_empty_rows_error():
    rng = np.random.default_rng(10)
    x = (rng.standard_normal((4, 50))).astype(np.float32)
    y = x.copy()
    x[:, ::7] = np.nan
    y[:, ::7] = -np.inf
    a = _sample(x, 1.0, 10, 0.9, want_lp=True)
    b = _sample(y, 1.0, 10, 0.9, want_lp=True)
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["lp"], b["lp"])
    z = np.full((2, 9), -np.inf, np.float32)
    z[1, 3] = np.nan
    r = _sample(z, 1.0, 0, 1.0, want_lp=True)
    assert list(r["ids"]) == [-1, -1] and r["error_word"] == oracle.ERR_NO_FINITE
    assert np.all(np.isnan(r["lp"]))


def test_bad_indices_set_error_bits():
    x = np.zeros((4, 8), np.float32)
    r = _sample(x, 1.0, 0, 1.0, gather_indices=np.array([0, 4, -1, 3], np.int32), nreq=4)
    assert list(r["ids"][[1, 2]]) == [-1, -1] and r["ids"][0] >= 0 and r["ids"][3] >= 0
    assert r["error_word"] == oracle.ERR_BAD_GATHER
    r = _sample(x, 1.0, 0, 1.0, token_to_request_index=np.array([0, 1, 2, 9], np.int32), nreq=4)
    assert r["ids"][3] == -1 and r["error_word"] == oracle.ERR_BAD_REQUEST


def test_same_step_reproduces_and_new_step_refreshes():
    w = W.make_decode(rows=64, vocab=2000)
    a = oracle.sample(w.logits, BF16, w.n, w.temperature, w.top_k, w.top_p, w.seed, step=5, want_kept=False)
    b = oracle.sample(w.logits, BF16, w.n, w.temperature, w.top_k, w.top_p, w.seed, step=5, want_kept=False)
    c = oracle.sample(w.logits, BF16, w.n, w.temperature, w.top_k, w.top_p, w.seed, step=6, want_kept=False)
    assert np.array_equal(a["ids"], b["ids"])
    assert np.mean(a["ids"] != c["ids"]) > 0.2
    assert oracle.gumbel_at(3, 5, 0, 11) != oracle.gumbel_at(3, 6, 0, 11)
    assert oracle.gumbel_at(3, 5, 0, 11) != oracle.gumbel_at(3, 5, 1, 11)
    assert oracle.gumbel_at(3, 5, 0, 11) != oracle.gumbel_at(4, 5, 0, 11)


def test_steps_give_the_filtered_softmax_over_time():
    """One request, one row, 20000 consecutive steps: the ids follow the
    filtered softmax (fresh randomness per step)."""
    rng = np.random.default_rng(11)
    row = (rng.standard_normal(10) * 1.2).astype(np.float32)
    kept = np.zeros(10, bool)
    kept[_brute_kept(row, 1.0, 6, 1.0)] = True
    ids = [int(_sample(row[None, :], 1.0, 6, 1.0, step=s, want_kept=False)["ids"][0]) for s in range(20000)]
    assert _chi2_pvalue(np.array(ids), _filtered_softmax(row, 1.0, kept)) > 1e-3


# --------------------------------------------------------------------------
# speculative layout
# --------------------------------------------------------------------------
@pytest.mark.parametrize("D,P,S", [(128, 32, 4), (0, 5, 3), (7, 0, 0), (3, 2, 1), (0, 0, 2)])
def test_speculative_mapping_counts(D, P, S):
    """Decode requests contribute 1 + S rows, prefill requests 1; decode rows
    come first and each request's rows are contiguous."""
    m = oracle.speculative_mapping(D, P, S)
    assert len(m) == D * (1 + S) + P
    counts = np.bincount(m, minlength=D + P) if len(m) else np.zeros(D + P, int)
    assert np.all(counts[:D] == 1 + S) and np.all(counts[D:] == 1)
    assert np.all(np.diff(m) >= 0) and np.all(np.diff(m) <= 1)


# --------------------------------------------------------------------------
# exemption flags
# --------------------------------------------------------------------------
def test_score_tie_flag():
    """Two kept entries whose perturbed scores coincide are flagged."""
    g0 = oracle.gumbel_at(0, 0, 0, 0)
    g1 = oracle.gumbel_at(0, 0, 0, 1)
    row = np.array([0.0, np.float32(g0 - g1)], np.float32)
    r = _sample(row[None, :], 1.0, 0, 1.0)
    assert r["flags"][0] & oracle.FLAG_SCORE_TIE
    far = np.array([0.0, np.float32(g0 - g1 + 1.0)], np.float32)
    assert not (_sample(far[None, :], 1.0, 0, 1.0)["flags"][0] & oracle.FLAG_SCORE_TIE)


def test_top_p_tie_flag():
    """Two entries of equal mass and p = 0.5: the cut sits exactly on p * S."""
    row = np.array([[1.0, 1.0 - 1e-7, -np.inf]], np.float32)
    r = _sample(row, 1.0, 0, 0.5)
    assert r["flags"][0] & oracle.FLAG_TOP_P_TIE
    clear = np.array([[3.0, 0.0, -5.0]], np.float32)
    assert not (_sample(clear, 1.0, 0, 0.5)["flags"][0] & oracle.FLAG_TOP_P_TIE)


def test_top_p_tie_band_kept_sets():
    """Closed forms.  Logits (1, 0, -1, -2) at T = 1 weigh 1, e^-1, e^-2, e^-3
    relative to the maximum.  With p = 1 / S the first value alone carries the
    target mass, so the row is flagged, the kept set is {0}, the tight set (a
    target 1e-5 S lower) {0} and the loose set (a target 1e-5 S higher) {0, 1}.
    Under top_k = 2 the loose set stays inside the top-k set.  A deep tail of
    many tiny, distinct masses puts several values inside the band: the loose
    set then reaches past the next value.  Unflagged rows: tight = loose = kept."""
    def below(x):  # the largest float32 not above x: p * S stays at or below the first value's mass
        f = np.float32(x)
        return f if float(f) <= x else np.nextafter(f, np.float32(0))

    row = np.array([[1.0, 0.0, -1.0, -2.0]], np.float32)
    S = 1.0 + math.exp(-1) + math.exp(-2) + math.exp(-3)
    r = _sample(row, 1.0, 0, below(1.0 / S))
    assert r["flags"][0] & oracle.FLAG_TOP_P_TIE
    assert list(np.nonzero(r["kept"][0])[0]) == [0]
    assert list(np.nonzero(r["kept_tight"][0])[0]) == [0]
    assert list(np.nonzero(r["kept_loose"][0])[0]) == [0, 1]
    lp = oracle.log_probs(row, F32, 1, np.float32([1.0]), np.int32([0]), np.float32([below(1.0 / S)]))
    for key in ("kept", "kept_loose", "kept_tight"):
        assert np.array_equal(lp[key], r[key]), key
    rk = _sample(row, 1.0, 2, below(1.0 / (1.0 + math.exp(-1))))
    assert rk["flags"][0] & oracle.FLAG_TOP_P_TIE
    assert list(np.nonzero(rk["kept"][0])[0]) == [0]
    assert list(np.nonzero(rk["kept_loose"][0])[0]) == [0, 1]
    # value 0 carries mass 1; fifty distinct tail values near ln(2e-6) carry
    # about 2e-6 each (1e-4 together).  With the target inside the tail
    # (p = 1 - 5e-5) the band of +-1e-5 S spans about five tail values on
    # each side of the cut: tight < kept < loose by several values each
    tail = np.array([0.0] + [math.log(2e-6) - 0.001 * t for t in range(50)], np.float32)[None, :]
    rt = _sample(tail, 1.0, 0, np.float32(1.0 - 5e-5))
    kt, kc, kl = (int(rt[key][0].sum()) for key in ("kept_tight", "kept", "kept_loose"))
    assert rt["flags"][0] & oracle.FLAG_TOP_P_TIE
    assert np.all(rt["kept_tight"][0] <= rt["kept"][0]) and np.all(rt["kept"][0] <= rt["kept_loose"][0])
    assert kt + 3 <= kc <= kl - 3, (kt, kc, kl)
    clear = _sample(np.array([[3.0, 0.0, -5.0, 1.0]], np.float32), 1.0, 0, 0.5)
    assert clear["flags"][0] == 0
    assert np.array_equal(clear["kept_loose"], clear["kept"]) and np.array_equal(clear["kept_tight"], clear["kept"])
    rng = np.random.default_rng(3)
    many = _sample((rng.standard_normal((64, 40)) * 2).astype(np.float32), 0.9, 5, 0.8)
    for i in range(64):
        if not many["flags"][i] & oracle.FLAG_TOP_P_TIE:
            assert np.array_equal(many["kept_loose"][i], many["kept"][i])
            assert np.array_equal(many["kept_tight"][i], many["kept"][i])
        assert np.all(many["kept_loose"][i] >= many["kept"][i]) and np.all(many["kept"][i] >= many["kept_tight"][i])


# --------------------------------------------------------------------------
# selected-token log-prob under the raw logits
# --------------------------------------------------------------------------
def test_selected_log_prob_closed_forms():
    """Uniform rows give -ln V; a lone finite entry gives 0 (others -inf); two
    finite entries a, b give -ln(1 + e^(b - a))."""
    for V in (1, 2, 7, 1000):
        x = np.full((3, V), 0.25, np.float32)
        lp = oracle.selected_log_probs(x, F32, [0, V - 1, V // 2])
        assert np.allclose(lp, -np.log(V), rtol=0, atol=1e-12)
    x = np.full((1, 6), -np.inf, np.float32)
    x[0, 4] = 3.5
    assert oracle.selected_log_probs(x, F32, [4])[0] == 0.0
    assert oracle.selected_log_probs(x, F32, [1])[0] == -np.inf
    for a, b in [(0.0, 0.0), (1.0, -2.0), (-3.25, 7.5)]:
        x = np.full((1, 5), -np.inf, np.float32)
        x[0, 1], x[0, 3] = a, b
        got = oracle.selected_log_probs(x, F32, [1])[0]
        assert abs(got - (-np.log1p(np.exp(b - a)))) < 1e-12


def test_selected_log_prob_normalises_and_shifts():
    """exp of the selected log-probs over every id sums to 1, and adding a
    constant to the row (exactly representable) changes nothing."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((1, 9)) * 3).astype(np.float32)
    lp = oracle.selected_log_probs(np.repeat(x, 9, axis=0), F32, np.arange(9))
    assert abs(np.exp(lp).sum() - 1.0) < 1e-12
    x2 = (x + np.float32(16.0)).astype(np.float32)
    lp2 = oracle.selected_log_probs(np.repeat(x2, 9, axis=0), F32, np.arange(9))
    assert np.allclose(lp, lp2, rtol=0, atol=1e-5)  # x + 16 rounds in fp32


def test_selected_log_prob_special_values():
    """NaN is read as -inf; a +inf maximum shares the mass among +inf entries;
    bad ids and rows give NaN; bf16 rows widen exactly."""
    x = np.array([[np.nan, 0.0, 0.0]], np.float32)
    assert abs(oracle.selected_log_probs(x, F32, [1])[0] + np.log(2)) < 1e-15
    x = np.array([[np.inf, 1.0, np.inf, 2.0]], np.float32)
    lp = oracle.selected_log_probs(np.repeat(x, 2, axis=0), F32, [0, 3])
    assert abs(lp[0] + np.log(2)) < 1e-15 and lp[1] == -np.inf
    assert np.isnan(oracle.selected_log_probs(np.zeros((1, 4), np.float32), F32, [4])[0])
    assert np.isnan(oracle.selected_log_probs(np.zeros((1, 4), np.float32), F32, [0], gather_indices=[3])[0])
    assert np.isnan(oracle.selected_log_probs(np.full((1, 4), -np.inf, np.float32), F32, [0])[0])
    from logits_sampling_gb300 import workloads as W
    xf = np.array([[1.0, -2.5, 0.375, 3.0]], np.float32)
    assert np.array_equal(oracle.selected_log_probs(W.to_bf16_bits(xf), oracle.DTYPE_BF16, [2]),
                          oracle.selected_log_probs(xf, F32, [2]))


# --------------------------------------------------------------------------
# speculative chain verification
# --------------------------------------------------------------------------
def test_verify_chain_hand_cases():
    """Request 0: every draft matches the previous target token (all three
    accepted); request 1: the first draft misses (none); request 2: the second
    draft misses (one); request 3: a later match after a miss does not count."""
    cand = np.array([[5, 10, 11, 12],
                     [5, 99, 11, 12],
                     [5, 20, 98, 22],
                     [5, 30, 0, 32]], np.int32)
    tgt = np.array([10, 11, 12, 13,
                    40, 41, 42, 43,
                    20, 21, 22, 23,
                    31, 32, 33, 34], np.int32)
    pred, ai, an = oracle.verify_chain(cand, tgt)
    assert an.tolist() == [3, 0, 1, 0]
    assert ai.tolist() == [[0, 1, 2, 3], [4, -1, -1, -1], [8, 9, -1, -1], [12, -1, -1, -1]]
    assert pred.tolist() == [10, 11, 12, 13, 40, -7, -7, -7, 20, 21, -7, -7, 31, -7, -7, -7]


def test_verify_chain_single_position_and_brute_force():
    """n = 1 accepts only the root; for random small cases the accepted count is
    the length of the matching prefix, found here by direct comparison."""
    pred, ai, an = oracle.verify_chain(np.array([[3], [4]], np.int32), np.array([8, 9], np.int32))
    assert an.tolist() == [0, 0] and ai.tolist() == [[0], [1]] and pred.tolist() == [8, 9]
    rng = np.random.default_rng(2)
    for _ in range(50):
        bs, n = rng.integers(1, 5), rng.integers(1, 6)
        cand = rng.integers(0, 3, (bs, n)).astype(np.int32)
        tgt = rng.integers(0, 3, bs * n).astype(np.int32)
        _, ai, an = oracle.verify_chain(cand, tgt)
        for b in range(bs):
            k = 0
            while k + 1 < n and cand[b, k + 1] == tgt[b * n + k]:
                k += 1
            assert an[b] == k
            assert (ai[b] >= 0).sum() == k + 1


# --------------------------------------------------------------------------
# regression anchor
# --------------------------------------------------------------------------
def test_tiny_golden_regression():
    """The oracle still reproduces the stored tiny-workload results (written by
    tests/golden/make_golden.py from the oracle itself)."""
    import json
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")
    g = json.load(open(path))
    x = np.array([[float.fromhex(v) for v in row] for row in g["logits_hex"]], np.float32)
    r = oracle.sample(x, F32, len(x), np.array(g["temperature"], np.float32), np.array(g["top_k"], np.int32),
                      np.array(g["top_p"], np.float32), np.array(g["seed"], np.uint64), step=g["step"],
                      want_lp=True)
    assert r["ids"].tolist() == g["ids"]
    for i in range(len(x)):
        assert np.nonzero(r["kept"][i])[0].tolist() == g["kept"][i]
        assert [float(v).hex() for v in r["lp"][i][r["kept"][i]]] == g["log_probs_kept_hex"][i]
