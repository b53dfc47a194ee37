"""CPU oracle for the token-sampling hot path (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and bench.py (its cpu_baseline leg and
``--impl reference``) may import this package.  It is a thin ctypes wrapper
around ``ls_oracle.c``: plain, slow, double-precision, sort-based.  It shares
no code with the CUDA library.

Functions and the passages they follow are documented in ``ls_oracle.c``.
Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
tests/test_oracle_pins.py (no function is unpinned).
"""
import ctypes
import os

import numpy as np

from .build import LIB, build_oracle

DTYPE_F32 = 0
DTYPE_BF16 = 1

ERR_BAD_GATHER = 1
ERR_BAD_REQUEST = 2
ERR_NO_FINITE = 4

FLAG_SCORE_TIE = 1
FLAG_TOP_P_TIE = 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = build_oracle()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_noise_word.argtypes = [u64, u64, u32, i64]
        lib.oracle_noise_word.restype = u32
        lib.oracle_uniform.argtypes = [u32]
        lib.oracle_uniform.restype = ctypes.c_double
        lib.oracle_gumbel.argtypes = [u32]
        lib.oracle_gumbel.restype = ctypes.c_double
        lib.oracle_gumbel_at.argtypes = [u64, u64, u32, i64]
        lib.oracle_gumbel_at.restype = ctypes.c_double
        lib.oracle_speculative_mapping.argtypes = [i32, i32, i32, P]
        lib.oracle_speculative_mapping.restype = None
        lib.oracle_sample.argtypes = [P, ctypes.c_int, i64, i64, i64, i32, P, P, P, P, P, P, i32, u64,
                                      ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P, ctypes.c_int]
        lib.oracle_sample.restype = ctypes.c_int
        lib.oracle_log_probs.argtypes = [P, ctypes.c_int, i64, i64, i64, i32, P, P, P, P, P, i32, P, P, P, P, P,
                                         P, ctypes.c_int]
        lib.oracle_log_probs.restype = ctypes.c_int
        lib.oracle_selected_log_probs.argtypes = [P, ctypes.c_int, i64, i64, i64, i32, P, P, P]
        lib.oracle_selected_log_probs.restype = ctypes.c_int
        lib.oracle_verify_chain.argtypes = [P, P, i32, i32, P, P, P]
        lib.oracle_verify_chain.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def default_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def philox4x32_10(counter, key):
    """One Philox4x32-10 block: counter (4 uint32), key (2 uint32) -> 4 uint32."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def noise_word(seed, step, row, j):
    return int(_load().oracle_noise_word(seed, step, row, j))


def uniform(x):
    return float(_load().oracle_uniform(x))


def gumbel(x):
    return float(_load().oracle_gumbel(x))


def gumbel_at(seed, step, row, j):
    return float(_load().oracle_gumbel_at(seed, step, row, j))


def speculative_mapping(num_decode, num_prefill, num_speculative_tokens):
    n = num_decode * (1 + num_speculative_tokens) + num_prefill
    out = np.zeros(n, dtype=np.int32)
    _load().oracle_speculative_mapping(num_decode, num_prefill, num_speculative_tokens, _ptr(out))
    return out


def _logits_args(logits, dtype):
    """logits: float32 array [rows, stride] or uint16 bf16 bit patterns."""
    a = np.ascontiguousarray(logits)
    if dtype == DTYPE_BF16:
        assert a.dtype == np.uint16, "bf16 logits are passed as their uint16 bit patterns"
    else:
        assert a.dtype == np.float32
    return a


def sample(logits, dtype, n, temperature, top_k, top_p, seed, step=0, no_top_k=False, no_top_p=False,
           gather_indices=None, token_to_request_index=None, vocab=None, want_kept=True, want_lp=False,
           nthreads=None):
    """Reference sampling.  Returns a dict with ids [n], kept [n, V] (bool),
    kept_loose / kept_tight [n, V] (bool, with want_kept: for a row flagged as
    a top-p near-tie, the kept sets at the lowest and the highest cut that a
    target within the 1e-5 band gives; the kept set on every other row),
    lp [n, V] (float64, optional), flags [n], top2 [n, 2], error_word."""
    a = _logits_args(logits, dtype)
    rows, stride = a.shape
    V = stride if vocab is None else vocab
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    top_k = np.ascontiguousarray(top_k, dtype=np.int32)
    top_p = np.ascontiguousarray(top_p, dtype=np.float32)
    seed = np.ascontiguousarray(seed, dtype=np.uint64)
    nreq = len(temperature)
    assert len(top_k) == nreq and len(top_p) == nreq and len(seed) == nreq
    g = None if gather_indices is None else np.ascontiguousarray(gather_indices, dtype=np.int32)
    t = None if token_to_request_index is None else np.ascontiguousarray(token_to_request_index, dtype=np.int32)
    ids = np.zeros(n, dtype=np.int32)
    kept = np.zeros((n, V), dtype=np.uint8) if want_kept else None
    kept_loose = np.zeros((n, V), dtype=np.uint8) if want_kept else None
    kept_tight = np.zeros((n, V), dtype=np.uint8) if want_kept else None
    lp = np.zeros((n, V), dtype=np.float64) if want_lp else None
    flags = np.zeros(n, dtype=np.int32)
    top2 = np.zeros((n, 2), dtype=np.float64)
    err = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_sample(_ptr(a), dtype, rows, V, stride, n, _ptr(g), _ptr(t), _ptr(temperature),
                               _ptr(top_k), _ptr(top_p), _ptr(seed), nreq, int(step), int(bool(no_top_k)),
                               int(bool(no_top_p)), _ptr(ids), _ptr(kept), _ptr(kept_loose), _ptr(kept_tight),
                               _ptr(lp), _ptr(flags), _ptr(top2), _ptr(err), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_sample failed ({rc})")
    return {"ids": ids, "kept": None if kept is None else kept.astype(bool),
            "kept_loose": None if kept_loose is None else kept_loose.astype(bool),
            "kept_tight": None if kept_tight is None else kept_tight.astype(bool), "lp": lp, "flags": flags,
            "top2": top2, "error_word": int(err[0])}


def log_probs(logits, dtype, num_rows, temperature, top_k, top_p, gather_indices=None,
              token_to_request_index=None, vocab=None, nthreads=None):
    """Reference log-probs [num_rows, V] (float64) of the processed distribution,
    with kept, kept_loose, kept_tight (as for sample), flags and error_word."""
    a = _logits_args(logits, dtype)
    rows, stride = a.shape
    V = stride if vocab is None else vocab
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    top_k = np.ascontiguousarray(top_k, dtype=np.int32)
    top_p = np.ascontiguousarray(top_p, dtype=np.float32)
    nreq = len(temperature)
    g = None if gather_indices is None else np.ascontiguousarray(gather_indices, dtype=np.int32)
    t = None if token_to_request_index is None else np.ascontiguousarray(token_to_request_index, dtype=np.int32)
    lp = np.zeros((num_rows, V), dtype=np.float64)
    kept = np.zeros((num_rows, V), dtype=np.uint8)
    kept_loose = np.zeros((num_rows, V), dtype=np.uint8)
    kept_tight = np.zeros((num_rows, V), dtype=np.uint8)
    flags = np.zeros(num_rows, dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_log_probs(_ptr(a), dtype, rows, V, stride, num_rows, _ptr(g), _ptr(t),
                                  _ptr(temperature), _ptr(top_k), _ptr(top_p), nreq, _ptr(lp), _ptr(kept),
                                  _ptr(kept_loose), _ptr(kept_tight), _ptr(flags), _ptr(err),
                                  int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_log_probs failed ({rc})")
    return {"lp": lp, "kept": kept.astype(bool), "kept_loose": kept_loose.astype(bool),
            "kept_tight": kept_tight.astype(bool), "flags": flags, "error_word": int(err[0])}


def selected_log_probs(logits, dtype, ids, gather_indices=None, vocab=None):
    """Reference log-probability of ids[i] under the raw logits of row i
    (log-softmax of the row, no temperature or filter), float64 [n]."""
    a = _logits_args(logits, dtype)
    rows, stride = a.shape
    V = stride if vocab is None else vocab
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    g = None if gather_indices is None else np.ascontiguousarray(gather_indices, dtype=np.int32)
    out = np.zeros(len(ids), dtype=np.float64)
    _load().oracle_selected_log_probs(_ptr(a), dtype, rows, V, stride, len(ids), _ptr(g), _ptr(ids), _ptr(out))
    return out


def verify_chain(candidates, target_sampled, predicts_init=None):
    """Reference chain verification.  candidates int32 [bs, n], target_sampled
    int32 [bs * n]; returns predicts [bs * n] (predicts_init where not accepted),
    accept_index [bs, n] and accept_token_num [bs]."""
    c = np.ascontiguousarray(candidates, dtype=np.int32)
    bs, n = c.shape
    t = np.ascontiguousarray(target_sampled, dtype=np.int32).reshape(-1)
    pred = (np.full(bs * n, -7, np.int32) if predicts_init is None
            else np.ascontiguousarray(predicts_init, dtype=np.int32).copy())
    ai = np.zeros((bs, n), np.int32)
    an = np.zeros(bs, np.int32)
    _load().oracle_verify_chain(_ptr(c), _ptr(t), bs, n, _ptr(pred), _ptr(ai), _ptr(an))
    return pred, ai, an
