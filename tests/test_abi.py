"""The C ABI library on a host without a GPU: it builds, loads, exports every
entry point include/*.h declares, and rejects bad arguments on the host before
any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from logits_sampling_gb300 import build as b
    path = b.build()
    from logits_sampling_gb300 import _binding
    return _binding.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s+(ls_[a-z_0-9]+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_calls():
    names = _declared_functions()
    assert {"ls_sample", "ls_sample_speculative", "ls_log_probs", "ls_sample_log_probs", "ls_sample_device_step",
            "ls_argmax", "ls_verify_chain", "ls_sample_verify", "ls_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_split_policy_values(lib):
    """ls_set_split_policy accepts 0, -1, 1, 2, 4, 8 and rejects anything else
    on the host (no GPU needed)."""
    for bad in (3, 5, 16, -2, 7):
        assert lib.ls_set_split_policy(bad) == 1, bad
    for good in (-1, 1, 2, 4, 8, 0):
        assert lib.ls_set_split_policy(good) == 0, good


def test_log_prob_write_policy_values(lib):
    """ls_set_log_prob_write_policy accepts 0, 1, -1 and rejects anything else
    on the host (no GPU needed)."""
    for bad in (2, -2, 8):
        assert lib.ls_set_log_prob_write_policy(bad) == 1, bad
    for good in (1, -1, 0):
        assert lib.ls_set_log_prob_write_policy(good) == 0, good


def test_no_torch_in_the_abi():
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        assert "at::" not in text and "torch::" not in text and "Tensor" not in text


def test_host_validation_before_any_launch(lib):
    from logits_sampling_gb300._binding import _Params
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails validation first
    prm = _Params(fake, fake, fake, fake, 4)
    byref = ctypes.byref
    # n < 0
    assert lib.ls_sample(fake, 0, 4, 10, 10, -1, None, None, byref(prm), 0, 0, 0, fake, None, None) == 1
    # n == 0: OK, nothing launched
    assert lib.ls_sample(fake, 0, 4, 10, 10, 0, None, None, byref(prm), 0, 0, 0, fake, None, None) == 0
    # null logits, bad dtype, vocab < 1, stride < vocab, null out
    assert lib.ls_sample(None, 0, 4, 10, 10, 2, None, None, byref(prm), 0, 0, 0, fake, None, None) == 1
    assert lib.ls_sample(fake, 7, 4, 10, 10, 2, None, None, byref(prm), 0, 0, 0, fake, None, None) == 1
    assert lib.ls_sample(fake, 0, 4, 0, 10, 2, None, None, byref(prm), 0, 0, 0, fake, None, None) == 1
    assert lib.ls_sample(fake, 0, 4, 10, 9, 2, None, None, byref(prm), 0, 0, 0, fake, None, None) == 1
    assert lib.ls_sample(fake, 0, 4, 10, 10, 2, None, None, byref(prm), 0, 0, 0, None, None, None) == 1
    # n > logits_rows without gather; n > num_requests without a mapping
    assert lib.ls_sample(fake, 0, 4, 10, 10, 5, None, None, byref(prm), 0, 0, 0, fake, None, None) == 1
    prm2 = _Params(fake, fake, fake, fake, 2)
    assert lib.ls_sample(fake, 0, 4, 10, 10, 3, None, None, byref(prm2), 0, 0, 0, fake, None, None) == 1
    # missing parameter arrays
    prm3 = _Params(fake, None, fake, fake, 4)
    assert lib.ls_sample(fake, 0, 4, 10, 10, 2, None, None, byref(prm3), 0, 0, 0, fake, None, None) == 1
    # speculative: negative counts, too many rows / requests
    assert lib.ls_sample_speculative(fake, 1, 4, 10, 10, -1, 0, 0, None, byref(prm), 0, 0, 0, fake, None, None,
                                     None) == 1
    assert lib.ls_sample_speculative(fake, 1, 4, 10, 10, 2, 1, 1, None, byref(prm), 0, 0, 0, fake, None, None,
                                     None) == 1
    assert lib.ls_sample_speculative(fake, 1, 100, 10, 10, 3, 2, 0, None, byref(prm), 0, 0, 0, fake, None, None,
                                     None) == 1
    assert lib.ls_sample_speculative(fake, 1, 100, 10, 10, 0, 0, 3, None, byref(prm), 0, 0, 0, fake, None, None,
                                     None) == 0
    # log-probs
    lp = lib.ls_log_probs
    assert lp(fake, 1, 4, 10, 10, -2, None, None, byref(prm), fake, None, 0, None, None) == 1
    assert lp(fake, 1, 4, 10, 10, 0, None, None, byref(prm), fake, None, 0, None, None) == 0
    assert lp(fake, 1, 4, 10, 10, 2, None, None, byref(prm), None, None, 0, None, None) == 1
    # the optional workspace: 16 bytes per row, 16-byte aligned
    assert lib.ls_log_probs_workspace_bytes(3) == 48 and lib.ls_log_probs_workspace_bytes(0) == 0
    assert lp(fake, 1, 4, 10, 10, 2, None, None, byref(prm), fake, fake, 31, None, None) == 1
    assert lp(fake, 1, 4, 10, 10, 2, None, None, byref(prm), fake, P(0x1008), 32, None, None) == 1
    # fused sample + log-probs: the ls_sample checks, and out_ids is required
    f = lib.ls_sample_log_probs
    assert f(fake, 1, 4, 10, 10, -1, None, None, byref(prm), 0, 0, 0, fake, fake, fake, None, 0, None, None) == 1
    assert f(fake, 1, 4, 10, 10, 0, None, None, byref(prm), 0, 0, 0, fake, fake, fake, None, 0, None, None) == 0
    assert f(fake, 1, 4, 10, 10, 2, None, None, byref(prm), 0, 0, 0, None, fake, fake, None, 0, None, None) == 1
    assert f(fake, 1, 4, 10, 10, 5, None, None, byref(prm), 0, 0, 0, fake, fake, fake, None, 0, None, None) == 1
    assert f(fake, 1, 4, 10, 10, 3, None, None, byref(prm2), 0, 0, 0, fake, None, fake, None, 0, None, None) == 1
    assert f(fake, 1, 4, 10, 10, 2, None, None, byref(prm), 0, 0, 0, fake, fake, fake, fake, 16, None, None) == 1
    # the fixed-scratch fused call: more rows than its scratch are refused
    # before any CUDA call; n == 0 launches nothing
    nf = lib.ls_sample_log_probs_noalloc
    assert nf(fake, 1, 5000, 10, 10, 4097, None, None, byref(prm), 0, 0, 0, fake, fake, fake, None, None) == 2
    assert nf(fake, 1, 4, 10, 10, 0, None, None, byref(prm), 0, 0, 0, fake, fake, fake, None, None) == 0
    # device step word: the ls_sample checks, and the step pointer is required
    d = lib.ls_sample_device_step
    assert d(fake, 1, 4, 10, 10, 2, None, None, byref(prm), None, 0, 0, fake, None, None) == 1
    assert d(fake, 1, 4, 10, 10, -1, None, None, byref(prm), fake, 0, 0, fake, None, None) == 1
    assert d(fake, 1, 4, 10, 10, 0, None, None, byref(prm), fake, 0, 0, fake, None, None) == 0
    assert d(fake, 1, 4, 10, 10, 5, None, None, byref(prm), fake, 0, 0, fake, None, None) == 1
    # greedy fast path
    assert lib.ls_argmax(fake, 1, 4, 10, 10, -1, None, fake, None, None) == 1
    assert lib.ls_argmax(fake, 1, 4, 10, 10, 0, None, fake, None, None) == 0
    assert lib.ls_argmax(fake, 1, 4, 10, 10, 2, None, None, None, None) == 1
    assert lib.ls_argmax(fake, 1, 4, 10, 10, 5, None, fake, None, None) == 1
    assert lib.ls_argmax(None, 1, 4, 10, 10, 2, None, fake, None, None) == 1
    # chain verification
    v = lib.ls_verify_chain
    assert v(fake, fake, -1, 2, fake, fake, fake, None) == 1
    assert v(fake, fake, 3, 0, fake, fake, fake, None) == 1
    assert v(fake, fake, 0, 2, fake, fake, fake, None) == 0
    assert v(fake, None, 3, 2, fake, fake, fake, None) == 1
    sv = lib.ls_sample_verify
    assert sv(fake, 1, 100, 10, 10, 2, 3, None, byref(prm), 0, 0, 0, None, fake, fake, fake, fake, None, None) == 1
    assert sv(fake, 1, 100, 10, 10, 5, 3, None, byref(prm), 0, 0, 0, fake, fake, fake, fake, fake, None, None) == 1
    assert sv(fake, 1, 5, 10, 10, 2, 3, None, byref(prm), 0, 0, 0, fake, fake, fake, fake, fake, None, None) == 1
    assert sv(fake, 1, 100, 10, 10, 0, 3, None, byref(prm), 0, 0, 0, fake, fake, fake, fake, fake, None, None) == 0


def test_status_strings(lib):
    for s in range(4):
        assert lib.ls_status_string(s)
    assert b"INVALID" in lib.ls_status_string(1)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from logits_sampling_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "PKG", str(tmp_path))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _binding.load_library()
