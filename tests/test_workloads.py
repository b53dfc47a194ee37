"""The seeded workload generators against the input recipe they state: shapes,
dtypes, value distributions and per-request parameters.  Small instances
(same makers, reduced sizes) stand in for the full-size ones, whose default
sizes are checked from the makers' signatures."""
import inspect

import numpy as np

from logits_sampling_gb300 import workloads as W


def _values(w):
    if w.dtype == W.BF16:
        return (w.logits.astype(np.uint32) << 16).view(np.float32)
    return w.logits


def _defaults(fn):
    return {k: v.default for k, v in inspect.signature(fn).parameters.items()}


def test_full_size_defaults():
    assert _defaults(W.make_tiny) == {"rows": 4, "vocab": 1000, "seed": 0}
    assert _defaults(W.make_decode) == {"rows": 64, "vocab": 32000, "seed": 1}
    assert _defaults(W.make_top_p) == {"rows": 256, "vocab": 128256, "seed": 2, "head": 200}
    assert _defaults(W.make_speculative) == {"buffer_rows": 1024, "vocab": 151936, "num_decode": 128,
                                             "num_prefill": 32, "num_spec": 4, "seed": 3}
    assert _defaults(W.make_large) == {"rows": 1024, "vocab": 262144, "seed": 4, "head": 200}
    assert set(W.MAKERS) == {"tiny", "decode", "top_p", "speculative", "large"}


def test_tiny():
    w = W.make_tiny()
    assert w.dtype == W.F32 and w.logits.shape == (4, 1000) and w.n == 4
    assert np.all(w.temperature == 1.0) and np.all(w.top_k == 50) and np.all(w.top_p == np.float32(0.9))
    assert not w.no_top_k and not w.no_top_p
    assert abs(float(np.std(w.logits)) - 2.0) < 0.1
    np.testing.assert_array_equal(w.seed, np.arange(4, dtype=np.uint64))


def test_decode():
    w = W.make_decode()
    x = _values(w)
    assert w.dtype == W.BF16 and x.shape == (64, 32000) and w.n == 64
    assert np.all((w.temperature >= 0.5) & (w.temperature <= 1.5))
    assert set(np.unique(w.top_k).tolist()) <= {0, 20, 50}
    assert set(np.unique(w.top_p).tolist()) <= {np.float32(1.0), np.float32(0.9), np.float32(0.95)}
    # background N(0, 3): the median absolute value of N(0, s) is 0.6745 s
    assert abs(float(np.median(np.abs(x))) / 0.6745 - 3.0) < 0.05


def test_top_p_head():
    w = W.make_top_p(rows=8, vocab=4096)
    x = _values(w)
    assert w.dtype == W.BF16 and x.shape == (8, 4096)
    assert np.all(w.temperature == np.float32(0.8)) and np.all(w.top_k == 0) and np.all(w.top_p == np.float32(0.9))
    assert w.no_top_k and not w.no_top_p
    # the Zipf head: rank r holds H - 1.1 ln r with H = 20 (bf16-rounded)
    head = np.sort(x, axis=1)[:, ::-1][:, :3]
    want = W.to_bf16_bits((20.0 - 1.1 * np.log(np.arange(1, 4))).astype(np.float32)[None, :])
    np.testing.assert_array_equal(W.to_bf16_bits(head), np.broadcast_to(want, head.shape))


def test_speculative_layout():
    w = W.make_speculative(buffer_rows=64, vocab=512, num_decode=8, num_prefill=4, num_spec=4)
    assert w.dtype == W.BF16 and w.logits.shape == (64, 512)
    assert w.spec == (8, 4, 4) and w.n == 8 * 5 + 4
    g = w.gather_indices
    assert g.dtype == np.int32 and len(np.unique(g)) == w.n and g.min() >= 0 and g.max() < 64
    assert len(w.top_k) == 12 and set(np.unique(w.top_k).tolist()) <= {20, 40}
    assert np.all(w.top_p == np.float32(0.95)) and np.all(w.temperature == 1.0)


def test_large_mix():
    w = W.make_large(rows=256, vocab=2048)
    x = _values(w)
    assert w.dtype == W.F32 and x.shape == (256, 2048)
    k_on = w.top_k > 0
    p_on = w.top_p < 1.0
    assert np.all((w.top_k[k_on] >= 1) & (w.top_k[k_on] <= 128))
    assert np.all((w.top_p[p_on] >= 0.5) & (w.top_p[p_on] < 1.0))
    assert np.all((w.temperature >= 0.3) & (w.temperature <= 1.5))
    # all four per-request modes occur
    assert {(a, b) for a, b in zip(k_on.tolist(), p_on.tolist())} == {(False, False), (True, False),
                                                                      (False, True), (True, True)}
    assert np.all(x.max(axis=1) == np.float32(24.0))


def test_algorithmic_bytes_of_the_headline_workload():
    w = W.Workload("top_p", W.BF16, np.empty((256, 128256), np.uint16), 256,
                   temperature=np.ones(256, np.float32), top_k=np.zeros(256, np.int32),
                   top_p=np.full(256, 0.9, np.float32), seed=np.arange(256, dtype=np.uint64),
                   no_top_k=True, no_top_p=False)
    # the sampled rows once, 28 bytes of parameters and indices and a 4-byte id per row
    assert W.algorithmic_bytes(w) == 256 * 128256 * 2 + 256 * 32
    assert W.algorithmic_bytes(w, with_log_probs=True) == 256 * 128256 * (2 + 4)
