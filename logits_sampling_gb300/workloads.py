"""Seeded synthetic sampler workloads.

This module only draws inputs: random logits of the stated shapes and value
distributions, per-request sampling parameters, gather indices and seeds.  It
holds none of the sampler's arithmetic, so both the CUDA path and the CPU oracle
can take their inputs from it.

The five workloads follow the sampler's serving configurations:

* ``tiny``        4 x 1000 fp32 ~ N(0, 2); T=1, top_k=50, top_p=0.9; joint route.
* ``decode``      64 x 32000 bf16 ~ N(0, 3) plus 5 spikes of +8 per row; per
                  request T ~ U[0.5, 1.5], top_k in {disabled, 20, 50},
                  top_p in {1.0, 0.9, 0.95}; mixed batch -> joint route.
* ``top_p``       256 x 128256 bf16 ~ N(0, 3) with a Zipf(1.1)-shaped head over
                  200 random ids per row; T=0.8, top_k disabled, top_p=0.9;
                  top-p-only route.
* ``speculative`` 128 decode requests x (1 + 4 draft) rows + 32 prefill rows,
                  selected from a 1024 x 151936 bf16 ~ N(0, 3) buffer by random
                  distinct gather indices; per request top_k in {20, 40},
                  top_p=0.95, T=1.0; joint route; plus log-probs.
* ``large``       1024 x 262144 fp32 ~ N(0, 4) with a Zipf head; per request a
                  random mix of no filter / top_k in [1, 128] / top_p in
                  [0.5, 1.0) / both, T ~ U[0.3, 1.5]; joint route; plus log-probs.

Zipf head (reading of "Zipf(1.1)-shaped head"): 200 distinct random ids per
row; the id of rank r (r = 1..200) gets the logit H - 1.1 ln r in place of its
background value, H = 20 when the background sigma is 3 and H = 24 when it is
4.  The second parameter of N(mu, sigma) is read as the standard deviation.
Top-k "disabled" is written as 0 and top-p "disabled" as 1.0.  The Philox seed
of request r is r.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclass
class Workload:
    name: str
    dtype: str                      # "f32" or "bf16"
    logits: np.ndarray              # float32 values, or uint16 bf16 bit patterns, [logits_rows, vocab]
    n: int                          # rows sampled
    temperature: np.ndarray         # float32 [num_requests]
    top_k: np.ndarray               # int32 [num_requests]
    top_p: np.ndarray               # float32 [num_requests]
    seed: np.ndarray                # uint64 [num_requests]
    no_top_k: bool
    no_top_p: bool
    gather_indices: Optional[np.ndarray] = None          # int32 [n]
    token_to_request_index: Optional[np.ndarray] = None  # int32 [n]
    spec: Optional[tuple] = None    # (num_decode, num_prefill, num_speculative_tokens)
    log_probs: bool = False
    step: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def vocab(self):
        return self.logits.shape[1]

    @property
    def logits_rows(self):
        return self.logits.shape[0]

    @property
    def elem_bytes(self):
        return 2 if self.dtype == BF16 else 4

    @property
    def num_requests(self):
        return len(self.temperature)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even, via torch) and return
    the uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _zipf_head(rng, x, head, H):
    rows, V = x.shape
    ranks = np.arange(1, head + 1, dtype=np.float64)
    vals = (H - 1.1 * np.log(ranks)).astype(np.float32)
    for r in range(rows):
        ids = rng.choice(V, size=head, replace=False)
        x[r, ids] = vals


def make_tiny(rows=4, vocab=1000, seed=0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, vocab), dtype=np.float32) * np.float32(2.0)).astype(np.float32)
    return Workload("tiny", F32, x, rows,
                    temperature=np.full(rows, 1.0, np.float32), top_k=np.full(rows, 50, np.int32),
                    top_p=np.full(rows, 0.9, np.float32), seed=np.arange(rows, dtype=np.uint64),
                    no_top_k=False, no_top_p=False, log_probs=True)


def make_decode(rows=64, vocab=32000, seed=1):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, vocab), dtype=np.float32) * np.float32(3.0)).astype(np.float32)
    for r in range(rows):
        ids = rng.choice(vocab, size=5, replace=False)
        x[r, ids] += np.float32(8.0)
    temperature = rng.uniform(0.5, 1.5, rows).astype(np.float32)
    top_k = rng.choice(np.array([0, 20, 50], np.int32), size=rows)
    top_p = rng.choice(np.array([1.0, 0.9, 0.95], np.float32), size=rows)
    return Workload("decode", BF16, to_bf16_bits(x), rows, temperature=temperature, top_k=top_k.astype(np.int32),
                    top_p=top_p.astype(np.float32), seed=np.arange(rows, dtype=np.uint64),
                    no_top_k=bool(np.all(top_k <= 0)), no_top_p=bool(np.all(top_p >= 1.0)))


def make_top_p(rows=256, vocab=128256, seed=2, head=200):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, vocab), dtype=np.float32) * np.float32(3.0)).astype(np.float32)
    _zipf_head(rng, x, min(head, vocab), 20.0)
    return Workload("top_p", BF16, to_bf16_bits(x), rows,
                    temperature=np.full(rows, 0.8, np.float32), top_k=np.zeros(rows, np.int32),
                    top_p=np.full(rows, 0.9, np.float32), seed=np.arange(rows, dtype=np.uint64),
                    no_top_k=True, no_top_p=False)


def make_speculative(buffer_rows=1024, vocab=151936, num_decode=128, num_prefill=32, num_spec=4, seed=3):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((buffer_rows, vocab), dtype=np.float32) * np.float32(3.0)).astype(np.float32)
    n = num_decode * (1 + num_spec) + num_prefill
    assert n <= buffer_rows
    gather = rng.choice(buffer_rows, size=n, replace=False).astype(np.int32)
    nreq = num_decode + num_prefill
    top_k = rng.choice(np.array([20, 40], np.int32), size=nreq).astype(np.int32)
    return Workload("speculative", BF16, to_bf16_bits(x), n,
                    temperature=np.full(nreq, 1.0, np.float32), top_k=top_k,
                    top_p=np.full(nreq, 0.95, np.float32), seed=np.arange(nreq, dtype=np.uint64),
                    no_top_k=False, no_top_p=False, gather_indices=gather,
                    spec=(num_decode, num_prefill, num_spec), log_probs=True)


def make_large(rows=1024, vocab=262144, seed=4, head=200):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, vocab), dtype=np.float32) * np.float32(4.0)).astype(np.float32)
    _zipf_head(rng, x, min(head, vocab), 24.0)
    mode = rng.integers(0, 4, rows)  # 0 none, 1 top-k, 2 top-p, 3 both
    k = rng.integers(1, 129, rows).astype(np.int32)
    p = rng.uniform(0.5, 1.0, rows).astype(np.float32)
    top_k = np.where((mode == 1) | (mode == 3), k, 0).astype(np.int32)
    top_p = np.where((mode == 2) | (mode == 3), p, np.float32(1.0)).astype(np.float32)
    temperature = rng.uniform(0.3, 1.5, rows).astype(np.float32)
    return Workload("large", F32, x, rows, temperature=temperature, top_k=top_k, top_p=top_p,
                    seed=np.arange(rows, dtype=np.uint64), no_top_k=False, no_top_p=False, log_probs=True)


MAKERS = {"tiny": make_tiny, "decode": make_decode, "top_p": make_top_p, "speculative": make_speculative,
          "large": make_large}


def algorithmic_bytes(w: Workload, with_log_probs=False):
    """Bytes one sampling call must move at minimum: the n sampled rows of
    logits, 28 bytes of per-row parameters and indices, and the 4-byte id; the
    log-probs call moves the n rows plus a 4-byte float per entry."""
    sample = w.n * w.vocab * w.elem_bytes + w.n * (28 + 4)
    if with_log_probs:
        return w.n * w.vocab * (w.elem_bytes + 4)
    return sample
