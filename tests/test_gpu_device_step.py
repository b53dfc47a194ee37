"""GPU: the device-resident Philox step word (ls_sample_device_step).  The ids
equal ls_sample's at the step the word held; the word advances by one per call;
a CUDA graph that captured the call draws fresh noise at every replay, where a
captured ls_sample (step passed by value) replays the same ids."""
import numpy as np
import pytest

from logits_sampling_gb300 import workloads as W

from gpu_util import check_ids, oracle_sample, params_of, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the -m gpu tests need a CUDA device")
    import logits_sampling_gb300 as ls
    ls.load_library()


def test_device_step_matches_host_step_and_advances():
    import torch
    import logits_sampling_gb300 as ls
    w = W.make_decode(rows=32, vocab=6000)
    x, prm = to_device(w), params_of(w)
    s0 = (1 << 33) + 5
    step = torch.tensor([s0], dtype=torch.int64, device="cuda")
    got = [ls.sample_device_step(x, w.n, prm, step, w.no_top_k, w.no_top_p).clone() for _ in range(3)]
    want = [ls.sample(x, w.n, prm, s0 + t, w.no_top_k, w.no_top_p) for t in range(3)]
    torch.cuda.synchronize()
    assert int(step.item()) == s0 + 3
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    check_ids(got[1].cpu().numpy(), oracle_sample(w, step=s0 + 1), "device step")
    assert not torch.equal(got[0], got[1])


def test_graph_replay_draws_fresh_noise():
    import torch
    import logits_sampling_gb300 as ls
    w = W.make_top_p(rows=16, vocab=20000)
    w.temperature[:] = 1.5  # flat rows: different steps give different ids
    x, prm = to_device(w), params_of(w)
    step = torch.tensor([100], dtype=torch.int64, device="cuda")
    out = torch.empty(w.n, dtype=torch.int32, device="cuda")
    out_fixed = torch.empty(w.n, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # load the kernels before capturing
        ls.sample(x, w.n, prm, 0, w.no_top_k, w.no_top_p, out=out_fixed)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        ls.sample_device_step(x, w.n, prm, step, w.no_top_k, w.no_top_p, out=out)
        ls.sample(x, w.n, prm, 100, w.no_top_k, w.no_top_p, out=out_fixed)
    torch.cuda.synchronize()
    assert int(step.item()) == 100  # capture launches nothing
    seen, fixed = [], []
    for t in range(3):
        g.replay()
        torch.cuda.synchronize()
        seen.append(out.clone())
        fixed.append(out_fixed.clone())
        assert torch.equal(seen[-1], ls.sample(x, w.n, prm, 100 + t, w.no_top_k, w.no_top_p))
    assert int(step.item()) == 103
    assert all(torch.equal(fixed[0], f) for f in fixed[1:])  # by-value step: the same noise every replay
    assert not torch.equal(seen[0], seen[1]) and not torch.equal(seen[1], seen[2])
    check_ids(seen[2].cpu().numpy(), oracle_sample(w, step=102), "graph replay")
