"""Helpers shared by the GPU parity tests: move a workload to the device, run
the CUDA path through the C ABI, and compare with the CPU oracle under the
parity rules (ids, kept sets and the index mapping bit-exact except on rows the
oracle flags as near-ties; log-probs within 1e-4 absolute, or two float32 ulps
where the value is too large for float32 to resolve 1e-4)."""
import numpy as np

import oracle
from logits_sampling_gb300 import workloads as W

LOGPROB_ATOL = 1e-4


def odt(w):
    return oracle.DTYPE_BF16 if w.dtype == W.BF16 else oracle.DTYPE_F32


def to_device(w):
    import torch
    if w.dtype == W.BF16:
        x = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16)
    else:
        x = torch.from_numpy(w.logits)
    return x.cuda()


def params_of(w):
    from logits_sampling_gb300 import SamplingParams
    return SamplingParams.from_host(w.temperature, w.top_k, w.top_p, w.seed)


def gpu_sample(w, logits_dev=None, route=None, step=None, t2r=None):
    import torch
    import logits_sampling_gb300 as ls
    x = to_device(w) if logits_dev is None else logits_dev
    nk, np_ = (w.no_top_k, w.no_top_p) if route is None else route
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = w.step if step is None else step
    if w.spec is not None and t2r is None:
        D, P, S = w.spec
        g = None if w.gather_indices is None else torch.from_numpy(w.gather_indices).cuda()
        mp = torch.full((w.n,), -7, dtype=torch.int32, device="cuda")
        ids = ls.sample_speculative(x, D, P, S, params_of(w), step, nk, np_, gather_indices=g,
                                    out_token_to_request_index=mp, error_word=err)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), int(err.item()), mp.cpu().numpy()
    g = None if w.gather_indices is None else torch.from_numpy(w.gather_indices).cuda()
    tt = w.token_to_request_index if t2r is None else t2r
    t = None if tt is None else torch.from_numpy(np.ascontiguousarray(tt, np.int32)).cuda()
    ids = ls.sample(x, w.n, params_of(w), step, nk, np_, gather_indices=g, token_to_request_index=t,
                    error_word=err)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), int(err.item()), None


def gpu_log_probs(w, logits_dev=None, gather=None, t2r=None, num_rows=None):
    import torch
    import logits_sampling_gb300 as ls
    x = to_device(w) if logits_dev is None else logits_dev
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = None if gather is None else torch.from_numpy(np.ascontiguousarray(gather, np.int32)).cuda()
    t = None if t2r is None else torch.from_numpy(np.ascontiguousarray(t2r, np.int32)).cuda()
    out = ls.log_probs(x, params_of(w), num_rows=num_rows, gather_indices=g, token_to_request_index=t,
                       error_word=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def oracle_mapping(w):
    if w.spec is not None:
        return oracle.speculative_mapping(*w.spec)
    return w.token_to_request_index


def oracle_sample(w, step=None, route=None, want_kept=True):
    nk, np_ = (w.no_top_k, w.no_top_p) if route is None else route
    return oracle.sample(w.logits, odt(w), w.n, w.temperature, w.top_k, w.top_p, w.seed,
                         step=w.step if step is None else step, no_top_k=nk, no_top_p=np_,
                         gather_indices=w.gather_indices, token_to_request_index=oracle_mapping(w),
                         want_kept=want_kept)


def check_ids(gpu_ids, ref, where=""):
    """Bit-exact on unflagged rows; flagged rows must still give a kept id
    (score near-tie) or a valid id (top-p near-tie).  Returns #flagged rows."""
    ids, flags = ref["ids"], ref["flags"]
    n = len(ids)
    assert gpu_ids.shape == (n,)
    bad = []
    for i in range(n):
        if flags[i] == 0:
            if gpu_ids[i] != ids[i]:
                bad.append((i, int(gpu_ids[i]), int(ids[i])))
        elif flags[i] & oracle.FLAG_TOP_P_TIE:
            assert 0 <= gpu_ids[i] < ref["kept"].shape[1], (where, i)
        else:
            assert ref["kept"][i][gpu_ids[i]], (where, i, int(gpu_ids[i]))
    assert not bad, f"{where}: {len(bad)} of {n} rows differ, e.g. (row, gpu, oracle) {bad[:8]}"
    return int(np.count_nonzero(flags))


def check_log_probs(gpu_lp, ref_lp, ref_kept, ref_flags, where=""):
    """Kept set (finite entries) identical on rows without a top-p near-tie;
    finite log-probs within LOGPROB_ATOL; error rows NaN on both sides."""
    n = ref_lp.shape[0]
    for i in range(n):
        if np.all(np.isnan(ref_lp[i])):
            assert np.all(np.isnan(gpu_lp[i])), (where, i)
            continue
        fin = np.isfinite(gpu_lp[i])
        if not (ref_flags[i] & oracle.FLAG_TOP_P_TIE):
            diff = np.nonzero(fin != ref_kept[i])[0]
            assert diff.size == 0, (where, i, diff[:10])
            assert np.all(np.isneginf(gpu_lp[i][~fin])), (where, i)
        both = fin & ref_kept[i]
        if both.any():
            ref = ref_lp[i][both]
            # 1e-4 absolute; for |lp| beyond ~800 the float32 output itself cannot
            # resolve 1e-4, so there the bar is two float32 ulps of the value.
            tol = np.maximum(LOGPROB_ATOL, 2.0 * np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64))
            err = np.abs(gpu_lp[i][both].astype(np.float64) - ref)
            assert np.all(err <= tol), (where, i, float(np.max(err - tol)))
