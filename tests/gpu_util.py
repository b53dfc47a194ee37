"""Helpers shared by the GPU parity tests: move a workload to the device, run
the CUDA path through the C ABI, and compare with the CPU oracle under the
parity rules (ids, kept sets and the index mapping bit-exact except on rows the
oracle flags as near-ties; log-probs within 1e-4 absolute, widened only where
float32 cannot hold 1e-4 at the value, to the rounding of the kernel's
arithmetic: see logprob_tolerance)."""
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


def _ulp32(x):
    """Spacing of float32 at |x|, as float64."""
    return np.spacing(np.abs(np.asarray(x, np.float64)).astype(np.float32)).astype(np.float64)


def logprob_tolerance(ref_lp_kept):
    """Per-entry bar for the kept log-probs of one row (oracle values, float64).

    1e-4 absolute wherever float32 holds that resolution.  Beyond it the bar
    is the rounding of the kernel's own arithmetic, which forms
    lp = fl(fl(fl(v - M) / T) - ln S) once |b| = |(v - M) / T| >= 256: the
    subtraction v - M and the correctly rounded division each add at most
    half an ulp of b (one and a half ulps of b once the first error is carried
    through the division), and the final subtraction half an ulp of lp.  (Below
    |b| = 256 the kernel multiplies by RN(1/T) instead, within
    3 2^-24 256 + half an ulp < 1e-4.)  The oracle's b is lp - max(lp) over
    the kept set (the maximum's log-prob is -ln S).  For |lp| below about 500
    the bar is 1e-4."""
    lp = np.asarray(ref_lp_kept, np.float64)
    b = lp - np.max(lp)
    return np.maximum(LOGPROB_ATOL, 1.5 * _ulp32(b) + 0.5 * _ulp32(lp))


def selected_tolerance(ref_sel):
    """Bar for the selected token's raw log-prob l_id - ln sum exp(l): the
    kernel forms fl(fl(v - M) - ln S), half an ulp of |v - M| <= |lp| plus
    half an ulp of lp: 1e-4 absolute, or one float32 ulp of the value."""
    return np.maximum(LOGPROB_ATOL, _ulp32(ref_sel))


def check_ids(gpu_ids, ref, where=""):
    """Bit-exact on unflagged rows.  A row flagged as a score near-tie must
    still give an id of the oracle's kept set; a row flagged as a top-p
    near-tie an id of the loose kept set (the lowest cut a target within the
    1e-5 band allows: the widest set a correct sampler can draw from there).
    Returns the number of flagged rows."""
    ids, flags = ref["ids"], ref["flags"]
    n = len(ids)
    assert gpu_ids.shape == (n,)
    bad = []
    for i in range(n):
        if flags[i] == 0:
            if gpu_ids[i] != ids[i]:
                bad.append((i, int(gpu_ids[i]), int(ids[i])))
            continue
        assert 0 <= gpu_ids[i] < ref["kept"].shape[1], (where, i, int(gpu_ids[i]))
        if flags[i] & oracle.FLAG_TOP_P_TIE:
            assert ref["kept_loose"][i][gpu_ids[i]], (where, i, int(gpu_ids[i]), "outside the loose kept set")
        else:
            assert ref["kept"][i][gpu_ids[i]], (where, i, int(gpu_ids[i]), "outside the kept set")
    assert not bad, f"{where}: {len(bad)} of {n} rows differ, e.g. (row, gpu, oracle) {bad[:8]}"
    return int(np.count_nonzero(flags))


def check_log_probs(gpu_lp, ref, where=""):
    """ref: the oracle's result (lp, kept, kept_loose, kept_tight, flags).
    Kept set (the finite entries) identical, except on rows flagged as top-p
    near-ties, where it must lie between the tight and the loose kept sets;
    -inf exactly outside it; kept log-probs within logprob_tolerance wherever
    the kept sets agree; error rows NaN on both sides."""
    ref_lp, ref_kept, ref_flags = ref["lp"], ref["kept"], ref["flags"]
    n = ref_lp.shape[0]
    for i in range(n):
        if np.all(np.isnan(ref_lp[i])):
            assert np.all(np.isnan(gpu_lp[i])), (where, i)
            continue
        fin = np.isfinite(gpu_lp[i])
        assert np.all(np.isneginf(gpu_lp[i][~fin])), (where, i)
        if not np.array_equal(fin, ref_kept[i]):
            assert ref_flags[i] & oracle.FLAG_TOP_P_TIE, (where, i, np.nonzero(fin != ref_kept[i])[0][:10])
            assert np.all(fin[ref["kept_tight"][i]]) and not np.any(fin & ~ref["kept_loose"][i]), \
                (where, i, "kept set outside the band between the tight and the loose cut")
            continue
        if fin.any():
            ref_v = ref_lp[i][fin]
            tol = logprob_tolerance(ref_v)
            err = np.abs(gpu_lp[i][fin].astype(np.float64) - ref_v)
            assert np.all(err <= tol), (where, i, float(np.max(err - tol)))
