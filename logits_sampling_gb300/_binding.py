"""ctypes binding of include/ls_sampler.h (argument marshalling only)."""
import ctypes
import os
from dataclasses import dataclass

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libls_sampler.so"

LS_OK, LS_ERR_INVALID_ARG, LS_ERR_UNSUPPORTED, LS_ERR_CUDA = 0, 1, 2, 3
LS_DTYPE_F32, LS_DTYPE_BF16 = 0, 1
LS_ROW_ERR_BAD_GATHER, LS_ROW_ERR_BAD_REQUEST, LS_ROW_ERR_NO_FINITE = 1, 2, 4

_lib = None


class LSError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


class _Params(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_void_p), ("top_k", ctypes.c_void_p), ("top_p", ctypes.c_void_p),
                ("seed", ctypes.c_void_p), ("num_requests", ctypes.c_int32)]


def lib_path():
    return os.path.join(PKG, LIB_NAME)


def load_library():
    """Load libls_sampler.so from the package directory (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m logits_sampling_gb300.build` "
                           "(there is no CPU fallback)")
    _lib = configure(ctypes.CDLL(path))
    return _lib


def configure(lib):
    """Declare the C signatures of include/ls_sampler.h on a loaded library
    (the package's own, or a test-only variant build of the same sources)."""
    P, i32, i64, u64, ci = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
    PP = ctypes.POINTER(_Params)
    lib.ls_sample.argtypes = [P, ci, i64, i64, i64, i32, P, P, PP, u64, ci, ci, P, P, P]
    lib.ls_sample.restype = ci
    lib.ls_sample_speculative.argtypes = [P, ci, i64, i64, i64, i32, i32, i32, P, PP, u64, ci, ci, P, P, P, P]
    lib.ls_sample_speculative.restype = ci
    sz = ctypes.c_size_t
    lib.ls_log_probs.argtypes = [P, ci, i64, i64, i64, i32, P, P, PP, P, P, sz, P, P]
    lib.ls_log_probs.restype = ci
    lib.ls_log_probs_workspace_bytes.argtypes = [i32]
    lib.ls_log_probs_workspace_bytes.restype = sz
    lib.ls_sample_log_probs.argtypes = [P, ci, i64, i64, i64, i32, P, P, PP, u64, ci, ci, P, P, P, P, sz, P, P]
    lib.ls_sample_log_probs.restype = ci
    lib.ls_sample_log_probs_noalloc.argtypes = [P, ci, i64, i64, i64, i32, P, P, PP, u64, ci, ci, P, P, P, P, P]
    lib.ls_sample_log_probs_noalloc.restype = ci
    lib.ls_set_log_prob_write_policy.argtypes = [ci]
    lib.ls_set_log_prob_write_policy.restype = ci
    lib.ls_sample_device_step.argtypes = [P, ci, i64, i64, i64, i32, P, P, PP, P, ci, ci, P, P, P]
    lib.ls_sample_device_step.restype = ci
    lib.ls_argmax.argtypes = [P, ci, i64, i64, i64, i32, P, P, P, P]
    lib.ls_argmax.restype = ci
    lib.ls_verify_chain.argtypes = [P, P, i32, i32, P, P, P, P]
    lib.ls_verify_chain.restype = ci
    lib.ls_sample_verify.argtypes = [P, ci, i64, i64, i64, i32, i32, P, PP, u64, ci, ci, P, P, P, P, P, P, P]
    lib.ls_sample_verify.restype = ci
    lib.ls_status_string.argtypes = [ci]
    lib.ls_status_string.restype = ctypes.c_char_p
    lib.ls_max_vocab.argtypes = [ci]
    lib.ls_max_vocab.restype = i64
    lib.ls_set_split_policy.argtypes = [ci]
    lib.ls_set_split_policy.restype = ci
    return lib


def status_string(status):
    try:
        return load_library().ls_status_string(int(status)).decode()
    except Exception:  # pragma: no cover
        return f"status {status}"


def max_vocab(dtype=LS_DTYPE_BF16):
    return int(load_library().ls_max_vocab(dtype))


def set_log_prob_write_policy(policy):
    """ls_set_log_prob_write_policy: 0 from the batch shape, 1 the tiled write
    kernel, -1 the row kernel's own write (calls with a workspace)."""
    st = load_library().ls_set_log_prob_write_policy(int(policy))
    if st != LS_OK:
        raise LSError(st, f"ls_set_log_prob_write_policy({policy})")


def set_split_policy(ctas_per_row):
    """ls_set_split_policy: 0 = per-call choice from the batch shape; 1, 2, 4, 8
    = the streaming sampler with that many CTAs per row; -1 = the one-CTA row
    kernel.  Applies to every later sampling call of the process."""
    st = load_library().ls_set_split_policy(int(ctas_per_row))
    if st != LS_OK:
        raise LSError(st, "ls_set_split_policy")


@dataclass
class SamplingParams:
    """Per-request parameters as device tensors (float32 temperature, int32
    top_k, float32 top_p, int64/uint64 seed), all of length num_requests."""
    temperature: object
    top_k: object
    top_p: object
    seed: object = None

    def as_struct(self):
        n = int(self.temperature.numel())
        for name in ("top_k", "top_p", "seed"):
            t = getattr(self, name)
            if t is not None and int(t.numel()) != n:
                raise ValueError(f"{name} has {t.numel()} entries, temperature has {n}")
        import torch
        if self.temperature.dtype != torch.float32 or self.top_p.dtype != torch.float32:
            raise TypeError("temperature and top_p must be float32")
        if self.top_k.dtype != torch.int32:
            raise TypeError("top_k must be int32")
        if self.seed is not None and self.seed.dtype not in (torch.int64, torch.uint64):
            raise TypeError("seed must be int64 or uint64")
        return _Params(_dptr(self.temperature), _dptr(self.top_k), _dptr(self.top_p),
                       _dptr(self.seed) if self.seed is not None else None, n)

    @staticmethod
    def from_host(temperature, top_k, top_p, seed, device="cuda"):
        import numpy as np
        import torch
        return SamplingParams(
            torch.from_numpy(np.ascontiguousarray(temperature, np.float32)).to(device),
            torch.from_numpy(np.ascontiguousarray(top_k, np.int32)).to(device),
            torch.from_numpy(np.ascontiguousarray(top_p, np.float32)).to(device),
            torch.from_numpy(np.ascontiguousarray(seed, np.uint64).view(np.int64)).to(device))


def _dptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _logits_desc(logits):
    import torch
    if logits.dim() != 2:
        raise ValueError("logits must be 2-D [rows, vocab]")
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")
    if logits.dtype == torch.float32:
        dt = LS_DTYPE_F32
    elif logits.dtype == torch.bfloat16:
        dt = LS_DTYPE_BF16
    else:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    return ctypes.c_void_p(logits.data_ptr()), dt, logits.shape[0], logits.shape[1], logits.stride(0)


def _i32(t, what):
    import torch
    if t is None:
        return None
    if t.dtype != torch.int32:
        raise TypeError(f"{what} must be int32")
    return _dptr(t)


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _on(stream):
    """The stream a call runs on (the current stream when None) and a context
    that makes it current: outputs and temporaries are allocated and filled on
    the stream the kernels use, so an explicit stream never races with the
    call's own set-up, and the caching allocator reuses their memory only in
    that stream's order."""
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s, torch.cuda.stream(s)


def sample(logits, n, params, step, no_top_k, no_top_p, gather_indices=None, token_to_request_index=None,
           out=None, error_word=None, stream=None):
    """ls_sample: returns out (int32 [n] on the logits' device)."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=logits.device)
        prm = params.as_struct()
        st = lib.ls_sample(ptr, dt, rows, V, stride, int(n), _i32(gather_indices, "gather_indices"),
                           _i32(token_to_request_index, "token_to_request_index"), ctypes.byref(prm), int(step),
                           int(bool(no_top_k)), int(bool(no_top_p)), _i32(out, "out"),
                           _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_sample")
    return out


def sample_speculative(required_logits, num_decode, num_prefill, num_speculative_tokens, params, step, no_top_k,
                       no_top_p, gather_indices=None, out=None, out_token_to_request_index=None, error_word=None,
                       stream=None):
    """ls_sample_speculative: returns out (int32 [num_decode*(1+S)+num_prefill])."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(required_logits)
    n = num_decode * (1 + num_speculative_tokens) + num_prefill
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=required_logits.device)
        prm = params.as_struct()
        st = lib.ls_sample_speculative(ptr, dt, rows, V, stride, int(num_decode), int(num_prefill),
                                       int(num_speculative_tokens), _i32(gather_indices, "gather_indices"),
                                       ctypes.byref(prm), int(step), int(bool(no_top_k)), int(bool(no_top_p)),
                                       _i32(out, "out"),
                                       _i32(out_token_to_request_index, "out_token_to_request_index"),
                                       _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_sample_speculative")
    return out


# Rows of ls_sample_log_probs_noalloc's fixed scratch (LS_NOALLOC_MAX_ROWS).
NOALLOC_MAX_ROWS = 4096

# Default of the log-prob calls' `workspace` argument (True: allocate one).
LOG_PROBS_WORKSPACE = True


def _workspace(lib, n, device, workspace):
    """The log-prob calls' optional workspace: True allocates one (on the
    current stream), False passes none (the row kernel then writes the rows
    itself), None takes LOG_PROBS_WORKSPACE, or a caller's tensor.  Returns
    (tensor or None, bytes)."""
    import torch
    if workspace is None:
        workspace = LOG_PROBS_WORKSPACE
    if workspace is False:
        return None, 0
    if workspace is True:
        nbytes = int(lib.ls_log_probs_workspace_bytes(int(n)))
        workspace = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def log_probs(logits, params, num_rows=None, gather_indices=None, token_to_request_index=None, out=None,
              error_word=None, stream=None, workspace=None):
    """ls_log_probs: returns out (float32 [num_rows, vocab])."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    if num_rows is None:
        num_rows = len(gather_indices) if gather_indices is not None else rows
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty((num_rows, V), dtype=torch.float32, device=logits.device)
        if out.dtype != torch.float32 or not out.is_contiguous() or out.numel() < num_rows * V:
            raise ValueError("out must be a contiguous float32 tensor of num_rows * vocab entries")
        prm = params.as_struct()
        ws, wsb = _workspace(lib, num_rows, logits.device, workspace)
        st = lib.ls_log_probs(ptr, dt, rows, V, stride, int(num_rows), _i32(gather_indices, "gather_indices"),
                              _i32(token_to_request_index, "token_to_request_index"), ctypes.byref(prm),
                              _dptr(out), _dptr(ws), wsb, _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_log_probs")
    return out


def sample_log_probs(logits, n, params, step, no_top_k, no_top_p, gather_indices=None, token_to_request_index=None,
                     want_log_probs=True, want_selected=True, out=None, out_log_probs=None, out_selected=None,
                     error_word=None, stream=None, workspace=None):
    """ls_sample_log_probs: returns (ids int32 [n], log_probs float32 [n, vocab] or None,
    selected float32 [n] or None) from one read of the logits."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=logits.device)
        if want_log_probs and out_log_probs is None:
            out_log_probs = torch.empty((n, V), dtype=torch.float32, device=logits.device)
        if want_selected and out_selected is None:
            out_selected = torch.empty(n, dtype=torch.float32, device=logits.device)
        if not want_log_probs:
            out_log_probs = None
        if not want_selected:
            out_selected = None
        if out_log_probs is not None and (out_log_probs.dtype != torch.float32
                                          or not out_log_probs.is_contiguous() or out_log_probs.numel() < n * V):
            raise ValueError("out_log_probs must be a contiguous float32 tensor of n * vocab entries")
        if out_selected is not None and (out_selected.dtype != torch.float32 or out_selected.numel() < n):
            raise ValueError("out_selected must be a float32 tensor of n entries")
        prm = params.as_struct()
        ws, wsb = _workspace(lib, n, logits.device, workspace if out_log_probs is not None else False)
        st = lib.ls_sample_log_probs(ptr, dt, rows, V, stride, int(n), _i32(gather_indices, "gather_indices"),
                                     _i32(token_to_request_index, "token_to_request_index"), ctypes.byref(prm),
                                     int(step), int(bool(no_top_k)), int(bool(no_top_p)), _i32(out, "out"),
                                     _dptr(out_log_probs), _dptr(out_selected), _dptr(ws), wsb,
                                     _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_sample_log_probs")
    return out, out_log_probs, out_selected


def sample_log_probs_noalloc(logits, n, params, step, no_top_k, no_top_p, gather_indices=None,
                             token_to_request_index=None, out=None, out_log_probs=None, out_selected=None,
                             error_word=None, stream=None):
    """ls_sample_log_probs_noalloc: as sample_log_probs with both outputs,
    the outputs given or allocated here; the library's fixed scratch replaces
    the workspace (n at most LS_NOALLOC_MAX_ROWS; calls in flight together
    race on it)."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=logits.device)
        if out_log_probs is None:
            out_log_probs = torch.empty((n, V), dtype=torch.float32, device=logits.device)
        if out_selected is None:
            out_selected = torch.empty(n, dtype=torch.float32, device=logits.device)
        prm = params.as_struct()
        st = lib.ls_sample_log_probs_noalloc(ptr, dt, rows, V, stride, int(n), _i32(gather_indices, "gather_indices"),
                                             _i32(token_to_request_index, "token_to_request_index"),
                                             ctypes.byref(prm), int(step), int(bool(no_top_k)), int(bool(no_top_p)),
                                             _i32(out, "out"), _dptr(out_log_probs), _dptr(out_selected),
                                             _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, f"ls_sample_log_probs_noalloc (n = {n}; at most {NOALLOC_MAX_ROWS} rows)")
    return out, out_log_probs, out_selected


def sample_device_step(logits, n, params, step, no_top_k, no_top_p, gather_indices=None,
                       token_to_request_index=None, out=None, error_word=None, stream=None):
    """ls_sample_device_step: `step` is a device int64/uint64 tensor of one
    element, read by the call and advanced by one on the device (graph-safe).
    Returns out (int32 [n])."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    if step.dtype not in (torch.int64, torch.uint64) or step.numel() != 1:
        raise TypeError("step must be a one-element int64/uint64 device tensor")
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=logits.device)
        prm = params.as_struct()
        st = lib.ls_sample_device_step(ptr, dt, rows, V, stride, int(n), _i32(gather_indices, "gather_indices"),
                                       _i32(token_to_request_index, "token_to_request_index"), ctypes.byref(prm),
                                       _dptr(step), int(bool(no_top_k)), int(bool(no_top_p)), _i32(out, "out"),
                                       _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_sample_device_step")
    return out


def argmax(logits, n=None, gather_indices=None, out=None, error_word=None, stream=None):
    """ls_argmax: the lowest index of each row's maximum (all-greedy batches).
    Returns out (int32 [n])."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    if n is None:
        n = len(gather_indices) if gather_indices is not None else rows
    s, ctx = _on(stream)
    with ctx:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=logits.device)
        st = lib.ls_argmax(ptr, dt, rows, V, stride, int(n), _i32(gather_indices, "gather_indices"),
                           _i32(out, "out"), _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_argmax")
    return out


def verify_chain(candidates, target_sampled, predicts=None, accept_index=None, accept_token_num=None, stream=None):
    """ls_verify_chain: candidates int32 [bs, n] and target_sampled int32 [bs * n]
    on the device.  Returns (predicts [bs * n], accept_index [bs, n],
    accept_token_num [bs])."""
    import torch
    lib = load_library()
    bs, n = candidates.shape
    dev = candidates.device
    s, ctx = _on(stream)
    with ctx:
        if predicts is None:
            predicts = torch.full((bs * n,), -1, dtype=torch.int32, device=dev)
        if accept_index is None:
            accept_index = torch.empty((bs, n), dtype=torch.int32, device=dev)
        if accept_token_num is None:
            accept_token_num = torch.empty(bs, dtype=torch.int32, device=dev)
        cand = candidates.contiguous()
        st = lib.ls_verify_chain(_i32(cand, "candidates"), _i32(target_sampled, "target_sampled"),
                                 int(bs), int(n), _i32(predicts, "predicts"), _i32(accept_index, "accept_index"),
                                 _i32(accept_token_num, "accept_token_num"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_verify_chain")
    return predicts, accept_index, accept_token_num


def sample_verify(logits, candidates, params, step, no_top_k, no_top_p, gather_indices=None, error_word=None,
                  stream=None):
    """ls_sample_verify: sample the bs * n verify rows, then verify the chains.
    Returns (target_sampled, predicts, accept_index, accept_token_num)."""
    import torch
    lib = load_library()
    ptr, dt, rows, V, stride = _logits_desc(logits)
    bs, n = candidates.shape
    dev = logits.device
    s, ctx = _on(stream)
    with ctx:
        target = torch.empty(bs * n, dtype=torch.int32, device=dev)
        predicts = torch.full((bs * n,), -1, dtype=torch.int32, device=dev)
        accept_index = torch.empty((bs, n), dtype=torch.int32, device=dev)
        accept_token_num = torch.empty(bs, dtype=torch.int32, device=dev)
        cand = candidates.contiguous()
        prm = params.as_struct()
        st = lib.ls_sample_verify(ptr, dt, rows, V, stride, int(bs), int(n),
                                  _i32(gather_indices, "gather_indices"), ctypes.byref(prm), int(step),
                                  int(bool(no_top_k)), int(bool(no_top_p)), _i32(cand, "candidates"),
                                  _i32(target, "target"), _i32(predicts, "predicts"),
                                  _i32(accept_index, "accept_index"), _i32(accept_token_num, "accept_token_num"),
                                  _i32(error_word, "error_word"), _stream(s))
    if st != LS_OK:
        raise LSError(st, "ls_sample_verify")
    return target, predicts, accept_index, accept_token_num
