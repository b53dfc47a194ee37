"""GB300 token sampler: thin Python binding of libls_sampler.so.

The binding only marshals arguments (torch tensors -> device pointers, the
current CUDA stream) and calls the C ABI declared in include/ls_sampler.h:
``ls_sample``, ``ls_sample_speculative``, ``ls_log_probs``,
``ls_sample_log_probs``, ``ls_sample_log_probs_noalloc``, ``ls_sample_device_step``,
``ls_argmax``, ``ls_verify_chain``, ``ls_sample_verify``, ``ls_set_split_policy`` and
``ls_set_log_prob_write_policy``.  Every step of the
sampling path runs in the library's CUDA kernels; there is no CPU fallback.
If the library has not been built (``python -m logits_sampling_gb300.build``)
or no CUDA device is present, the calls raise.
"""
from ._binding import (  # noqa: F401
    LS_DTYPE_BF16,
    LS_DTYPE_F32,
    LS_ROW_ERR_BAD_GATHER,
    LS_ROW_ERR_BAD_REQUEST,
    LS_ROW_ERR_NO_FINITE,
    NOALLOC_MAX_ROWS,
    LSError,
    SamplingParams,
    argmax,
    lib_path,
    load_library,
    log_probs,
    max_vocab,
    sample,
    sample_device_step,
    sample_log_probs,
    sample_log_probs_noalloc,
    sample_speculative,
    sample_verify,
    set_log_prob_write_policy,
    set_split_policy,
    status_string,
    verify_chain,
)
