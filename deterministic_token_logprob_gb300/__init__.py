"""deterministic_token_logprob_gb300 -- deterministic, batch-invariant `linear_logp` on GB300.

The operator returns logp[t] = h_t . W_{y_t} - logsumexp_{v < V_true}(h_t . W_v)
(fp32) without materialising the [T, V] logits, plus dH / dW of
sum_t g_t logp_t. It is a C ABI shared library (include/rlk.h, built into
``_build/librlk.so`` from ``csrc/``) with hand-written sm_103a kernels
(tcgen05 / TMEM / TMA); this package is its thin ctypes binding.
"""
from ._binding import (  # noqa: F401
    LEAF_WIDTH, MAX_SHARDS, RLK_BWD_DH, RLK_BWD_DW, RLK_BWD_DZ, RLK_ERR_CUDA, RLK_ERR_INVALID_ARG,
    RLK_ERR_UNSUPPORTED, RLK_ERR_WORKSPACE, RLK_FLAG_BAD_TARGET, RLK_FLAG_BOUNDS, RLK_FLAG_NONFINITE,
    RLK_FLAG_TIMEOUT, RLK_OK, RlkError, bwd_workspace_bytes, debug_checks, fwd_workspace_bytes, lib,
    library, library_path, linear_logp_bwd, linear_logp_bwd_fp8, linear_logp_bwd_saved,
    linear_logp_bwd_saved_probs, linear_logp_fwd, linear_logp_fwd_fp8, linear_logp_fwd_save,
    linear_logp_fwd_save_probs, lse_merge, quantize_rows_e4m3, saved_logits_buffer,
    saved_logits_bytes, saved_probs_bytes, selftest_bounds_check, selftest_wait_timeout,
    shard_bounds, shard_sum_bf16, version)
from .autograd import LinearLogp, linear_logp  # noqa: F401
