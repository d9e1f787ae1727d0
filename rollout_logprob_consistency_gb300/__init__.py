"""Batch-invariant linear logprob and three-way score comparison for GB300 (sm_103a).

The compute runs in ``libtim.so`` (hand-written CUDA for sm_103a, C ABI in
``include/tim.h``); ``binding`` marshals torch tensors into it.  Build with
``rollout_logprob_consistency_gb300.build.build()``.
"""
from .binding import (  # noqa: F401
    TimError, Workspace, compare, compare_diag, compare_workspace_size, diag_to_dicts, lib,
    logprob, logprob_stages, logprob_workspace_size, stats_to_dicts, SEQ_DIAG_DTYPE,
    SEQ_STATS_DTYPE, STATUS, STATUS_NAMES, vocab_shard, logprob_shard, logprob_merge_shards,
    gather_shard_records, logprob_vocab_parallel, logprob_vocab_parallel_emulated,
    processed_logprob, quantize_fp8_rows, logprob_fp8, split_tf32, logprob_fp32,
    logprob_backward, selftest_wait_timeout, rmsnorm_backward, linear_logprob,
    logprob_noalloc,
)
