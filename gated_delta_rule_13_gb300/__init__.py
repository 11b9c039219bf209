"""GB300-native (sm_103a) KDA recurrence: chunked prefill, in-place decode and
replay of accepted speculative-decode tokens.

The compute lives in ``libkda.so`` (hand-written CUDA kernels behind a C ABI,
``include/kda.h``); ``kda`` is its thin Python binding.
"""
from .kda import (KDAError, kda_chunk_fwd, kda_chunk_fwd_host, kda_chunk_fwd_noalloc,
                  kda_chunk_fwd_transitions,
                  kda_chunk_fwd_workspace_size, kda_decode_replay, kda_decode_step,
                  kda_post_fwd, kda_prep_fwd, kda_read_chunk_stats, kda_read_device_status,
                  kda_state_combine, kda_version, library, library_path)

__all__ = ["KDAError", "kda_chunk_fwd", "kda_chunk_fwd_host", "kda_chunk_fwd_noalloc", "kda_chunk_fwd_transitions",
           "kda_chunk_fwd_workspace_size", "kda_decode_replay", "kda_decode_step",
           "kda_post_fwd", "kda_prep_fwd", "kda_read_chunk_stats", "kda_read_device_status",
           "kda_state_combine", "kda_version", "library", "library_path"]
