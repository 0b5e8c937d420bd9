"""Hybrid long-context attention (sliding window + CSA / HCA) for NVIDIA B300.

The compute lives in libhybridattn.so (hand-written CUDA for sm_103a, C ABI in
include/hybrid_attn.h); `binding` marshals torch tensors into those calls,
`cache_state` turns appends of tokens into the compressor's arguments, and
`synth` makes the seeded synthetic inputs of the benchmark workloads.
"""
from . import binding  # noqa: F401
from .binding import (HAError, Params, make_params, hca_compress_kv, csa_compress_kv,  # noqa: F401
                      csa_index_scores, csa_topk, hybrid_attn_decode, hybrid_attn_prefill,
                      ha_workspace_size)
from .cache_state import CacheState  # noqa: F401
