"""mlp_latency_gb300 -- CTA-pipelined GEMM chains on one GB300 (sm_103a).

The compute path is libmlp_chain.so (hand-written tcgen05/TMA CUDA, C ABI in
include/mlp_chain.h); this package only builds it and marshals arguments to it.
"""
from ._lib import build, load, LIB_PATH  # noqa: F401
from .chain import (Chain, MlpChainError, deps_build, protocol_model, scoreboard_build, EVENT_DTYPE,  # noqa: F401
                    OK, ERR_TIMEOUT, ERR_BAD_TILE, ERR_INVALID_ARG, ERR_UNSUPPORTED)
