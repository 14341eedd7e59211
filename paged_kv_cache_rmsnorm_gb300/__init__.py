"""GB300 (sm_103a) paged-KV attention step for Qwen3-style attention.

Three calls, each a C-ABI entry point of libpkv.so (include/pkv.h) backed by
hand-written CUDA kernels:

* ``qknorm_rope_store`` — per-head q/k RMSNorm + RoPE (theta 1e6) + the
  slot_mapping scatter of K/V into the 256-token-block cache;
* ``attn_decode`` — split-K paged GQA decode attention;
* ``attn_prefill`` — causal varlen paged GQA prefill attention.

Next to the step: ``add_rmsnorm`` — the decoder layer's RMSNorm over the
hidden size with the pending residual add folded in; ``qkv_rope_store`` —
the QKV projection on tcgen05 with ``qknorm_rope_store``'s work as its
epilogue.
"""

from ._build import LIB_PATH, build, library_is_fresh  # noqa: F401
from .ops import (  # noqa: F401
    BLOCK_SIZE,
    HEAD_DIM,
    MAX_POSITION,
    NUM_KV_HEADS,
    NUM_Q_HEADS,
    HIDDEN,
    PkvError,
    QKV_OUT,
    add_rmsnorm,
    qkv_rope_store,
    attn_decode,
    attn_decode_noalloc,
    attn_prefill,
    check_errors,
    decode_workspace,
    decode_workspace_size,
    init,
    load_library,
    qknorm_rope_store,
)
