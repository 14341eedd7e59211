"""CPU oracle for the paged-KV attention step — TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 NumPy statement of what the step computes: per-head q/k
RMSNorm, RoPE (theta = 1e6), the slot_mapping scatter into the paged cache,
and causal GQA attention read through block tables (decode and varlen
prefill); next to it, the decoder layer's RMSNorm with the residual add
folded in (``add_rms_norm``) and, in ``oracle.block_manager``, a plain model
of the host-side block manager that produces block tables and slot mappings.  It shares no code with the CUDA library and imports nothing from
it.  Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import it; the product path never does.

Sources ("the pages"):
  [NV] "Nano-vLLM深度解读（下）" (devpress.csdn.net) — §2 模型基础 (Qwen3
       model code), §4 与 KV Cache 数据面结合 (attention.py, store kernel).
  [Q3] "同一个 Qwen3，两种写法：从 transformers 到 nano-vllm 的推理改造"
       (violet-quartz.github.io) — §2 config, §2.2 KV-cache sizes, §3.2 flat
       varlen layout, §3.3 paged KV cache, §3.4 attention entry points and
       repeat_kv, §3.5 RoPE, §3.6 RMSNorm with the residual add.

Every function is pinned by tests under ``tests/test_oracle_*.py`` against
values the pages print (``tests/golden/``), closed forms, library routines
(torch SDPA in fp64) and brute force on tiny inputs; the compositions
(``qk_norm_rope``: norm, then RoPE, with the q weight on q and the k weight
on k, at the token's own position) have closed-form pins of their own, and
planted mistakes in each function must fail at least one pin.
"""

from .reference import *  # noqa: F401,F403
from .reference import __all__  # noqa: F401
