"""CUDA-graph replay of the decode step (store + paged decode).

A decode step of a small batch is two short kernels whose launch cost is a
large part of the step.  ``DecodeGraph`` captures ``pkv_qknorm_rope_store``
followed by ``pkv_attn_decode`` once, on fixed device buffers, and replays
the pair as one graph launch; the caller writes each step's q, k, v,
positions, slot_mapping, context_lens and block_table into those buffers
before ``replay()`` (the buffers keep their addresses, so the captured
kernel arguments stay valid).  The pages' model runner replays its decode
step the same way ("同一个 Qwen3，两种写法" §3, Qwen3ForCausalLM: decode takes the
replayed-graph path, which is why forward and compute_logits are separate).

Nothing here computes: the two launches are the library's, captured as they
are issued on the capture stream.
"""

from __future__ import annotations

import torch

from . import ops


class DecodeGraph:
    """Store + decode for a fixed batch shape, captured once and replayed."""

    def __init__(self, q, k, v, positions, slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache, context_lens,
                 block_table, max_context: int, scale: float):
        self.q, self.k, self.v = q, k, v
        self.positions, self.slot_mapping = positions, slot_mapping
        self.q_norm_w, self.k_norm_w = q_norm_w, k_norm_w
        self.k_cache, self.v_cache = k_cache, v_cache
        self.context_lens, self.block_table = context_lens, block_table
        self.max_context, self.scale = int(max_context), float(scale)
        self.out = torch.empty_like(q)
        # everything the launches need is allocated before capture: the RoPE
        # table (per-device state) and the split-K workspace
        ops.init(q.device.index)
        self.workspace = ops.decode_workspace(q.shape[0], self.max_context, q.device)
        self.graph = None

    def _launch(self, stream=None):
        ops.qknorm_rope_store(self.q, self.k, self.v, self.positions, self.slot_mapping, self.q_norm_w,
                              self.k_norm_w, self.k_cache, self.v_cache, stream=stream)
        ops.attn_decode(self.q, self.k_cache, self.v_cache, self.context_lens, self.block_table, self.max_context,
                        self.scale, out=self.out, workspace=self.workspace, stream=stream)

    def eager(self):
        """The same two launches without the graph (one step)."""
        self._launch()
        return self.out

    def capture(self):
        """Capture the step.  The buffers' current contents are used once by
        a warm-up launch outside the graph, so reload them before replaying."""
        side = torch.cuda.Stream(device=self.q.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._launch()  # warm-up: first-use work (kernel loading) stays out of the graph
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize(self.q.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._launch()
        return self

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
        return self.out
