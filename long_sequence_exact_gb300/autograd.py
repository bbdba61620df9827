"""torch.autograd wrapper of the chunked path, checkpointed at the attention
output (DistFlashAttn, core concepts: rematerialization-aware checkpointing).

``checkpoint="output"`` keeps O and LSE from the forward, so the backward runs
``attn_chunked_bwd`` straight from them.  ``checkpoint="inputs"`` keeps only
Q, K and V, as checkpointing at a layer boundary would; its backward must run
the forward again first.  Both give the same gradients; the first saves one
forward pass per backward.  Argument marshalling only: the work is done by
the library's kernels.
"""

from __future__ import annotations

import torch

from .attention import chunked_bwd, chunked_fwd


class ChunkedAttention(torch.autograd.Function):
    """O = softmax(scale Q K^T [+ causal mask]) V over chunks of ``chunk_len``."""

    @staticmethod
    def forward(ctx, q, k, v, chunk_len, causal, scale, keep_output):
        o, lse = chunked_fwd(q, k, v, chunk_len, causal, scale)
        if keep_output:
            ctx.save_for_backward(q, k, v, o, lse)
        else:
            ctx.save_for_backward(q, k, v)
        ctx.cfg = (chunk_len, causal, scale, keep_output)
        return o

    @staticmethod
    def backward(ctx, d_o):
        chunk_len, causal, scale, keep_output = ctx.cfg
        if keep_output:
            q, k, v, o, lse = ctx.saved_tensors
        else:
            q, k, v = ctx.saved_tensors
            o, lse = chunked_fwd(q, k, v, chunk_len, causal, scale)  # the re-run
        if d_o.stride(-1) != 1:
            d_o = d_o.contiguous()
        dq, dk, dv = chunked_bwd(q, k, v, o, lse, d_o, chunk_len, causal, scale)
        return dq, dk, dv, None, None, None, None


def chunked_attention(q, k, v, chunk_len=4096, causal=True, scale=None, checkpoint="output"):
    """Differentiable exact attention, q [B, Hq, N, d], k, v [B, Hkv, N, d].

    checkpoint: "output" (keep O and LSE; the backward does not re-run the
    forward) or "inputs" (keep Q, K, V only; the backward re-runs it)."""
    if checkpoint not in ("output", "inputs"):
        raise ValueError("checkpoint must be 'output' or 'inputs'")
    return ChunkedAttention.apply(q, k, v, int(chunk_len), bool(causal), scale,
                                  checkpoint == "output")
