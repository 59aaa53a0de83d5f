"""fp64 CPU oracle of the batch-1 quantised MoE expert block.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never calls it, and it shares no code with the CUDA path:
the blob format, unpacking, dequantisation, routing and combine are written
here a second time, from the definitions below, in plain numpy float64.

What is computed (all in fp64; fp32 and bf16 inputs are widened exactly):

* unpack      element c of a packed row is bits [(c mod m)*bits, +bits) of
              word floor(c/m), m = 32/bits (lowest bits first)
* layout      gate/up rows as records; the down projection by column, its
              (scale,bias) words by group of 64 columns (this project's byte
              order; the pages fix only one contiguous blob per expert)
* dequantise  W[r, c] = q[r, c] * s[r, c//64] + b[r, c//64]
              ("nibble * scale + bias", flash-moe write-up on discuss.pytorch.kr,
              section "FMA-optimised dequant kernel")
* expert FFN  a = Wg x, u = Wu x, h = silu(a) * u, y = Wd h
              (the same write-up, section "hand-written Metal compute shaders":
              4/2-bit dequant matvec and fused SwiGLU)
* route       top-K of the router logits by value (ties: lower expert id
              first), weights = softmax over the K selected logits
              (same write-up, section "per-layer pipeline": CPU softmax + top-K)
* router      logits = W_r x, W_r bf16 [E][H] (same write-up, section
              "per-layer pipeline": the routing logits come from the GPU)
* shared gate g = sigmoid(w_sg . x) scaling the always-on shared expert
              (same write-up: model section "K=4 of 512 experts plus one
              shared expert", shader list "MoE combine + residual + sigmoid gate")
* combine     out = residual + sum_k w_k y_k + g y_shared
* RMSNorm     x / sqrt(mean(x^2) + eps), unit weight (shader list: two-stage
              RMS normalisation), used pre-norm between stacked blocks; times
              a learned weight vector when one is given
* o_proj      y = W x (+ residual) for a dense quantised matrix in row records
              (same write-up, "per-layer pipeline": CMD2's o_proj)

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(hand-worked examples, closed forms, brute force and invariants); see the
docstring of each function for the pin that covers it.
"""
from .moe import (  # noqa: F401
    GROUP,
    layout,
    part_rows,
    unpack_codes,
    bf16_to_f64,
    dequantize,
    dequantize_codes,
    expert_weights,
    silu,
    sigmoid,
    expert_ffn,
    route,
    router_logits,
    shared_gate,
    combine,
    moe_block,
    rms_norm,
    dense_record_words,
    dense_weights,
    dense_matvec,
    stack_decode,
)
