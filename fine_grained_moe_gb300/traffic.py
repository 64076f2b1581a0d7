"""Algorithmic HBM bytes of one verify step (the roofline numerator).

The "llm-decoding" post sizes a batch-1 decode step by the weight bytes it
must stream, hand-counted from the config shapes (§"So the question became:
how many bytes" and §"Where the 7.36 GB goes"): a step cannot finish faster
than those bytes divided by the HBM bandwidth. The verify step of this
library streams, per layer, the router and every *distinct* expert picked by
the M tokens plus the shared expert, each exactly once, and then the tied
embedding once. Bytes that the step never needs (the other experts) are not
counted.
"""

from __future__ import annotations

HIDDEN = 2816
FFN = 704
EXPERTS = 128
VOCAB = 262144


def expert_bytes(weight_bytes: int = 1, with_scales: bool = True, hidden: int = HIDDEN,
                 ffn: int = FFN) -> int:
    """gate + up [ffn, hidden] and down [hidden, ffn], plus fp32 row scales."""
    b = 3 * hidden * ffn * weight_bytes
    if with_scales:
        b += 4 * (2 * ffn + hidden)
    return b


def router_bytes(experts: int = EXPERTS, hidden: int = HIDDEN, with_bias: bool = True) -> int:
    return experts * hidden * 2 + (experts * 4 if with_bias else 0)


def lm_head_bytes(vocab: int = VOCAB, hidden: int = HIDDEN, weight_bytes: int = 2) -> int:
    return vocab * hidden * weight_bytes


def lm_head_fp8_bytes(vocab: int = VOCAB, hidden: int = HIDDEN) -> int:
    """The embedding as E4M3 codes plus one fp32 scale per row."""
    return vocab * hidden + 4 * vocab


def dense_mlp_bytes(width: int = 3 * FFN, hidden: int = HIDDEN) -> int:
    """An always-on dense gated-GELU MLP of the given width: gate/up [W, H] and
    down [H, W] in E4M3, plus fp32 row scales (2W + H)."""
    return 3 * hidden * width + 4 * (2 * width + hidden)


def layer_dense_bytes(unique: int, width: int = 3 * FFN, with_bias: bool = True) -> int:
    """Unique bytes of one layer whose shared expert is the dense MLP: router,
    the distinct routed experts, and the MLP."""
    return int(unique) * expert_bytes() + dense_mlp_bytes(width) + router_bytes(with_bias=with_bias)


def step_bytes(unique_per_layer, *, vocab: int = VOCAB, with_lm_head: bool = True,
               n_shared: int = 1, with_bias: bool = True, fp8_lm_head: bool = False,
               dense_width: int = 0) -> int:
    """Unique bytes of one step: for each layer the router and (unique routed +
    shared) experts, or with ``dense_width`` the unique routed experts and a
    dense MLP of that width in place of the shared expert; then the tied
    embedding once (bf16, or E4M3 with row scales)."""
    total = 0
    for u in unique_per_layer:
        if dense_width:
            total += layer_dense_bytes(u, dense_width, with_bias=with_bias)
        else:
            total += (int(u) + n_shared) * expert_bytes() + router_bytes(with_bias=with_bias)
    if with_lm_head:
        total += lm_head_fp8_bytes(vocab) if fp8_lm_head else lm_head_bytes(vocab)
    return total
