"""Seeded synthetic inputs for the batch-1 fine-grained MoE verify step.

Shared by the tests, the smoke check and the benchmark, for both the oracle
and the CUDA library. The module draws random numbers and prepares them the
way a checkpoint loader would; it contains none of the step's arithmetic
(no routing, no matrix products, no activation, no argmax).

Recipe (shapes of the Gemma-4-26B-A4B decoder as printed in the
"llm-decoding" post, §"The exact architecture"; distributions fixed by the
benchmark configurations):
  * hidden states        ~N(0, 1), rounded to bf16;
  * router weight        [128, 2816] ~N(0, 0.02), rounded to bf16;
  * router bias          b_e = -s * ln(e + 1) (a Zipf(s) prior over experts,
                         s = 0 for no bias; the same in every layer);
  * expert weights       129 experts (128 routed + 1 shared, stored last):
                         gate and up [704, 2816], down [2816, 704],
                         ~N(0, 0.02) in fp32, then quantised per output row
                         to E4M3 with scale = max|row| / 448 (fp32) by
                         torch's float8_e4m3fn cast (round to nearest even);
  * dense shared MLP     (the wider always-on variant) gate/up [2112, 2816]
                         and down [2816, 2112], ~N(0, 0.02), quantised per
                         output row like the experts;
  * tied embedding       [V, 2816] ~N(0, 0.02), rounded to bf16;
                         its 8-bit copy for the FP8 lm_head: the expert
                         weights' per-row E4M3 quantiser applied to those
                         bf16 rows;
  * draft tokens         d_i equals the target token of position i-1 with
                         probability p (0.7), else uniform over [0, V).
Every draw comes from a torch.Generator seeded explicitly. Values depend on
the device the generator runs on (CPU and CUDA streams differ), so a test
generates on one device and copies from there.
"""

from __future__ import annotations

import torch

HIDDEN = 2816
FFN = 704
EXPERTS = 128
TOPK = 8
LAYERS = 30
VOCAB = 262144
WEIGHT_STD = 0.02
RMS_EPS = 1e-6
E4M3_MAX = 448.0

LAYER_KEYS = ("router_w", "router_b", "gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def zipf_bias(s: float, n_experts: int = EXPERTS) -> torch.Tensor:
    """Router logit bias -s*ln(e+1), e = 0..n-1 (float32, CPU)."""
    e = torch.arange(n_experts, dtype=torch.float64)
    return (-float(s) * torch.log(e + 1.0)).to(torch.float32)


def quantize_rows_e4m3(w: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Per-output-row E4M3 codes (uint8) and fp32 scales for an fp32 tensor [..., cols]."""
    amax = w.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (w / scale.unsqueeze(-1)).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale.to(torch.float32)


def layer(seed: int, *, device="cpu", s: float = 0.0, hidden: int = HIDDEN, ffn: int = FFN,
          experts: int = EXPERTS, n_shared: int = 1, std: float = WEIGHT_STD,
          zero_shared: bool = False) -> dict[str, torch.Tensor | None]:
    """One MoE layer's parameters on ``device``.

    Keys: router_w bf16 [E, H]; router_b f32 [E] or None (s == 0);
    gate_q/up_q uint8 [E+S, F, H]; gate_s/up_s f32 [E+S, F];
    down_q uint8 [E+S, H, F]; down_s f32 [E+S, H].
    ``zero_shared`` zeroes the shared expert's weights (scale 1, codes 0).
    """
    g = _gen(seed, device)
    n_all = experts + n_shared
    out: dict[str, torch.Tensor | None] = {}
    rw = torch.randn((experts, hidden), generator=g, device=device, dtype=torch.float32) * std
    out["router_w"] = rw.to(torch.bfloat16)
    out["router_b"] = zipf_bias(s, experts).to(device) if s != 0.0 else None
    for name, shape in (("gate", (n_all, ffn, hidden)), ("up", (n_all, ffn, hidden)),
                        ("down", (n_all, hidden, ffn))):
        w = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
        if zero_shared and n_shared:
            w[experts:] = 0.0
        q, sc = quantize_rows_e4m3(w)
        del w
        out[name + "_q"] = q
        out[name + "_s"] = sc
    return out


def dense_mlp(seed: int, *, width: int = 3 * FFN, device="cpu", hidden: int = HIDDEN,
              std: float = WEIGHT_STD) -> dict[str, torch.Tensor]:
    """An always-on gated-GELU MLP of the given width (the 2816 x 2112 dense
    MLP of the page's byte list): gate_q/up_q uint8 [W, H] with gate_s/up_s
    f32 [W]; down_q uint8 [H, W] with down_s f32 [H], each quantised per
    output row (down rows are W wide)."""
    g = _gen(seed, device)
    out: dict[str, torch.Tensor] = {}
    for name, shape in (("gate", (width, hidden)), ("up", (width, hidden)), ("down", (hidden, width))):
        w = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
        out[name + "_q"], out[name + "_s"] = quantize_rows_e4m3(w)
        del w
    return out


def dense_mlp_as_experts(mlp: dict[str, torch.Tensor], ffn: int = FFN) -> dict[str, torch.Tensor]:
    """The same MLP laid out as width / ffn experts of FFN width `ffn`:
    expert p takes gate/up rows [p ffn, (p+1) ffn) and down columns of the
    same range; every expert keeps the full-width down rows' scales. A re-
    layout only: no value changes."""
    W, H = mlp["gate_q"].shape
    assert W % ffn == 0
    n = W // ffn
    return {
        "gate_q": mlp["gate_q"].reshape(n, ffn, H).contiguous(),
        "gate_s": mlp["gate_s"].reshape(n, ffn).contiguous(),
        "up_q": mlp["up_q"].reshape(n, ffn, H).contiguous(),
        "up_s": mlp["up_s"].reshape(n, ffn).contiguous(),
        "down_q": mlp["down_q"].reshape(H, n, ffn).permute(1, 0, 2).contiguous(),
        "down_s": mlp["down_s"].unsqueeze(0).expand(n, H).contiguous(),
    }


def hidden_states(seed: int, m: int, *, device="cpu", hidden: int = HIDDEN) -> torch.Tensor:
    """M hidden rows ~N(0, 1) rounded to bf16."""
    g = _gen(seed, device)
    return torch.randn((m, hidden), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def embedding(seed: int, *, vocab: int = VOCAB, device="cpu", hidden: int = HIDDEN,
              std: float = WEIGHT_STD, chunk_rows: int = 1 << 15) -> torch.Tensor:
    """Tied embedding [V, H] ~N(0, std) rounded to bf16, drawn in row chunks."""
    g = _gen(seed, device)
    e = torch.empty((vocab, hidden), device=device, dtype=torch.bfloat16)
    for r0 in range(0, vocab, chunk_rows):
        r1 = min(vocab, r0 + chunk_rows)
        e[r0:r1] = (torch.randn((r1 - r0, hidden), generator=g, device=device,
                                dtype=torch.float32) * std).to(torch.bfloat16)
    return e


def embedding_fp8(emb: torch.Tensor, *, chunk_rows: int = 1 << 14) -> tuple[torch.Tensor, torch.Tensor]:
    """The tied embedding stored in 8 bits: per-row E4M3 codes (uint8 [V, H]) and
    fp32 row scales [V], by the quantiser of the expert weights applied to the
    bf16 rows (on the tensor's device, in row chunks)."""
    V, H = emb.shape
    q = torch.empty((V, H), dtype=torch.uint8, device=emb.device)
    sc = torch.empty(V, dtype=torch.float32, device=emb.device)
    for r0 in range(0, V, chunk_rows):
        r1 = min(V, r0 + chunk_rows)
        q[r0:r1], sc[r0:r1] = quantize_rows_e4m3(emb[r0:r1].to(torch.float32))
    return q, sc


def uniforms(seed: int, n: int) -> torch.Tensor:
    """n uniforms in [0, 1) (float32, CPU) for the sampling verify's decisions."""
    return torch.rand(n, generator=_gen(seed, "cpu"), dtype=torch.float32)


def drafts(seed: int, target, *, vocab: int = VOCAB, p: float = 0.7) -> torch.Tensor:
    """gamma = len(target) - 1 draft tokens (int32, CPU): d_i = target[i-1] with
    probability p, else uniform over [0, vocab)."""
    t = torch.as_tensor(target, dtype=torch.int64).cpu()
    gamma = t.numel() - 1
    g = _gen(seed, "cpu")
    hit = torch.rand(gamma, generator=g) < p
    rnd = torch.randint(0, vocab, (gamma,), generator=g)
    return torch.where(hit, t[:gamma], rnd).to(torch.int32)


