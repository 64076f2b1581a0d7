"""Test-only glue: turns the seeded synthetic tensors into the oracle's host
arrays. Holds no arithmetic of the step."""

import numpy as np
import torch

import oracle


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_values(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def to_oracle_layer(p: dict, k: int = 8, n_shared: int = 1) -> oracle.LayerParams:
    def host(name):
        v = p[name]
        return None if v is None else v.detach().cpu().contiguous().numpy()
    return oracle.LayerParams(
        router_w=bf16_bits(p["router_w"]),
        router_b=host("router_b"),
        gate_q=host("gate_q"), gate_s=host("gate_s"),
        up_q=host("up_q"), up_s=host("up_s"),
        down_q=host("down_q"), down_s=host("down_s"),
        k=k, n_shared=n_shared)


def dequant_torch(q: np.ndarray, s: np.ndarray) -> torch.Tensor:
    """Library decode of E4M3 codes (torch's float8 view), times the row scales, in fp64."""
    codes = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64)
    return codes * torch.from_numpy(np.ascontiguousarray(s)).to(torch.float64).unsqueeze(-1)


# ---------------------------------------------------------------- comparison rules
# Tolerance stated for the step: hidden states and logits within a maximum
# relative error of 1e-2 of the bf16-rounded oracle, read per token row as
# max|gpu - bf16(oracle)| / max|bf16(oracle)|. Router ids and accepted lengths
# must be bit-exact wherever the oracle's decision margin exceeds 1e-2.
REL_TOL = 1e-2
MARGIN = 1e-2


def rowwise_rel_err(gpu_bf16: torch.Tensor, ref_f64: np.ndarray) -> np.ndarray:
    g = gpu_bf16.detach().cpu().to(torch.float64).numpy()
    r = oracle.bf16_to_f64(oracle.bf16_round(ref_f64))
    return np.abs(g - r).max(axis=1) / np.abs(r).max(axis=1)


# Elementwise form of the same tolerance, reported beside the row form: each
# element's error over max(|bf16(oracle)|, 1e-2 * rms of its row), so that small
# elements are compared too without dividing by values near zero. Bound: the
# two bf16 roundings alone may put the two sides one bf16 step apart (2^-8 of
# the element); the library's arithmetic (activations as three E4M3 terms, each
# within 2^-12 of its slice maximum, and fp32 sums over 704 or 2816 products)
# adds an absolute error of order 1e-4 of the row's rms, which is 1e-2 of the
# floor. ELEM_TOL = 2e-2 covers both with margin; the tests assert it.
ELEM_TOL = 2e-2
ELEM_FLOOR = 1e-2


def elementwise_rel_err(gpu_bf16: torch.Tensor, ref_f64: np.ndarray) -> np.ndarray:
    """Per row: max_k |gpu_k - bf16(oracle)_k| / max(|bf16(oracle)_k|, 1e-2 rms(bf16(oracle)))."""
    g = gpu_bf16.detach().cpu().to(torch.float64).numpy()
    r = oracle.bf16_to_f64(oracle.bf16_round(ref_f64))
    rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    den = np.maximum(np.abs(r), ELEM_FLOOR * rms)
    return (np.abs(g - r) / den).max(axis=1)


def to_bf16_tensor(values: np.ndarray, device="cuda") -> torch.Tensor:
    """fp64 host values rounded to bf16 (the oracle's rounding) as a bf16 tensor."""
    bits = oracle.bf16_round(values).astype(np.uint16).view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(device)


def id_sets_agree(gpu_ids: np.ndarray, ref_ids: np.ndarray) -> bool:
    return sorted(gpu_ids.tolist()) == sorted(ref_ids.tolist())


def ids_valid_at_tie(gpu_ids: np.ndarray, logits: np.ndarray, k: int = 8) -> bool:
    """A routing that differs from the oracle's is acceptable only if every
    chosen expert's oracle logit is within MARGIN of the oracle's k-th logit."""
    kth = np.sort(logits)[::-1][k - 1]
    return len(set(gpu_ids.tolist())) == k and bool(np.all(logits[gpu_ids] >= kth - MARGIN))
