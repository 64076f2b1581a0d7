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
