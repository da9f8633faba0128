"""Test helpers: storage-format arrays <-> device tensors, and the parity bar."""
import numpy as np
import torch

import oracle
from sequence_tensor_transformer_gb300 import synth

# rel. max error bounds: bf16 inputs with fp32 accumulation, and fp32
TOL = {"bf16": 2e-2, "fp32": 1e-5}


def dev_tensor(a: np.ndarray, dtype: str, device="cuda:0") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return synth.to_f64(a, dtype)


def rel_err(got, ref) -> float:
    return oracle.rel_max_error(got, ref)
