"""Marshalling helpers: numpy arrays from ``synth`` to torch tensors for the binding."""
from __future__ import annotations

import numpy as np
import torch


def weights_to_torch(w: dict, device="cuda") -> dict:
    """bf16 bit arrays (uint16) -> int16 tensors holding the same bits."""
    return {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).to(device) for k, v in w.items()}


def sampler_to_torch(s: dict, device="cuda") -> dict:
    return {
        "temperature": torch.from_numpy(np.ascontiguousarray(s["temperature"], np.float32)).to(device),
        "top_k": torch.from_numpy(np.ascontiguousarray(s["top_k"], np.int32)).to(device),
        "top_p": torch.from_numpy(np.ascontiguousarray(s["top_p"], np.float32)).to(device),
        "seed": torch.from_numpy(np.ascontiguousarray(s["seed"], np.uint64).view(np.int64)).to(device),
        "offset": torch.from_numpy(np.ascontiguousarray(s["offset"], np.int64)).to(device),
    }
