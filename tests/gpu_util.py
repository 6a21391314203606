"""Helpers shared by the GPU parity tests (test infrastructure)."""
import numpy as np
import pytest
import torch

DEV = torch.device("cuda:0")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def host(t):
    """Device tensor -> numpy (fp16 stays fp16; bf16 -> uint16 bits)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits(t):
    """Host fp16 / bf16 tensor -> uint16 bit array for the oracle."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(t):
    return t.detach().cpu().double().numpy()


def sync():
    torch.cuda.synchronize()
