"""Helpers shared by the GPU tests: host <-> device copies of bf16 bit patterns and codes."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_u8(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).cuda()


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().astype(np.uint8)


def host_bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def empty_u8(*shape) -> torch.Tensor:
    return torch.empty(*shape, dtype=torch.uint8, device="cuda")


def f32_scalar(v) -> torch.Tensor:
    return torch.tensor([np.float32(v)], dtype=torch.float32, device="cuda")
