"""Helpers for the GPU parity tests (host-side conversions and comparisons)."""
import numpy as np
import torch

import discrete_diffusion_block_gb300 as dgp


def dev():
    return torch.device("cuda", 0)


def bf16_to_f32(t):
    return t.float().cpu().numpy()


def bits_to_f32(u16):
    """bf16 bit patterns (uint16 numpy) -> fp32 values."""
    return (np.asarray(u16, np.uint32) << 16).view(np.float32)


def rel_err(got, ref):
    """Normwise relative error max|got - ref| / max|ref|."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def partial_planes(buf, rows, V):
    """Split a partials buffer (torch int32 tensor) into its five planes."""
    T = V // 256
    a = buf.cpu().numpy().view(np.uint8)[: rows * T * 20]
    planes = a.reshape(5, rows, T * 4)
    return dict(m=planes[0].view(np.float32).reshape(rows, T),
                a=planes[1].view(np.int32).reshape(rows, T),
                s=planes[2].view(np.float32).reshape(rows, T),
                gk=planes[3].view(np.float32).reshape(rows, T),
                gi=planes[4].view(np.int32).reshape(rows, T))


def new_partials(rows, V):
    return torch.zeros(dgp.partials_bytes(rows, V) // 4, dtype=torch.int32, device=dev())


def tiles_dev(t):
    """A row-major bf16 CPU tensor [rows][cols] as a device tensor in the
    library's operand-tile order (the LM head's operand layout)."""
    bits = t.contiguous().view(torch.int16).numpy()
    return torch.from_numpy(dgp.to_operand_tiles(bits)).view(torch.bfloat16).to(dev())


def top2_gap(x):
    s = np.sort(np.asarray(x, np.float64), axis=-1)
    return s[..., -1] - s[..., -2]
