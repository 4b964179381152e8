"""Host <-> device marshalling for the GPU tests (no arithmetic of the method)."""
import numpy as np
import torch


def dev():
    return torch.device("cuda:0")


def bf16_from_bits(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(dev()).view(torch.bfloat16)


def bits_of_bf16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of_bf16(t):
    return t.float().cpu().numpy().astype(np.float64)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def scales_to_gpu_layout(s_mg, ld=None):
    """oracle scales [M, G] -> device layout [G, ld] (ld >= M, multiple of 4)."""
    M, G = s_mg.shape
    ld = ld or max(4, (M + 3) // 4 * 4)
    out = np.zeros((G, ld), np.float32)
    out[:, :M] = s_mg.T
    return to_dev(out)


def scales_from_gpu_layout(t, M):
    return t.cpu().numpy()[:, :M].T


def rel_fro(got, ref):
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def bf16_ulp_diff(a_bits, b_bits):
    """|difference| in units of the last place between bf16 bit patterns (same-sign monotone order)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(a_bits) - key(b_bits))
