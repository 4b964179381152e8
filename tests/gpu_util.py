"""Host <-> device marshalling for the GPU tests (no arithmetic of the method)."""
import numpy as np
import torch


def dev():
    return torch.device("cuda", torch.cuda.current_device())


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


def gcorr_of(aq, a_s):
    """The activation correction the GEMMs consume: -1/2 * scale * (sum of the group's E4M3 values), fp32 [M, G].

    The sum is exact (float64 holds it), rounded once to fp32, then one fp32 product with the scale."""
    from oracle import e4m3
    M, K = aq.shape
    S = e4m3.decode(aq).reshape(M, K // 128, 128).sum(axis=2).astype(np.float32)
    return (np.float32(-0.5) * (np.asarray(a_s, np.float32) * S)).astype(np.float32)


def prepacked(lib, packed):
    """Canonical packed int4 (numpy uint8) -> prepacked device tensor (the library's one-time re-layout)."""
    return lib.w4a8_prepack_weights(to_dev(packed))


SIGN_NIBBLE = {0: 1, 1: 3, 2: 5, 3: 7, 4: 0, 5: 2, 6: 4, 7: 6}  # element e's sign: bit 3 of nibble SIGN_NIBBLE[e]


def decode_prepacked(words_u8):
    """Values of prepacked int4 bytes, read from the documented format (test-side decoder)."""
    w = np.ascontiguousarray(words_u8).view(np.uint32).astype(np.int64)
    out = np.empty(w.shape + (8,), np.int16)
    for e in range(8):
        m = (w >> (4 * e)) & 7
        s = (w >> (4 * SIGN_NIBBLE[e] + 3)) & 1
        half2 = np.where(s == 1, -(2 * m + 1), 2 * m + 1)  # 2 * (v + 1/2)
        out[..., e] = (half2 - 1) // 2
    return out.reshape(words_u8.shape[:-1] + (words_u8.shape[-1] * 2,))

