"""An NVFP4 decode that shares nothing with the oracle: the E2M1 magnitudes
read from tests/golden/e2m1_values.txt (the value set {0, 0.5, 1, 1.5, 2, 3,
4, 6} indexed by the low 3 bits, bit 3 the sign, element 2i in the low
nibble of byte i) and torch's float8_e4m3fn cast for the block scales."""
import numpy as np
import torch

from conftest import read_golden

E2M1 = np.array([float(m) for _, m in sorted(read_golden("e2m1_values.txt"), key=lambda r: int(r[0]))])
assert E2M1.shape == (8,)


def e4m3_torch(byte_array):
    return torch.from_numpy(np.asarray(byte_array, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant_independent(codes, sf, g):
    """Binary64 values code * scale * g of a quantized [rows, K] matrix from
    its codes [rows, K/2] and logical (unswizzled) scales [rows, K/16]."""
    codes = np.asarray(codes, np.uint8)
    lo, hi = codes & 15, codes >> 4
    nib = np.stack([lo, hi], -1).reshape(codes.shape[0], -1)
    val = np.where(nib & 8, -1.0, 1.0) * E2M1[nib & 7]
    scale = np.repeat(e4m3_torch(sf), 16, axis=1)
    return val * scale * float(g)
