"""bf16 helpers for the tests (numpy; independent of the oracle's C code)."""
import numpy as np


def to_bits(x) -> np.ndarray:
    """float -> bf16 bits, round to nearest even (via float32)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rnd(x) -> np.ndarray:
    """Round to the nearest bf16 value, returned as float64."""
    return to_f32(to_bits(x)).astype(np.float64)


def ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)
