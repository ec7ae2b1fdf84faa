"""bfloat16 bit patterns -> float64 (exact widening; the oracle's own copy)."""
import numpy as np


def widen(bits) -> np.ndarray:
    """bf16 bits (uint16) to float64: the 16 bits are the high half of an
    IEEE-754 binary32, so shifting them up is exact."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)
