"""bf16 bit patterns (uint16) widened to float64; exact, since bf16 is a prefix of fp32."""
import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)
