"""Small helpers the tests share: bf16 bit patterns and ulp distances."""
import numpy as np


def ordered(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are monotone in the value, with
    +0 and -0 both mapped to 0, so that |ordered(a) - ordered(b)| counts ulps."""
    b = np.asarray(bits).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a) - ordered(b))


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bits_torch(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 (RNE) bit patterns through torch's own conversion."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
