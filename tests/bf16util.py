"""Small helpers the tests share: bf16 bit patterns and ulp distances."""
import numpy as np


def ordered(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are monotone in the value, with
    +0 and -0 both mapped to 0, so that |ordered(a) - ordered(b)| counts ulps."""
    b = np.asarray(bits).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


# Distance reported for a pair that must match exactly and does not.
MISMATCH = 1 << 16


def is_nan(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits).astype(np.int32)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def is_inf(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.int32) & 0x7FFF) == 0x7F80


def ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """bf16 ulp distance of finite values (+0 == -0).  Non-finite values are
    compared by what they are: a NaN matches any NaN (sign and payload are not
    fixed by the arithmetic: the oracle keeps a quiet payload, the GPU's
    conversion returns one canonical NaN) and nothing else; an infinity
    matches only the same infinity.  A mismatch counts as MISMATCH ulps."""
    a, b = np.asarray(a), np.asarray(b)
    d = np.abs(ordered(a) - ordered(b))
    an, bn = is_nan(a), is_nan(b)
    d = np.where(an | bn, np.where(an & bn, 0, MISMATCH), d)
    ai, bi = is_inf(a), is_inf(b)
    special_inf = (ai | bi) & ~(an | bn)
    same = np.asarray(a).astype(np.int32) == np.asarray(b).astype(np.int32)
    return np.where(special_inf, np.where(same, 0, MISMATCH), d)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bits_torch(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 (RNE) bit patterns through torch's own conversion."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
