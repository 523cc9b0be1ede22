"""Helpers shared by the tests: moving seeded numpy inputs to the GPU and
comparison rules.  Holds none of the method's arithmetic."""
import re
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    """Every function declared in include/*.h."""
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(skv_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def bf16_dev(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on device."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def f16_dev(bits: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).to(device)


def dev(a: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def unpack_int4(q4: np.ndarray) -> np.ndarray:
    """Packed two's-complement nibbles -> int codes (last dim doubles)."""
    lo = (q4 & 15).astype(np.int16)
    hi = (q4 >> 4).astype(np.int16)
    codes = np.stack([lo, hi], axis=-1).reshape(q4.shape[:-1] + (2 * q4.shape[-1],))
    return np.where(codes >= 8, codes - 16, codes)


def assert_codes_match_except_ties(got_codes, ref_codes, ref_ratio, window=1e-4):
    """Codes equal, except a difference of one where the oracle's pre-rounding
    ratio lies within `window` of a rounding boundary (half-integer)."""
    diff = np.abs(got_codes.astype(np.int32) - ref_codes.astype(np.int32))
    frac = np.abs(np.abs(ref_ratio - np.floor(ref_ratio)) - 0.5)
    tie = frac < window * np.maximum(1.0, np.abs(ref_ratio))
    bad = (diff > 1) | ((diff == 1) & ~tie)
    assert not bad.any(), f"{int(bad.sum())} codes differ beyond rounding ties"
    return int((diff == 1).sum())


def assert_sets_within_tolerance(got_idx, ref_idx, ref_scores_of_token, kth_score, rel=1e-3):
    """Selections may differ only on tokens whose score is within rel*|s_k| of
    the k-th score (float scores, different summation order)."""
    g, r = set(map(int, got_idx)), set(map(int, ref_idx))
    assert len(g) == len(r)
    for t in g ^ r:
        s = float(ref_scores_of_token(t))
        assert abs(s - kth_score) <= rel * abs(kth_score) + 1e-30, (t, s, kth_score)
    return len(g ^ r)
