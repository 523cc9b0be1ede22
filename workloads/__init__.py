"""Seeded synthetic inputs for sparse long-context decode.

This module only DRAWS inputs: raw bf16 keys, values and queries, the frozen
sketch basis and its per-dimension quantiser step, request lengths and the
planted positions of the tiny workload.  It holds none of the method's
arithmetic (no projection, quantisation, scoring, selection or attention);
both the CUDA path and the CPU oracle consume what it returns.

Workloads (sizes from the pages' configurations):
  tiny    : 1 request x 8192 tokens, 8 query / 2 KV heads, head dim 256, bf16
            K/V ~ N(0,1), 32 planted tokens whose keys align with their group's
            queries; rank-64 fp32 sketch; top 512 + 64 sinks + 256 tail.
  sketch  : 8 requests x 250,000 tokens x 16 layers, 24 query / 4 KV heads,
            head dim 256, int8 K/V, int4 rank-64 sketch; top 2048 + 64 + 1024.
            Keys k = U (a * z) + 0.3 eps with U the frozen basis, a_j = 3 *
            0.95^j, z, eps ~ N(0, I), rescaled to unit per-element variance;
            queries follow the same law.
  pooled  : 4 requests x 1,048,576 tokens x 12 layers, 16 query / 2 KV heads,
            bf16 K/V, 128-dim bf16 indexer keys pooled by 4; top 512 blocks.
            16 clusters x 32 consecutive relevant blocks per request.

bf16 arrays are carried as numpy uint16 bit patterns on the CPU side.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

try:  # torch is only needed for the device-side generators and bf16 rounding
    import torch
except Exception:  # pragma: no cover
    torch = None


# ---------------------------------------------------------------------------
# Workload descriptions
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class SketchWorkload:
    name: str
    B: int
    T: int
    L: int
    Hq: int
    Hkv: int
    d: int
    r: int
    k: int
    S: int
    W: int
    kv: str            # "bf16" | "int8"
    sketch: str        # "f32" | "int4"
    seed: int

    @property
    def max_rows(self) -> int:
        return self.S + self.k + self.W

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


@dataclass(frozen=True)
class PooledWorkload:
    name: str
    B: int
    T: int
    L: int
    Hq: int
    Hkv: int
    d: int
    d_idx: int
    ratio: int
    k_blocks: int
    seed: int
    clusters: int = 16
    cluster_blocks: int = 32

    @property
    def max_rows(self) -> int:
        return self.ratio * self.k_blocks + self.ratio - 1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


TINY = SketchWorkload("tiny_1x8192_f32sketch_bf16kv", B=1, T=8192, L=1, Hq=8, Hkv=2, d=256,
                      r=64, k=512, S=64, W=256, kv="bf16", sketch="f32", seed=1)
SKETCH = SketchWorkload("sketch_8x250000_16L_int4sketch_int8kv", B=8, T=250_000, L=16, Hq=24,
                        Hkv=4, d=256, r=64, k=2048, S=64, W=1024, kv="int8", sketch="int4",
                        seed=2)
POOLED = PooledWorkload("pooled_4x1048576_12L_bf16", B=4, T=1_048_576, L=12, Hq=16, Hkv=2,
                        d=256, d_idx=128, ratio=4, k_blocks=512, seed=3)


# ---------------------------------------------------------------------------
# Helpers
# ---------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), using torch's round-to-nearest-even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def orthonormal_basis(d: int, r: int, seed: int) -> np.ndarray:
    """Random d x r matrix with orthonormal columns (QR of a Gaussian), fp32."""
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((d, r))
    qm, rm = np.linalg.qr(g)
    qm = qm * np.sign(np.diag(rm))[None, :]
    return np.ascontiguousarray(qm, dtype=np.float32)


def lowrank_amplitudes(r: int) -> np.ndarray:
    """a_j = 3 * 0.95^j: the spectrum of the keys' dominant subspace."""
    return 3.0 * 0.95 ** np.arange(r, dtype=np.float64)


def lowrank_norm(a: np.ndarray, d: int, noise: float) -> float:
    """nu such that k / nu has unit mean per-element variance."""
    return math.sqrt((float(np.sum(a * a)) + noise * noise * d) / d)


def sketch_step(Hkv: int, r: int, d: int, noise: float = 0.3, clip_sigmas: float = 4.5) -> np.ndarray:
    """Per-(head, dim) int4 quantiser step c[h][j] of the frozen sketch artifact.

    Under the key law, coordinate j of the projection on the basis is Gaussian
    with std sigma_j = sqrt(a_j^2 + noise^2) / nu.  The step is set to
    clip_sigmas * sigma_j / 7, i.e. the expected largest |projection| over a
    ~250K-token context divided by the largest code 7.  It is part of the
    offline artifact (like the basis), not computed per step.
    """
    a = lowrank_amplitudes(r)
    nu = lowrank_norm(a, d, noise)
    sig = np.sqrt(a * a + noise * noise) / nu
    c = (clip_sigmas * sig / 7.0).astype(np.float32)
    return np.ascontiguousarray(np.broadcast_to(c, (Hkv, r)))


# ---------------------------------------------------------------------------
# CPU (numpy) generators, used by the tests and the oracle baseline
# ---------------------------------------------------------------------------

def lowrank_rows(rng: np.random.Generator, n: int, U: np.ndarray, noise: float = 0.3) -> np.ndarray:
    """n rows of the key law k = (U (a*z) + noise*eps) / nu, fp32 [n][d]."""
    d, r = U.shape
    a = lowrank_amplitudes(r)
    nu = lowrank_norm(a, d, noise)
    z = rng.standard_normal((n, r))
    eps = rng.standard_normal((n, d))
    k = (z * a[None, :]) @ U.astype(np.float64).T + noise * eps
    return (k / nu).astype(np.float32)


def tiny_inputs(w: SketchWorkload = TINY, T: int | None = None) -> dict:
    """The tiny workload: bf16 K/V ~ N(0,1) with 32 planted tokens per request.

    A planted token's key for KV head h is 2*sqrt(d) * unit(sum of the group's
    queries), i.e. aligned with the group query and twice the norm of a random
    key.  Planted positions are uniform without replacement in [S, T - W).
    """
    T = w.T if T is None else T
    rng = np.random.default_rng(w.seed)
    B, Hq, Hkv, d = w.B, w.Hq, w.Hkv, w.d
    G = Hq // Hkv
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    K = rng.standard_normal((B, T, Hkv, d)).astype(np.float32)
    V = rng.standard_normal((B, T, Hkv, d)).astype(np.float32)
    n_plant = min(32, max(0, T - w.S - w.W))
    planted = np.zeros((B, n_plant), np.int64)
    qb = bf16_bits_to_f32(to_bf16_bits(q))
    for b in range(B):
        pos = np.sort(rng.choice(np.arange(w.S, T - w.W), size=n_plant, replace=False)) if n_plant else []
        planted[b, :n_plant] = pos
        for h in range(Hkv):
            gsum = qb[b, h * G:(h + 1) * G].astype(np.float64).sum(axis=0)
            u = gsum / np.linalg.norm(gsum)
            for t in pos:
                K[b, t, h] = (2.0 * math.sqrt(d) * u).astype(np.float32)
    return {
        "q": to_bf16_bits(q), "K": to_bf16_bits(K), "V": to_bf16_bits(V),
        "basis": orthonormal_basis(d, w.r, w.seed + 1000),
        "planted": planted, "lengths": np.full((B,), T, np.int32),
    }


def sketch_inputs_cpu(B: int, T: int | list, Hq: int, Hkv: int, d: int, r: int, seed: int,
                      noise: float = 0.3) -> dict:
    """Small instances of the sketch workload's law on the CPU (for parity tests).

    T may be a list of per-request lengths (ragged batch); arrays are sized to
    the largest.  Returns bf16 bit arrays K, V [B][Tcap][Hkv][d], q [B][Hq][d],
    the basis U [d][r], the step c [Hkv][r] and the lengths.
    """
    rng = np.random.default_rng(seed)
    lengths = np.array(T if isinstance(T, (list, tuple)) else [T] * B, np.int32)
    Tcap = int(lengths.max())
    U = orthonormal_basis(d, r, seed + 1000)
    K = lowrank_rows(rng, B * Tcap * Hkv, U, noise).reshape(B, Tcap, Hkv, d)
    V = rng.standard_normal((B, Tcap, Hkv, d)).astype(np.float32)
    q = lowrank_rows(rng, B * Hq, U, noise).reshape(B, Hq, d)
    return {"K": to_bf16_bits(K), "V": to_bf16_bits(V), "q": to_bf16_bits(q), "basis": U,
            "c": sketch_step(Hkv, r, d, noise), "lengths": lengths}


def pooled_inputs_cpu(B: int, T: int | list, Hq: int, Hkv: int, d: int, d_idx: int, seed: int,
                      ratio: int = 4, clusters: int = 4, cluster_blocks: int = 8) -> dict:
    """Small instances of the pooled workload's law on the CPU.

    K, V ~ N(0,1) bf16; raw indexer keys N(0,1), except inside `clusters`
    runs of `cluster_blocks` consecutive blocks per request, whose keys are
    1.5 * sqrt(d_idx) * unit(q_idx) + N(0,1).
    """
    rng = np.random.default_rng(seed)
    lengths = np.array(T if isinstance(T, (list, tuple)) else [T] * B, np.int32)
    Tcap = int(lengths.max())
    Tcap4 = ((Tcap + ratio - 1) // ratio) * ratio
    K = rng.standard_normal((B, Tcap, Hkv, d)).astype(np.float32)
    V = rng.standard_normal((B, Tcap, Hkv, d)).astype(np.float32)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    q_idx = rng.standard_normal((B, d_idx)).astype(np.float32)
    idx_keys = rng.standard_normal((B, Tcap4, d_idx)).astype(np.float32)
    for b in range(B):
        nb = int(lengths[b]) // ratio
        u = q_idx[b] / np.linalg.norm(q_idx[b])
        if nb > cluster_blocks:
            starts = rng.choice(nb - cluster_blocks, size=min(clusters, nb - cluster_blocks), replace=False)
            for s0 in starts:
                t0, t1 = s0 * ratio, (s0 + cluster_blocks) * ratio
                idx_keys[b, t0:t1] += (1.5 * math.sqrt(d_idx) * u).astype(np.float32)
    return {"K": to_bf16_bits(K), "V": to_bf16_bits(V), "q": to_bf16_bits(q),
            "q_idx": to_bf16_bits(q_idx), "idx_keys": to_bf16_bits(idx_keys), "lengths": lengths}


def fp8_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 values -> fp8 e4m3 bytes (round to nearest even, saturating at
    +-448), through torch's float8_e4m3fn type on the CPU."""
    import torch
    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def mla_inputs_cpu(B: int, n_pool_rows: int, seed: int, Hq: int = 128, d: int = 576) -> dict:
    """Small instances of the latent-row workload: rows ~ N(0,1) as fp8 e4m3,
    absorbed queries ~ N(0,1) bf16."""
    rng = np.random.default_rng(seed)
    pool = fp8_e4m3_codes(rng.standard_normal((n_pool_rows, d)).astype(np.float32))
    q = to_bf16_bits(rng.standard_normal((B, Hq, d)).astype(np.float32))
    return {"pool": pool, "q": q}


def pick_sequence(rng: np.random.Generator, lo: int, hi: int, k: int, n_steps: int, keep: float) -> list:
    """Drifting selections for resolver tests: each step keeps about `keep` of
    the previous step's tokens and draws the rest uniformly from [lo, hi).
    Returns n_steps sorted unique int32 arrays of k tokens (k <= hi - lo)."""
    seq = []
    prev = np.zeros((0,), np.int64)
    for _ in range(n_steps):
        n_keep = min(len(prev), int(round(keep * k)))
        kept = rng.choice(prev, size=n_keep, replace=False) if n_keep else prev[:0]
        pool = np.setdiff1d(np.arange(lo, hi), kept)
        new = rng.choice(pool, size=k - n_keep, replace=False)
        cur = np.sort(np.concatenate([kept, new]))
        seq.append(cur.astype(np.int32))
        prev = cur
    return seq


# ---------------------------------------------------------------------------
# Device (torch) generators, used by the benchmark at full size
# ---------------------------------------------------------------------------

def device_generator(seed: int, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def lowrank_rows_torch(gen, n: int, U_dev, noise: float = 0.3, out_dtype=None):
    """Device version of lowrank_rows (torch RNG, so not bit-equal to numpy)."""
    d, r = U_dev.shape
    a = torch.tensor(lowrank_amplitudes(r), dtype=torch.float32, device=U_dev.device)
    nu = lowrank_norm(lowrank_amplitudes(r), d, noise)
    z = torch.randn((n, r), generator=gen, device=U_dev.device, dtype=torch.float32)
    k = (z * a) @ U_dev.t()
    k.add_(torch.randn((n, d), generator=gen, device=U_dev.device, dtype=torch.float32), alpha=noise)
    k.mul_(1.0 / nu)
    return k.to(out_dtype or torch.bfloat16)


def randn_torch(gen, shape, device="cuda", dtype=None):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype or torch.bfloat16)


def pooled_index_keys_torch(gen, B: int, T: int, q_idx, ratio: int = 4, clusters: int = 16,
                            cluster_blocks: int = 32, device="cuda"):
    """Device version of the pooled workload's raw indexer keys (torch RNG).

    Keys N(0,1) bf16 [B][T][d_idx], except `clusters` runs of `cluster_blocks`
    consecutive blocks per request at seeded random block offsets, whose keys
    are 1.5 * sqrt(d_idx) * unit(q_idx[b]) + N(0,1).
    """
    d_idx = q_idx.shape[-1]
    keys = torch.empty((B, T, d_idx), dtype=torch.bfloat16, device=device)
    nb = T // ratio
    for b in range(B):
        x = torch.randn((T, d_idx), generator=gen, device=device, dtype=torch.float32)
        if nb > cluster_blocks:
            u = q_idx[b].float()
            u = u / u.norm()
            starts = torch.randperm(nb - cluster_blocks, generator=gen, device=device)[:clusters].tolist()
            for s0 in starts:
                x[s0 * ratio:(s0 + cluster_blocks) * ratio] += 1.5 * math.sqrt(d_idx) * u
        keys[b].copy_(x)
        del x
    return keys
