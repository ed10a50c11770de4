"""Seeded synthetic workloads for FAVOR+ forward attention.

Everything here is input generation: Gaussian draws, the orthogonal random
projection blocks that the method draws once per head, and rounding to the
storage dtype.  No attention arithmetic lives here; the oracle and the CUDA
library both receive the arrays produced by these functions.

Projection matrix omega (per head, shape [m, d]):
  * orthogonal ("R-ORF", Rethinking Attention with Performers, §2.4 and
    App. B.2 (1)): each d x d block has exactly orthogonal rows taken from the
    QR factorisation of a Gaussian matrix (signs fixed by diag(R) so the
    block is Haar distributed); row r is then rescaled by an independent
    chi(d) length ||g_r||, g_r ~ N(0, I_d), which keeps each row marginally
    N(0, I_d) (App. F.4: orthogonal samples keep the Gaussian marginals and
    have independent lengths).  m > d stacks ceil(m/d) independent blocks; a
    partial last block keeps its first rows.
  * iid: every entry N(0, 1) (§2.3, Eq. 5 with D = N(0, I_d)).
  * regularized (SMREG, §2.3 after Lemma 1): omega replaced by
    sqrt(d) omega / ||omega||, i.e. D = Unif(sqrt(d) S^{d-1}); with orthogonal
    blocks the rows keep their orthogonality and all have length sqrt(d).

Random stream order for one workload: a single numpy Generator(PCG64(seed))
draws omega for heads h = 0..H-1 in order, then Q, K, V, then (if asked)
the sharp-key row choice and nothing else.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["CONFIGS", "Workload", "make_omega_orf", "make_omega_iid",
           "make_qkv", "make_workload", "make_upstream_grad", "round_bf16"]


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    Pure bit arithmetic on the float32 pattern, so the result is exactly what a
    device conversion with round-to-nearest-even produces.  NaN is not
    expected in synthetic data and is not special-cased.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def make_omega_orf(rng: np.random.Generator, m: int, d: int, regularized: bool = False) -> np.ndarray:
    """Orthogonal Gaussian projection rows [m, d] (float64); lengths sqrt(d) if regularized."""
    nblocks = -(-m // d)
    rows = []
    for _ in range(nblocks):
        g = rng.standard_normal((d, d))
        qmat, rmat = np.linalg.qr(g)
        qmat = qmat * np.sign(np.diag(rmat))[None, :]
        block = qmat.T                      # rows are orthonormal
        lengths = np.linalg.norm(rng.standard_normal((d, d)), axis=1)
        if regularized:
            lengths = np.full(d, np.sqrt(d))
        rows.append(block * lengths[:, None])
    return np.concatenate(rows, axis=0)[:m]


def make_omega_iid(rng: np.random.Generator, m: int, d: int, regularized: bool = False) -> np.ndarray:
    """Independent N(0, 1) projection rows [m, d] (float64); rescaled to length sqrt(d) if regularized."""
    w = rng.standard_normal((m, d))
    if regularized:
        w = w * (np.sqrt(d) / np.linalg.norm(w, axis=1, keepdims=True))
    return w


def make_qkv(rng: np.random.Generator, B: int, H: int, L: int, d: int, dv: int,
             std: float, sharp_frac: float = 0.0, sharp_mult: float = 1.0):
    """Q, K [B,H,L,d] and V [B,H,L,dv] ~ N(0, std^2), float32.

    With ``sharp_frac`` > 0, floor(sharp_frac * L) distinct key rows per
    (b, h), chosen uniformly, are multiplied by ``sharp_mult`` (all d
    entries) to produce sharp attention rows.
    """
    q = rng.standard_normal((B, H, L, d), dtype=np.float32)
    k = rng.standard_normal((B, H, L, d), dtype=np.float32)
    v = rng.standard_normal((B, H, L, dv), dtype=np.float32)
    if std != 1.0:
        q *= np.float32(std)
        k *= np.float32(std)
        v *= np.float32(std)
    nsharp = int(math.floor(sharp_frac * L))
    if nsharp > 0:
        for b in range(B):
            for h in range(H):
                idx = rng.choice(L, size=nsharp, replace=False)
                k[b, h, idx, :] *= np.float32(sharp_mult)
    return q, k, v


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic FAVOR+ workload (shapes, distribution, kernel, dtype)."""
    name: str
    B: int
    H: int
    L: int
    d: int
    dv: int
    m: int
    dtype: str                 # "f32" or "bf16"
    std: float                 # per-element std of Q, K, V before input_scale
    input_scale: float         # Q, K, V multiplied by this at generation
    data_scale: float          # s passed to the library: x = s*q, y = s*k
    ortho: bool = True
    regularized: bool = False      # SMREG projection rows (length sqrt(d))
    sharp_frac: float = 0.0
    sharp_mult: float = 1.0
    modes: tuple = ("bidir",)
    kinds: tuple = ("softmax_pos",)

    @property
    def tokens_heads(self) -> int:
        return self.B * self.H * self.L

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # Tiny fp32: N(0,1) inputs already scaled by d^-1/4, two 16x16 ORF blocks.
    "tiny_f32": Workload("tiny_f32", 1, 1, 64, 16, 16, 32, "f32", 1.0, 16 ** -0.25, 1.0,
                         modes=("bidir", "causal")),
    # Approximation-error shape (L=4096, d=16, m swept), fp32.
    "approx_f32": Workload("approx_f32", 1, 8, 4096, 16, 16, 256, "f32", 1.0, 16 ** -0.25, 1.0),
    # Bidirectional encoder, bf16.
    "bidir_bf16": Workload("bidir_bf16", 8, 12, 4096, 64, 64, 256, "bf16", 0.5, 1.0, 64 ** -0.25),
    # Causal long sequence with 1% sharp key rows (x4), bf16.
    "causal_bf16": Workload("causal_bf16", 4, 8, 8192, 64, 64, 256, "bf16", 0.5, 1.0, 64 ** -0.25,
                            sharp_frac=0.01, sharp_mult=4.0, modes=("causal",)),
    # Very long context, bf16, both modes and both feature kinds.
    "long_bf16": Workload("long_bf16", 1, 16, 65536, 64, 64, 256, "bf16", 0.5, 1.0, 64 ** -0.25,
                          modes=("bidir", "causal"), kinds=("softmax_pos", "relu")),
}


def make_workload(w: Workload, seed: int = 0):
    """Draw (omega [H,m,d], q, k, v) for workload ``w`` as float32 arrays.

    For bf16 workloads every array is rounded to bfloat16 values (kept in
    float32 storage), so the oracle and the device see identical numbers.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    make = make_omega_orf if w.ortho else make_omega_iid
    omega = np.stack([make(rng, w.m, w.d, w.regularized) for _ in range(w.H)]).astype(np.float32)
    q, k, v = make_qkv(rng, w.B, w.H, w.L, w.d, w.dv, w.std, w.sharp_frac, w.sharp_mult)
    if w.input_scale != 1.0:
        sc = np.float32(w.input_scale)
        q *= sc
        k *= sc
        v *= sc
    if w.dtype == "bf16":
        omega, q, k, v = (round_bf16(a) for a in (omega, q, k, v))
    return omega, q, k, v


def make_upstream_grad(w: Workload, seed: int = 0) -> np.ndarray:
    """Upstream gradient dO [B,H,L,dv] for a backward call on workload ``w``:
    N(0, 1) entries from Generator(PCG64(seed + 1_000_003)), a stream of its
    own so that adding it leaves the forward inputs of ``seed`` unchanged;
    rounded to bfloat16 values for bf16 workloads."""
    rng = np.random.Generator(np.random.PCG64(seed + 1_000_003))
    g = rng.standard_normal((w.B, w.H, w.L, w.dv), dtype=np.float32)
    return round_bf16(g) if w.dtype == "bf16" else g
