"""Seeded synthetic inputs for kernelized linear attention.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds none of the method's arithmetic: it only draws Gaussian
numbers from numpy's PCG64 generator, scales them, rounds them to the storage
dtype and builds packed-sequence boundaries.  The random numbers that the
FAVOR+ feature map needs (the Gaussian blocks that are orthogonalised into the
projection matrix, and the Gaussian vectors whose lengths set the row norms)
are drawn here too and handed to both sides as inputs.

Workloads follow the five cases of the linear-attention benchmark plan:
a single-head fp32 case, a causal ELU+1 case, a bidirectional FAVOR+ encoder
case, a long causal FAVOR+ case and a packed variable-length causal FAVOR+
case.  Values: q, k ~ N(0,1) (scaled by d^-1/4 where the workload says so,
which folds the softmax temperature into q and k, as the Kernel Zoo page does
in §3.3), v ~ N(0,1).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

DATA_SEED_BASE = 2024
OMEGA_SEED = 7

MAP_IDS = {"identity": 0, "elu1": 1, "favor": 2}
DTYPE_IDS = {"f32": 0, "bf16": 1}


# ----------------------------------------------------------------------------
# bf16 storage: round-to-nearest-even from fp32, widening back is exact.
# ----------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    bias = ((u >> 16) & 1).astype(np.uint32) + np.uint32(0x7FFF)
    r = ((u + bias) >> 16).astype(np.uint16)
    if nan.any():
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to fp32 exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantise(x: np.ndarray, dtype: str) -> np.ndarray:
    """Return fp32 values that are exactly representable in `dtype`."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return bf16_to_f32(bf16_bits(x))
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    description: str
    H: int
    dk: int
    dv: int
    r: int
    map: str            # "identity" | "elu1" | "favor"
    causal: bool
    dtype: str          # "f32" | "bf16"
    lengths: list       # per-sequence token counts (packed in this order)
    qk_scale: float     # q, k ~ N(0,1) * qk_scale
    eps: float = 1e-6
    equal_lengths: bool = True   # True: a B x N batch (cu_seqlens may be omitted)
    seed: int = DATA_SEED_BASE
    norm: str = "attention"      # "attention" | "none" | "sum"
    carry: bool = False          # a state is carried in (state_in) and out (state_out)
    decode: bool = False         # one-token decode steps: lengths = [1] * B against a carried state
    n_prior: int = 0             # tokens the carried state stands for (carry / decode)
    backward: bool = False       # the gradients of sum(dout * out) rather than the forward

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def nseq(self) -> int:
        return len(self.lengths)

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n sequence lengths drawn uniformly from the integers lo..hi inclusive."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def workloads() -> dict:
    s = 64 ** -0.25
    w = {}
    w["fp32_n1024"] = Workload(
        "fp32_n1024", "single head, N=1024, d=64, fp32, FAVOR+ r=256 (also run with ELU+1, "
        "causal and bidirectional)", H=1, dk=64, dv=64, r=256, map="favor", causal=True,
        dtype="f32", lengths=[1024], qk_scale=s, seed=DATA_SEED_BASE + 0)
    w["elu_causal_b8h8n4096"] = Workload(
        "elu_causal_b8h8n4096", "causal ELU+1, B=8, H=8, N=4096, d=64, bf16",
        H=8, dk=64, dv=64, r=64, map="elu1", causal=True, dtype="bf16",
        lengths=[4096] * 8, qk_scale=1.0, seed=DATA_SEED_BASE + 1)
    w["favor_bidir_b4h8n16384"] = Workload(
        "favor_bidir_b4h8n16384", "bidirectional FAVOR+ r=256, B=4, H=8, N=16384, d=64, bf16",
        H=8, dk=64, dv=64, r=256, map="favor", causal=False, dtype="bf16",
        lengths=[16384] * 4, qk_scale=s, seed=DATA_SEED_BASE + 2)
    w["favor_causal_b1h16n65536"] = Workload(
        "favor_causal_b1h16n65536", "causal FAVOR+ r=256, B=1, H=16, N=65536, d=64, bf16",
        H=16, dk=64, dv=64, r=256, map="favor", causal=True, dtype="bf16",
        lengths=[65536], qk_scale=s, seed=DATA_SEED_BASE + 3)
    w["favor_causal_varlen64_h8"] = Workload(
        "favor_causal_varlen64_h8", "packed causal FAVOR+ r=256, H=8, d=64, bf16, 64 sequences "
        "with lengths uniform in [128, 8192]",
        H=8, dk=64, dv=64, r=256, map="favor", causal=True, dtype="bf16",
        lengths=varlen_lengths(64, 128, 8192, DATA_SEED_BASE + 4), qk_scale=s,
        equal_lengths=False, seed=DATA_SEED_BASE + 4)
    w["dpfp2_causal_b8h8n4096"] = Workload(
        "dpfp2_causal_b8h8n4096", "causal DPFP-2 (r = 256), B=8, H=8, N=4096, d=64, bf16",
        H=8, dk=64, dv=64, r=256, map="dpfp2", causal=True, dtype="bf16",
        lengths=[4096] * 8, qk_scale=1.0, seed=DATA_SEED_BASE + 5)
    w["favor_causal_b1h16n65536_carry"] = w["favor_causal_b1h16n65536"].with_(
        name="favor_causal_b1h16n65536_carry",
        description="causal FAVOR+ r=256, B=1, H=16, N=65536, d=64, bf16, continuing from a carried state "
                    "(state_in standing for 65536 earlier tokens) and returning the final state",
        carry=True, n_prior=65536, seed=DATA_SEED_BASE + 6)
    w["elu_causal_b8h8n4096_sum"] = w["elu_causal_b8h8n4096"].with_(
        name="elu_causal_b8h8n4096_sum",
        description="causal ELU+1 with sum normalisation, B=8, H=8, N=4096, d=64, bf16",
        norm="sum", seed=DATA_SEED_BASE + 7)
    w["favor_causal_b1h16n65536_none"] = w["favor_causal_b1h16n65536"].with_(
        name="favor_causal_b1h16n65536_none",
        description="causal FAVOR+ r=256, unnormalised output, B=1, H=16, N=65536, d=64, bf16",
        norm="none", seed=DATA_SEED_BASE + 8)
    w["favor_decode_b256h16"] = Workload(
        "favor_decode_b256h16", "one-token causal FAVOR+ decode step, r=256, B=256 sequences, H=16, d=64, "
        "bf16 q/k/v, fp32 state standing for 4096 earlier tokens (272 MB of state)",
        H=16, dk=64, dv=64, r=256, map="favor", causal=True, dtype="bf16", lengths=[1] * 256, qk_scale=s,
        decode=True, n_prior=4096, seed=DATA_SEED_BASE + 9)
    w["favor_causal_b4h8n4096_bwd"] = Workload(
        "favor_causal_b4h8n4096_bwd", "backward (dq, dk, dv) of causal FAVOR+ r=256, B=4, H=8, N=4096, d=64, bf16, "
        "dout ~ N(0, 1)", H=8, dk=64, dv=64, r=256, map="favor", causal=True, dtype="bf16",
        lengths=[4096] * 4, qk_scale=s, backward=True, seed=DATA_SEED_BASE + 10)
    return w


def random_state(nseq: int, H: int, r: int, dv: int, seed: int, z_mean: float, n_prior: int) -> np.ndarray:
    """A carried state [nseq, H, r, dv + 1] fp32 (row f: S[f, 0..dv-1], then z[f])
    with the magnitudes of sums over n_prior earlier tokens: z[f] = z_mean *
    n_prior * U(0.5, 1.5) (a sum of positive features whose mean is z_mean) and
    S[f, c] = z[f] * N(0, 1) / sqrt(n_prior) (feature-weighted sums of N(0, 1)
    values).  Random numbers only: no attention arithmetic."""
    rng = np.random.Generator(np.random.PCG64(seed))
    st = np.empty((nseq, H, r, dv + 1), np.float32)
    z = (z_mean * n_prior * rng.uniform(0.5, 1.5, size=(nseq, H, r))).astype(np.float32)
    st[..., dv] = z
    st[..., :dv] = z[..., None] * rng.standard_normal((nseq, H, r, dv), dtype=np.float32) / np.float32(
        np.sqrt(max(n_prior, 1)))
    return st


def mean_feature(kind: str, r: int) -> float:
    """Typical mean of one feature for q, k ~ N(0, 1)-scaled inputs: 1/sqrt(r)
    for FAVOR+ (its features are unbiased for exp(x^T y) with E = 1 per
    pair, spread over r features), 1 for the element-wise maps."""
    return 1.0 / np.sqrt(r) if kind == "favor" else 1.0


@dataclass
class Inputs:
    q: np.ndarray          # fp32 [T, H, dk], values exactly representable in the dtype
    k: np.ndarray
    v: np.ndarray          # fp32 [T, H, dv]
    cu_seqlens: np.ndarray  # int32 [nseq + 1]
    dtype: str

    def storage(self, name: str) -> np.ndarray:
        """Array in storage form: fp32, or the bf16 bit pattern viewed as int16."""
        a = getattr(self, name)
        if self.dtype == "f32":
            return a
        return bf16_bits(a).view(np.int16)


def make_qkv(w: Workload, seed: Optional[int] = None) -> Inputs:
    """Draw q, k, v for a workload (seeded), quantised to its dtype."""
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    T = w.T
    out = {}
    for name, d, scale in (("q", w.dk, w.qk_scale), ("k", w.dk, w.qk_scale), ("v", w.dv, 1.0)):
        x = rng.standard_normal((T, w.H, d), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[name] = quantise(x, w.dtype)
    return Inputs(out["q"], out["k"], out["v"], w.cu_seqlens, w.dtype)


def omega_gaussians(r: int, d: int, seed: int = OMEGA_SEED):
    """The random draws behind an orthogonal random-feature matrix.

    Returns (blocks, norm_vectors): blocks is [ceil(r/d), d, d] of iid N(0,1)
    (each block is orthogonalised row by row into d orthonormal directions),
    norm_vectors is [r, d] of iid N(0,1) (row i of the projection gets the
    length of norm_vectors[i], a chi(d) draw).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = -(-r // d)
    blocks = rng.standard_normal((nb, d, d))
    norms = rng.standard_normal((r, d))
    return blocks, norms


def random_inputs(T_lengths, H, dk, dv, dtype, seed, qk_scale=64 ** -0.25):
    """Small ad-hoc inputs for tests: lengths list -> Inputs."""
    w = Workload("adhoc", "adhoc", H=H, dk=dk, dv=dv, r=dk, map="favor", causal=True,
                 dtype=dtype, lengths=list(T_lengths), qk_scale=qk_scale, seed=seed)
    return make_qkv(w)
