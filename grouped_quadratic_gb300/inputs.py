"""Seeded synthetic OAL workloads (shared by the tests, the benchmark and smoke).

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle may use it.

The pages measure on post-RoPE Q/K/V of Qwen2.5-0.5B and Llama-3.2-1B, which
are not available here; these generators stand in for them.  They mimic the
structure the OAL paper reports ("Not All Dimensions Are Equal: Outlier-Aware
Attention Linearization with Grouped Quadratic Kernels", arXiv:2610.13674):
a few query-key dimensions per head with much larger magnitude (Sec. 3.1,
Fig. 1), grouped into a shared bulk group plus small tail groups
(Sec. 4.2, Fig. 2a: "60 bulk + 2 + 1 + 1"), and a random lower-triangular
factor L per query head (Sec. 4.3).

Recipe (numpy PCG64 streams, platform independent):
  * rng = numpy.random.default_rng(seed);
  * per KV head: n_out ~ U{2..6} outlier dims drawn without replacement, each
    with a scale ~ U[8, 20] (the tiny fp32 case instead fixes dims
    {3, 17, 40, 58} and scale 12);
  * Q, K, V ~ N(0, 1) in fp32; the outlier dims of K (for that KV head) and
    of Q (for every query head mapped to it) are multiplied by their scale;
    V is unscaled;
  * groups per query head: the tail is the KV head's outlier dims sorted by
    decreasing scale, padded with random bulk dims up to G-1 dims, dealt
    round-robin into groups 2..G; every other dim is group 1;
  * L per query head from default_rng([seed, 1, h]): strictly-lower entries
    N(0, 0.3^2), diagonal |N(0, 0.3^2)| + 0.5, upper triangle 0;
  * bf16 workloads round the fp32 draws to bf16 (nearest even) once; the
    rounded values are what both sides see.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

SEED_BASE = 20261000


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    d: int
    dv: int
    G: int
    dtype: str                 # "f32" or "bf16"
    eps: float
    Q: np.ndarray              # [B, Hq, T, d] fp32 (bf16-representable if dtype == bf16)
    K: np.ndarray              # [B, Hkv, T, d]
    V: np.ndarray              # [B, Hkv, T, dv]
    L: np.ndarray              # [Hq, G+1, G+1] fp32, lower triangular
    group: np.ndarray          # [Hq, d] int32, values 1..G
    outliers: list = field(default_factory=list)  # per KV head: (dims, scales)
    seed: int = 0
    decode_steps: int = 0      # > 0: the last decode_steps tokens are decoded one by one

    @property
    def T_prefill(self) -> int:
        return self.T - self.decode_steps

    def torch_inputs(self, device="cpu"):
        """Q, K, V as torch tensors in the workload dtype."""
        import torch
        tdt = torch.float32 if self.dtype == "f32" else torch.bfloat16
        return tuple(torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=tdt)
                     for a in (self.Q, self.K, self.V))


def bootstrap_indices(nboot: int, P: int, seed: int) -> np.ndarray:
    """[nboot, P] int32 prompt indices, each row drawn with replacement from
    0..P-1 (the prompt-level bootstrap replicates of the grouping step)."""
    return np.random.default_rng([seed, 7]).integers(0, P, size=(nboot, P)).astype(np.int32)


def random_L(rng: np.random.Generator, G: int, offdiag_std=0.3, diag_std=0.3,
             diag_shift=0.5) -> np.ndarray:
    L = np.zeros((G + 1, G + 1), np.float32)
    for g in range(G + 1):
        for c in range(g):
            L[g, c] = rng.normal(0.0, offdiag_std)
        L[g, g] = abs(rng.normal(0.0, diag_std)) + diag_shift
    return L


def make_workload(name: str, B: int, Hq: int, Hkv: int, T: int, G: int,
                  dtype: str = "bf16", d: int = 64, dv: int = 64,
                  seed: int = SEED_BASE, eps: float = 1e-6,
                  fixed_outliers: Optional[tuple] = None,
                  fixed_groups: Optional[list] = None,
                  decode_steps: int = 0) -> Workload:
    """Draw one workload following the module recipe.

    fixed_outliers: (dims, scale) applied to every KV head instead of drawing.
    fixed_groups: list of G-1 tail groups (lists of dims) for every query head.
    """
    assert Hq % Hkv == 0 and dtype in ("f32", "bf16") and G >= 1
    rng = np.random.default_rng(seed)
    rho = Hq // Hkv
    outliers = []
    for _ in range(Hkv):
        if fixed_outliers is not None:
            dims = np.asarray(fixed_outliers[0], np.int64)
            scales = np.full(dims.size, float(fixed_outliers[1]))
        else:
            n_out = int(rng.integers(2, 7))
            dims = rng.choice(d, size=n_out, replace=False).astype(np.int64)
            scales = rng.uniform(8.0, 20.0, size=n_out)
        outliers.append((dims, scales))
    Q = rng.standard_normal((B, Hq, T, d), dtype=np.float32)
    K = rng.standard_normal((B, Hkv, T, d), dtype=np.float32)
    V = rng.standard_normal((B, Hkv, T, dv), dtype=np.float32)
    for kv, (dims, scales) in enumerate(outliers):
        s = scales.astype(np.float32)
        K[:, kv][..., dims] *= s
        Q[:, kv * rho:(kv + 1) * rho][..., dims] *= s

    group = np.ones((Hq, d), np.int32)
    for h in range(Hq):
        if G == 1:
            continue
        if fixed_groups is not None:
            assert len(fixed_groups) == G - 1
            for gi, dims in enumerate(fixed_groups):
                group[h, np.asarray(dims)] = 2 + gi
            continue
        dims, scales = outliers[h // rho]
        tail = list(dims[np.argsort(-scales, kind="stable")])
        if len(tail) < G - 1:
            bulk = np.setdiff1d(np.arange(d), np.asarray(tail))
            pad = rng.choice(bulk, size=G - 1 - len(tail), replace=False)
            tail += list(pad)
        for k, r in enumerate(tail):
            group[h, r] = 2 + (k % (G - 1))

    L = np.stack([random_L(np.random.default_rng([seed, 1, h]), G) for h in range(Hq)])
    if dtype == "bf16":
        Q, K, V = round_to_bf16(Q), round_to_bf16(K), round_to_bf16(V)
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, T=T, d=d, dv=dv, G=G,
                    dtype=dtype, eps=eps, Q=Q, K=K, V=V, L=L, group=group,
                    outliers=outliers, seed=seed, decode_steps=decode_steps)


# The five named workloads (index = seed offset).
CONFIGS = {
    0: dict(name="tiny-fp32 B1 H1/1 T256 G4", B=1, Hq=1, Hkv=1, T=256, G=4, dtype="f32",
            fixed_outliers=([3, 17, 40, 58], 12.0), fixed_groups=[[3, 17], [40], [58]]),
    1: dict(name="qwen2.5-0.5b-prefill B1 H14/2 T4096 G4", B=1, Hq=14, Hkv=2, T=4096, G=4),
    2: dict(name="llama-3.2-1b-prefill B4 H32/8 T8192 G6", B=4, Hq=32, Hkv=8, T=8192, G=6),
    3: dict(name="qwen2.5-0.5b-decode B64 H14/2 T2048+1024 G4", B=64, Hq=14, Hkv=2,
            T=2048 + 1024, G=4, decode_steps=1024),
    4: dict(name="long-context-prefill B1 H14/2 T65536 G4", B=1, Hq=14, Hkv=2, T=65536, G=4),
}


def config(idx: int, **override) -> Workload:
    """Workload of named config ``idx`` (seed = SEED_BASE + idx)."""
    kw = dict(CONFIGS[idx])
    kw.update(override)
    kw.setdefault("seed", SEED_BASE + idx)
    return make_workload(**kw)
