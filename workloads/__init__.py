"""Seeded synthetic router workloads shared by the tests, the bench and the oracle.

This module only draws random numbers and rounds them to the input dtype; it
holds none of the router's arithmetic, so both the CUDA path and the CPU
oracle may take their inputs from it.

Each workload mirrors one of the five router configurations of the gate being
built (shapes, dtypes, value distributions and structure); there is no public
dataset involved.  Seeds: base seed 0; independent NumPy PCG64 streams per
role -- x: seed, W: seed + 1, bias: seed + 2, structure (outlier channels,
per-token factors, adversarial row contents): seed + 3.  Values are drawn in
float32 and, where the workload is bf16, rounded to bf16 with
round-to-nearest-even; the bf16 bit patterns (uint16) are the input of both
paths.
"""

from dataclasses import dataclass, replace

import numpy as np

SEED = 0


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    N: int
    k: int
    routed_scaling: float
    raw: bool
    dtype: str            # "f32" or "bf16" (x and W share it)
    x_kind: str           # "normal", "outlier_channels", "lognormal_rows", "adversarial"
    w_std: float
    bias_kind: str        # "uniform", "zero", "none"
    bias_range: float = 0.0
    tie_probe: bool = False   # adversarial variant: expert 2j+1 is a copy of 2j (j < 8)

    def with_T(self, T):
        return replace(self, T=T)

    def with_k(self, k):
        return replace(self, k=k)


WORKLOADS = {
    # tiny router: T=4, D=256, E=16, k=2, fp32 inputs
    "tiny": Workload("tiny", 4, 256, 16, 2, 1.0, False, "f32", "normal", 0.05, "uniform", 0.1),
    # decode router: T in {1, 8, 64}, D=7168, E=256, k=8, 1% outlier channels x50
    "decode": Workload("decode", 1, 7168, 256, 8, 2.5, False, "bf16", "outlier_channels", 0.02,
                       "uniform", 0.05),
    # prefill router: T=4096, per-token LogNormal(0,1) scale
    "prefill": Workload("prefill", 4096, 7168, 256, 8, 2.5, False, "bf16", "lognormal_rows", 0.02,
                        "uniform", 0.05),
    # large-batch adversarial router: T=16384, E=384, zero bias
    "adversarial": Workload("adversarial", 16384, 7168, 384, 8, 2.5, False, "bf16", "adversarial",
                            0.02, "zero"),
    # wide-N raw-logit head: T=32, N=129280, k=1 (argmax) and k=8
    "wide_n": Workload("wide_n", 32, 7168, 129280, 1, 1.0, True, "bf16", "normal", 0.02, "none"),
}


def float32_to_bf16_bits(a):
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_float32(bits):
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _to_dtype(a32, dtype):
    return float32_to_bf16_bits(a32) if dtype == "bf16" else np.ascontiguousarray(a32, np.float32)


def make_x(w: Workload, seed=SEED):
    """Activations [T, D]: float32 array, or uint16 bf16 bits."""
    T, D = w.T, w.D
    rng = np.random.default_rng(seed)
    srng = np.random.default_rng(seed + 3)
    x = rng.standard_normal((T, D), dtype=np.float32)
    if w.x_kind == "outlier_channels":
        ch = srng.choice(D, size=int(round(0.01 * D)), replace=False)
        x[:, ch] *= np.float32(50.0)
    elif w.x_kind == "lognormal_rows":
        x *= np.exp(srng.standard_normal(T)).astype(np.float32)[:, None]
    elif w.x_kind == "adversarial":
        cls = np.arange(T) % 4
        x[cls == 1] = 0.0
        rows2 = np.nonzero(cls == 2)[0]
        ch = srng.integers(0, D, size=rows2.size)
        x[rows2, ch] = np.float32(1.0e4)
        rows3 = np.nonzero(cls == 3)[0]
        c = srng.uniform(-2.0, 2.0, size=rows3.size).astype(np.float32)
        x[rows3] = c[:, None]
    elif w.x_kind != "normal":
        raise ValueError(w.x_kind)
    return _to_dtype(x, w.dtype)


def iter_w(w: Workload, rows_per_chunk=8192, seed=SEED):
    """Gate weight [N, D] in row chunks (same values whatever the chunk size)."""
    rng = np.random.default_rng(seed + 1)
    n0 = 0
    while n0 < w.N:
        n1 = min(w.N, n0 + rows_per_chunk)
        chunk = rng.standard_normal((n1 - n0) * w.D, dtype=np.float32).reshape(n1 - n0, w.D)
        chunk *= np.float32(w.w_std)
        yield n0, _to_dtype(chunk, w.dtype)
        n0 = n1


def make_w(w: Workload, seed=SEED):
    """Gate weight [N, D]: float32 array, or uint16 bf16 bits."""
    parts = [c for _, c in iter_w(w, rows_per_chunk=max(w.N, 1), seed=seed)]
    W = np.concatenate(parts, axis=0)
    if w.tie_probe:
        for j in range(8):
            if 2 * j + 1 < w.N:
                W[2 * j + 1] = W[2 * j]
    return W


def make_bias(w: Workload, seed=SEED):
    """Score-correction bias [N] float32, or None for RAW heads."""
    if w.bias_kind == "none":
        return None
    if w.bias_kind == "zero":
        return np.zeros(w.N, dtype=np.float32)
    rng = np.random.default_rng(seed + 2)
    return rng.uniform(-w.bias_range, w.bias_range, size=w.N).astype(np.float32)


def x_as_float32(x, w: Workload):
    """float32 view of a generated activation array (exact widening for bf16)."""
    return bf16_bits_to_float32(x) if w.dtype == "bf16" else np.asarray(x, np.float32)


# ------------------------------------------------------------------ hash router
# Token-id routing of the first MoE layers: a [vocab, k] int32 table of
# expert ids (k distinct experts per token id) and a batch of token ids.
# Table: a seeded random base expert per token id plus k distinct offsets
# shared by all rows, modulo the expert count; token ids uniform over the
# vocabulary.  Streams: table = seed + 4, token ids = seed + 5.

@dataclass(frozen=True)
class HashWorkload:
    name: str
    T: int
    vocab: int
    n_experts: int
    k: int
    routed_scaling: float

    def with_T(self, T):
        return replace(self, T=T)


HASH_ROUTER = HashWorkload("hash_router", 4096, 129280, 256, 8, 2.5)


def make_hash_table(h: HashWorkload, seed=SEED):
    rng = np.random.default_rng(seed + 4)
    base = rng.integers(0, h.n_experts, size=h.vocab)
    offs = rng.choice(h.n_experts, size=h.k, replace=False)
    return ((base[:, None] + offs[None, :]) % h.n_experts).astype(np.int32)


def make_token_ids(h: HashWorkload, seed=SEED):
    rng = np.random.default_rng(seed + 5)
    return rng.integers(0, h.vocab, size=h.T).astype(np.int32)
