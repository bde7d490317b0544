"""Counter-based random streams, exact bf16 rounding and the workload table.

Every tensor is a pure function of (workload, seed): a counter-based
splitmix64 stream per tensor, Box-Muller normals computed in fp64 and rounded
once, round-to-nearest-even, to bf16; Zipf targets by inverse CDF; ignored
rows picked by a seeded Fisher-Yates shuffle. Nothing here computes a loss or
a gradient.

The workload shapes are the ones the pages measure the method on: the
Gravity-16B-A3B head of the Trillion Labs note (V = 151,552, D = 2048,
B = 1, S = 8192), the Gemma 2 (2B) classifier of Cut Cross-Entropy Table 1
(8192 tokens, V = 256,000, D = 2304), a Llama-3-8B head and the 128K-context
Gravity case whose full logits the note says could not be allocated.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

IGNORE_INDEX = -100

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    """The splitmix64 output function (Steele, Lea and Flood, OOPSLA 2014)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _subseed(seed: int, tag: str) -> int:
    """Independent stream seed for one tensor: splitmix64 of seed xor a tag hash."""
    h = 0
    for ch in tag.encode():
        h = (h * 131 + ch) & 0xFFFFFFFFFFFFFFFF
    v = np.array([(seed ^ h) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix64(v + _GAMMA)[0])


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start..start+n-1 of the splitmix64 sequence seeded with `seed`.

    Output i is mix(seed + (i + 1) * gamma) modulo 2^64, which is what the
    sequential generator returns on its (i + 1)-th call.
    """
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        return _mix64(state)


def uniform01(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of each splitmix64 output."""
    return (splitmix64(seed, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (round to nearest, ties to even) in one step.

    The fp64 bit pattern keeps its sign, exponent and top 7 fraction bits; the
    45 dropped bits are rounded to nearest-even by integer addition (a carry
    into the exponent is the correct result). The rounded value has 8
    significant bits, so the cast to fp32 that follows is exact.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value cannot be rounded to bf16 here")
    b = x.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        b = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    f32 = b.view(np.float64).astype(np.float32)
    tiny = (f32 != 0) & (np.abs(f32) < np.float32(2.0 ** -126))
    if np.any(tiny):
        raise ValueError("value below the bf16 normal range")
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def normal_bf16(seed: int, shape: tuple[int, ...], std: float, shift: np.ndarray | None = None) -> np.ndarray:
    """N(0, std^2) samples as bf16 bit patterns (uint16), Box-Muller in fp64.

    Pair k uses uniforms u1 = U[2k], u2 = U[2k+1]; r = sqrt(-2 ln(1 - u1));
    element 2k = r cos(2 pi u2) * std, element 2k+1 = r sin(2 pi u2) * std.
    shift (fp64, one value per index of the last axis) is added to every
    row before the single rounding to bf16.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        u = uniform01(seed, 2 * (p1 - p0), start=2 * p0)
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        t = 2.0 * math.pi * u[1::2]
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        z *= std
        e0, e1 = 2 * p0, min(n, 2 * p1)
        if shift is not None:
            z[: e1 - e0] += shift[np.arange(e0, e1) % shape[-1]]
        out[e0:e1] = f64_to_bf16_bits(z[: e1 - e0])
    return out.reshape(shape)


def zipf_targets(seed: int, n: int, vocab: int, s: float) -> np.ndarray:
    """Token ids with P(id = r - 1) proportional to r^-s, r = 1..vocab (inverse CDF)."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = uniform01(seed, n)
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, vocab - 1).astype(np.int64)


def uniform_targets(seed: int, n: int, vocab: int, start: int = 0) -> np.ndarray:
    u = uniform01(seed, n, start)
    return np.minimum((u * vocab).astype(np.int64), vocab - 1)


def apply_ignore(y: np.ndarray, seed: int, frac: float) -> np.ndarray:
    """Set exactly round(frac * N) rows to IGNORE_INDEX, chosen by Fisher-Yates."""
    y = y.copy()
    n = y.shape[0]
    k = int(math.floor(frac * n + 0.5))
    if k == 0:
        return y
    perm = list(range(n))
    u = uniform01(seed, n)
    for i in range(n - 1, 0, -1):
        j = int(u[i] * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    y[np.array(perm[:k], dtype=np.int64)] = IGNORE_INDEX
    return y


def topk_targets(seed: int, h_bits: np.ndarray, w_bits: np.ndarray, k: int = 16,
                 p_top: float = 0.8, rows_per_block: int = 256) -> np.ndarray:
    """Peaky targets: with probability p_top a uniform pick among the row's k
    largest scores h.w_v (ties broken toward the lower id), else uniform.

    The scores only choose which token ids become targets; they are formed in
    fp64 from the exact bf16 values with a library matmul.
    """
    n, vocab = h_bits.shape[0], w_bits.shape[0]
    u = uniform01(seed, 3 * n).reshape(n, 3)
    w64 = bf16_bits_to_f64(w_bits)
    y = np.empty(n, dtype=np.int64)
    ids = np.arange(vocab, dtype=np.int64)
    for r0 in range(0, n, rows_per_block):
        r1 = min(n, r0 + rows_per_block)
        s = bf16_bits_to_f64(h_bits[r0:r1]) @ w64.T
        kk = min(k, vocab)
        thr = -np.partition(-s, kk - 1, axis=1)[:, kk - 1]
        for i in range(r1 - r0):
            row = r0 + i
            if u[row, 0] < p_top:
                cand = np.nonzero(s[i] >= thr[i])[0]
                order = np.lexsort((ids[cand], -s[i, cand]))
                top = cand[order[:kk]]
                y[row] = top[min(int(u[row, 1] * kk), kk - 1)]
            else:
                y[row] = min(int(u[row, 2] * vocab), vocab - 1)
    return y


@dataclasses.dataclass(frozen=True)
class Workload:
    """One input configuration: shapes, value distributions, target recipe."""
    name: str
    n_rows: int
    hidden: int
    vocab: int
    w_var_times_d: float      # Var(W) = w_var_times_d / D
    targets: str              # "uniform" | "zipf" | "top16"
    ignore_frac: float
    zipf_s: float = 1.1
    description: str = ""
    # H_n = N(0, I) + h_shared * sqrt(D) * u for one seeded unit vector u:
    # a component every row shares, which gives each token a logit offset
    # W_v . u common to all rows (a frequency prior of the vocabulary).
    h_shared: float = 0.0

    @property
    def w_std(self) -> float:
        return math.sqrt(self.w_var_times_d / self.hidden)

    def logits_bytes_bf16(self) -> int:
        """Bytes of the full bf16 [N,V] logits the fused path never allocates."""
        return self.n_rows * self.vocab * 2

    def grad_bytes_bf16(self) -> int:
        """Bytes of bf16 dH and dW together: the least any backward must write."""
        return (self.n_rows + self.vocab) * self.hidden * 2

    def scaled(self, n_rows: int | None = None, hidden: int | None = None,
               vocab: int | None = None) -> "Workload":
        return dataclasses.replace(
            self, name=f"{self.name}-scaled",
            n_rows=self.n_rows if n_rows is None else n_rows,
            hidden=self.hidden if hidden is None else hidden,
            vocab=self.vocab if vocab is None else vocab)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 256, 128, 4096, 1.0, "uniform", 0.05,
                     description="small oracle case, several tiles plus ragged tails"),
    "llama3_8b_head": Workload("llama3_8b_head", 8192, 4096, 128256, 1.0, "zipf", 0.02,
                               description="Llama-3-8B-shaped head, B=1 S=8192"),
    "gravity16b_head": Workload("gravity16b_head", 8192, 2048, 151552, 1.0, "zipf", 0.02,
                                description="Gravity-16B-A3B-shaped head, B=1 S=8192"),
    "gemma2_2b_head": Workload("gemma2_2b_head", 8192, 2304, 256000, 9.0, "top16", 0.0,
                               description="Gemma-2-2B-shaped head, peaky softmax"),
    "gravity16b_head_v65536": Workload("gravity16b_head_v65536", 8192, 2048, 65536, 1.0, "zipf", 0.02,
                                       description="Gravity-16B-A3B head with the vocabulary cut to 65536, "
                                                   "for profiler captures (about 1.3 GB on the device)"),
    "long128k_head": Workload("long128k_head", 131072, 2048, 151552, 1.0, "zipf", 0.10,
                              description="Gravity-16B-A3B head at 128K context"),
    "gemma2_2b_head_prior": Workload("gemma2_2b_head_prior", 8192, 2304, 256000, 9.0, "top16", 0.0,
                                     description="Gemma-2-2B-shaped head whose rows share a component, "
                                                 "so tokens carry a common logit prior", h_shared=2.0),
    "gemma2_2b_head_prior_v65536": Workload("gemma2_2b_head_prior_v65536", 8192, 2304, 65536, 9.0, "top16", 0.0,
                                            description="the same with the vocabulary cut to 65536, for "
                                                        "profiler captures", h_shared=2.0),
}


def make_inputs(wl: Workload, seed: int = 0) -> dict:
    """H [N,D] and W [V,D] as bf16 bit patterns (uint16) and y [N] int64."""
    shift = None
    if wl.h_shared != 0.0:
        u = np.array([0.0])
        while not np.linalg.norm(u) > 0.0:
            u = bf16_bits_to_f64(normal_bf16(_subseed(seed, "Hshared"), (wl.hidden,), 1.0))
        shift = u * (wl.h_shared * math.sqrt(wl.hidden) / np.linalg.norm(u))
    h = normal_bf16(_subseed(seed, "H"), (wl.n_rows, wl.hidden), 1.0, shift)
    w = normal_bf16(_subseed(seed, "W"), (wl.vocab, wl.hidden), wl.w_std)
    if wl.targets == "uniform":
        y = uniform_targets(_subseed(seed, "y"), wl.n_rows, wl.vocab)
    elif wl.targets == "zipf":
        y = zipf_targets(_subseed(seed, "y"), wl.n_rows, wl.vocab, wl.zipf_s)
    elif wl.targets == "top16":
        y = topk_targets(_subseed(seed, "y"), h, w, 16, 0.8)
    else:
        raise ValueError(wl.targets)
    y = apply_ignore(y, _subseed(seed, "ignore"), wl.ignore_frac)
    return {"H": h, "W": w, "y": y, "workload": wl, "seed": seed}
