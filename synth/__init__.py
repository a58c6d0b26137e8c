"""Seeded synthetic workloads for the quantized attention path.

This module only draws numbers.  It holds none of the attention method's
arithmetic: no K smoothing, no Q/K/V quantization of the dense path, no
softmax.  Both the CPU oracle (``oracle/``) and the CUDA path read the same
bytes from here, and nothing here depends on either of them.

Generator (one definition, counter-based so any slice can be drawn alone):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the c-th output for seed ``s`` is
  ``mix(s + (c + 1) * 0x9E3779B97F4A7C15)`` with the published finaliser
  ``mix``.  This equals the sequential generator started from state ``s``.
* Box-Muller (1958): normal ``i`` uses outputs ``2i`` and ``2i + 1`` as
  ``u = ((z >> 11) + 0.5) * 2**-53`` and returns
  ``sqrt(-2 ln u1) * cos(2 pi u2)`` in fp64.
* Storage: fp64 -> fp32 (round to nearest even) -> bf16 (round to nearest
  even) for bf16 tensors; fp64 -> fp32 for the K/V rows of the int8 KV cache.

The int8 KV cache of the prompt-attention workloads is written by a cache
writer upstream of the attention call (Strata PR #2092, "Setup": the engine
runs ``--kv int8``; the cache holds int8 K/V with per-token scales).  This
module only draws the fp32 rows that go into it: the device side writes the
cache with the library's own writer, the host side with the oracle's.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 0x5A6E2026
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20

# tensor ids inside one workload
T_Q, T_K, T_V, T_KOFF, T_OUTLIER = 1, 2, 3, 4, 5


def seed_for(config: int, tensor: int, sub: int = 0) -> int:
    """Seed of one tensor of one workload (``sub`` tells the sizes of a sweep apart)."""
    return SEED_BASE + 1000 * config + 100 * sub + tensor


def splitmix64(seed: int, first: int, count: int) -> np.ndarray:
    """Outputs ``first .. first+count-1`` of SplitMix64 started from state ``seed``."""
    c = np.arange(first + 1, first + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + c * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def normal_f64(seed: int, start: int, count: int) -> np.ndarray:
    """Standard normals ``start .. start+count-1`` of stream ``seed`` (fp64)."""
    out = np.empty(count, dtype=np.float64)
    done = 0
    while done < count:
        n = min(_CHUNK, count - done)
        z = splitmix64(seed, 2 * (start + done), 2 * n)
        u = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        out[done:done + n] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        done += n
    return out


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# dense (SageAttention-2 style) workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class DenseWorkload:
    name: str
    config: int
    B: int
    H: int
    Nq: int
    Nk: int
    block: int          # Q and K quantisation block, tokens
    sub: int = 0
    k_offset_std: float = 2.0
    d: int = 128

    @property
    def flops(self) -> int:
        """4 * Nq * Nk * d * H * B: the effective FLOP count of one forward."""
        return 4 * self.Nq * self.Nk * self.d * self.H * self.B


def dense_workloads() -> list[DenseWorkload]:
    """The dense workloads: tiny, the tile-boundary sweep, and the video-DiT layer."""
    out = [DenseWorkload("tiny_b1h2n256", 1, 1, 2, 256, 256, 64)]
    for i, n in enumerate((1, 63, 64, 65, 127, 128, 129, 191, 255, 257)):
        out.append(DenseWorkload(f"sweep_b1h4n{n}", 2, 1, 4, n, n, 64, sub=i))
    out.append(DenseWorkload("videodit_b1h24n37810", 3, 1, 24, 37810, 37810, 128))
    return out


def dense_workload(name: str) -> DenseWorkload:
    for w in dense_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


def dense_inputs(w: DenseWorkload, heads: tuple[int, int] | None = None) -> dict:
    """bf16 bit patterns of Q, K, V in [B, H, N, d] layout.

    ``heads=(h0, h1)`` draws only heads h0..h1-1 of batch 0 (used to check a
    few heads of a large workload on the CPU without drawing all of it).
    K carries a per-(b, h, channel) offset ~ N(0, k_offset_std^2).
    """
    B, H, d = w.B, w.H, w.d
    h0, h1 = (0, H) if heads is None else heads
    if heads is not None and B != 1:
        raise ValueError("head slices are for B == 1")
    nh = h1 - h0
    res = {}
    for key, tid, n in (("q", T_Q, w.Nq), ("k", T_K, w.Nk), ("v", T_V, w.Nk)):
        seed = seed_for(w.config, tid, w.sub)
        per_head = n * d
        arr = np.empty((B * nh, n, d), dtype=np.uint16)
        koff = None
        if key == "k":
            koff = normal_f64(seed_for(w.config, T_KOFF, w.sub), 0, B * H * d).reshape(B * H, d)
            koff = koff * w.k_offset_std
        for j in range(B * nh):
            bh = j if heads is None else h0 + j
            x = normal_f64(seed, bh * per_head, per_head).reshape(n, d)
            if koff is not None:
                x = x + koff[bh][None, :]
            arr[j] = f32_to_bf16_bits(x.astype(np.float32))
        res[key] = arr.reshape(B, nh, n, d)
    return res


# ----------------------------------------------------------------------------
# int8 KV cache prompt-attention workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Int8KVWorkload:
    name: str
    config: int
    Nq: int
    Nk: int
    Hq: int
    Hkv: int
    outlier_frac: float = 0.0
    outlier_gain: float = 8.0
    sub: int = 0
    d: int = 128

    @property
    def q_pos0(self) -> int:
        return self.Nk - self.Nq

    @property
    def flops(self) -> int:
        """4 * Nq * Nk * d * Hq (the dense formula; the causal part is slightly less)."""
        return 4 * self.Nq * self.Nk * self.d * self.Hq

    @property
    def visible_pairs(self) -> int:
        """Number of (query, key) pairs inside the causal window, per query head."""
        p0 = self.q_pos0
        return sum(p0 + i + 1 for i in range(self.Nq))


def int8kv_workloads() -> list[Int8KVWorkload]:
    return [
        Int8KVWorkload("tiny_kv_q96_k300", 6, 96, 300, 8, 2, 0.01),
        Int8KVWorkload("prompt32k_q1024", 4, 1024, 32768, 32, 8),
        Int8KVWorkload("prompt64k_q512_outliers", 5, 512, 65536, 32, 8, 0.01),
    ]


def int8kv_workload(name: str) -> Int8KVWorkload:
    for w in int8kv_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


def outlier_pairs(w: Int8KVWorkload) -> np.ndarray:
    """Distinct flat (kv head * d + channel) indices whose K values are scaled."""
    n = int(round(w.outlier_frac * w.Hkv * w.d))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    picked: list[int] = []
    c = 0
    seed = seed_for(w.config, T_OUTLIER, w.sub)
    while len(picked) < n:
        z = int(splitmix64(seed, c, 1)[0])
        c += 1
        idx = (z >> 11) % (w.Hkv * w.d)
        if idx not in picked:
            picked.append(idx)
    return np.array(sorted(picked), dtype=np.int64)


def int8kv_inputs(w: Int8KVWorkload, kv_heads: tuple[int, int] | None = None) -> dict:
    """q bf16 bits [Nq, Hq, d] and the fp32 K/V rows of the cache, k_raw / v_raw [Hkv, Nk, d].

    ``kv_heads=(g0, g1)`` draws only kv heads g0..g1-1 and the query heads that
    read them (q then has shape [Nq, (g1-g0)*Hq/Hkv, d]).
    """
    d, Nq, Hq, Hkv = w.d, w.Nq, w.Hq, w.Hkv
    g0, g1 = (0, Hkv) if kv_heads is None else kv_heads
    grp = Hq // Hkv
    q = np.empty((Nq, (g1 - g0) * grp, d), dtype=np.uint16)
    qseed = seed_for(w.config, T_Q, w.sub)
    for t in range(Nq):
        base = (t * Hq + g0 * grp) * d
        x = normal_f64(qseed, base, (g1 - g0) * grp * d)
        q[t] = f32_to_bf16_bits(x.astype(np.float32)).reshape((g1 - g0) * grp, d)
    raw = int8kv_raw(w, (g0, g1))
    return {"q": q, "k_raw": raw["k"], "v_raw": raw["v"]}


def int8kv_raw(w: Int8KVWorkload, kv_heads: tuple[int, int] | None = None) -> dict:
    """The fp32 K/V rows [Hkv, Nk, d] before the cache is quantised (outlier channels applied)."""
    d, Nk, Hkv = w.d, w.Nk, w.Hkv
    g0, g1 = (0, Hkv) if kv_heads is None else kv_heads
    outl = outlier_pairs(w)
    res = {}
    for key, tid in (("k", T_K), ("v", T_V)):
        seed = seed_for(w.config, tid, w.sub)
        x = np.empty((g1 - g0, Nk, d), dtype=np.float32)
        for j, g in enumerate(range(g0, g1)):
            x[j] = normal_f64(seed, g * Nk * d, Nk * d).astype(np.float32).reshape(Nk, d)
            if key == "k" and outl.size:
                chans = outl[(outl // d) == g] % d
                x[j][:, chans] *= np.float32(w.outlier_gain)
        res[key] = x
    return res
