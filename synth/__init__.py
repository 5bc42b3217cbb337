"""Seeded synthetic inputs for the routed-expert layer.

This module is shared by the CPU oracle, the tests and the benchmark.  It only
draws random numbers and lays them out in the shapes of the MoE workloads; it
holds none of the layer's arithmetic (no routing, no slot assignment, no GEMM).

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used in counter mode: draw ``n`` of a stream
with key ``k`` is ``mix(k + (n + 1) * 0x9E3779B97F4A7C15)``.  Normals come from
the Box-Muller transform of two consecutive draws.  Every tensor has its own
stream key derived from the workload seed and the tensor's name, so any slice
of any tensor can be regenerated independently.

bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
from the fp32 draw); fp32 tensors as ``float32``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, in place on a uint64 array (wrapping arithmetic)."""
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _mix_scalar(v: int) -> int:
    return int(_mix(np.array([v & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def stream_key(seed: int, name: str) -> int:
    """Key of the stream for tensor ``name`` of workload ``seed`` (FNV-1a of the name, mixed)."""
    h = 0xCBF29CE484222325
    for ch in name.encode():
        h ^= ch
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return _mix_scalar(h ^ _mix_scalar(seed * 0x9E3779B97F4A7C15 + 1))


def draws_u64(key: int, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of stream ``key`` as uint64."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        ctr *= _GAMMA
        ctr += np.uint64(key)
        return _mix(ctr)


def _normal_chunk(key: int, start: int, n: int) -> np.ndarray:
    raw = draws_u64(key, 2 * start, 2 * n)
    a = raw[0::2]
    b = raw[1::2]
    u1 = ((a >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u2 = (b >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def _uniform_chunk(key: int, start: int, n: int) -> np.ndarray:
    raw = draws_u64(key, start, n)
    return (raw >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _chunked(fn, key: int, n: int, out: np.ndarray, post) -> np.ndarray:
    starts = list(range(0, n, _CHUNK))

    def work(s):
        m = min(_CHUNK, n - s)
        out[s:s + m] = post(fn(key, s, m))

    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    return out


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    bits = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return ((bits + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(key: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _chunked(_normal_chunk, key, n, out, lambda z: (z * std).astype(np.float32))
    return out.reshape(shape)


def normal_bf16(key: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    _chunked(_normal_chunk, key, n, out,
             lambda z: f32_to_bf16_bits((z * std).astype(np.float32)))
    return out.reshape(shape)


def uniform_f64(key: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    _chunked(_uniform_chunk, key, n, out, lambda u: u)
    return out.reshape(shape)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class MoEConfig:
    """Shape and input recipe of one routed-expert layer workload.

    ``cap`` is the per-expert capacity ceil(cf * T * K / N) with cf = cf_num / cf_den,
    computed in integer arithmetic on the host, as a caller would before its loop.
    """
    name: str
    T: int
    d: int
    N: int
    K: int
    h: int
    cf_num: int
    cf_den: int
    seed: int
    router_std: float = 0.02
    weight_std: float = 0.02
    zipf_s: Optional[float] = None
    backward: bool = False

    @property
    def cap(self) -> int:
        return (self.cf_num * self.T * self.K + self.cf_den * self.N - 1) // (self.cf_den * self.N)

    @property
    def R(self) -> int:
        """Rows of a capacity buffer: the packed rows never exceed N*cap or T*K."""
        return min(self.N * self.cap, self.T * self.K)

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", T=256, d=128, N=8, K=2, h=256, cf_num=5, cf_den=4, seed=0),
    "olmoe": MoEConfig("olmoe", T=8192, d=2048, N=64, K=8, h=1024, cf_num=5, cf_den=4, seed=1),
    "fine_zipf": MoEConfig("fine_zipf", T=16384, d=2048, N=128, K=8, h=768, cf_num=1, cf_den=1,
                           seed=2, zipf_s=1.2),
    "wide": MoEConfig("wide", T=32768, d=4096, N=32, K=4, h=2048, cf_num=3, cf_den=2, seed=3,
                      router_std=0.01),
    "train": MoEConfig("train", T=8192, d=2048, N=64, K=8, h=1024, cf_num=5, cf_den=4, seed=4,
                       backward=True),
    # dropless: cap = T (an expert can take every token, since a token's K
    # experts are distinct), so no route is ever dropped; the capacity buffers
    # hold min(N*cap, T*K) = T*K rows
    "olmoe_dropless": MoEConfig("olmoe_dropless", T=8192, d=2048, N=64, K=8, h=1024, cf_num=8,
                                cf_den=1, seed=5),
}


def gen_x(cfg: MoEConfig) -> np.ndarray:
    """Token activations x ~ N(0, 1), bf16 bits [T, d]."""
    return normal_bf16(stream_key(cfg.seed, "x"), (cfg.T, cfg.d), 1.0)


def gen_router(cfg: MoEConfig) -> np.ndarray:
    """Router weight W_r ~ N(0, router_std^2), fp32 [N, d]."""
    return normal_f32(stream_key(cfg.seed, "w_router"), (cfg.N, cfg.d), cfg.router_std)


def gen_bias(cfg: MoEConfig) -> Optional[np.ndarray]:
    """Per-expert router logit offsets that create Zipf(s) load imbalance, fp32 [N], or None.

    A seeded permutation pi ranks the experts; p_e is proportional to
    (pi(e) + 1)^(-s); the offset is ln p_e minus its mean over experts.
    """
    if cfg.zipf_s is None:
        return None
    u = uniform_f64(stream_key(cfg.seed, "zipf_perm"), (cfg.N,))
    rank = np.empty(cfg.N, dtype=np.int64)
    rank[np.argsort(u, kind="stable")] = np.arange(cfg.N)
    lp = -cfg.zipf_s * np.log(rank.astype(np.float64) + 1.0)
    lp -= np.log(np.exp(lp).sum())
    return (lp - lp.mean()).astype(np.float32)


def gen_expert_weights(cfg: MoEConfig):
    """Stacked expert weights, bf16 bits: W_gate, W_up [N, h, d]; W_down [N, d, h]."""
    s = cfg.weight_std
    wg = normal_bf16(stream_key(cfg.seed, "w_gate"), (cfg.N, cfg.h, cfg.d), s)
    wu = normal_bf16(stream_key(cfg.seed, "w_up"), (cfg.N, cfg.h, cfg.d), s)
    wd = normal_bf16(stream_key(cfg.seed, "w_down"), (cfg.N, cfg.d, cfg.h), s)
    return wg, wu, wd


def gen_dy(cfg: MoEConfig) -> np.ndarray:
    """Upstream gradient dy ~ N(0, 1), bf16 bits [T, d]."""
    return normal_bf16(stream_key(cfg.seed, "dy"), (cfg.T, cfg.d), 1.0)


def gen_topk_idx(seed: int, T: int, N: int, K: int, name: str = "topk_idx") -> np.ndarray:
    """K distinct expert indices per token (uniform, partial Fisher-Yates), int32 [T, K]."""
    u = uniform_f64(stream_key(seed, name), (T, K))
    idx = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        perm = list(range(N))
        for k in range(K):
            j = k + int(u[t, k] * (N - k))
            perm[k], perm[j] = perm[j], perm[k]
        idx[t] = perm[:K]
    return idx


def gen_gates(seed: int, T: int, K: int, name: str = "gates") -> np.ndarray:
    """Positive per-route weights in (0, 1], fp32 [T, K] (not normalised)."""
    u = uniform_f64(stream_key(seed, name), (T, K))
    return (1.0 - u).astype(np.float32)


def gen_bf16(seed: int, shape, name: str, std: float = 1.0) -> np.ndarray:
    """Generic bf16 N(0, std^2) payload for standalone kernel cases."""
    return normal_bf16(stream_key(seed, name), shape, std)
