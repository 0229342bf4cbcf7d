"""Seeded synthetic inputs for the two-stage compressed decode path.

This module only draws numbers.  It holds none of the method's arithmetic:
no softmax, pooling, top-k, block bounds or attention.  Both the CPU oracle
(through the tests) and the CUDA path (through the tests and the benchmark)
take their inputs from here, so the two sides always see bit-identical bf16
values.

Every tensor slice is drawn from its own PCG64 stream keyed by
(workload seed, layer, tensor tag, batch row, head), so any single
(batch, head) slice can be regenerated without drawing the rest.  bf16
values are kept as uint16 bit patterns (round-to-nearest-even from fp32).

Workload shapes follow the long-context settings of "RocketKV: Accelerating
Long-Context LLM Inference via Two-Stage KV Cache Compression" (experiments:
Llama3.1-8B-Instruct and Mistral-7B-Instruct GQA shapes, NIAH at 109K tokens
with budget 256; the 70B batch-32 32K example of the introduction).  Model
weights and benchmark datasets are not used: synthetic Gaussian keys, values
and queries with planted outlier channels and planted "needle" keys stand in
for them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# bf16 bit helpers (storage format only)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (a single attention layer unless layers > 1)."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    S: int                 # prompt length (first turn for multi-turn workloads)
    t: int                 # total token budget per GQA group
    blk: int               # stage-2 block (page) size in tokens
    k1: int                # channels kept by the |q| top-k
    steps: int             # decode steps (per turn for multi-turn workloads)
    W: int = 32            # observation window
    P: int = 63            # stage-1 pooling kernel
    n_needles: int = 0
    outliers: int = 0      # outlier channels per KV head
    outlier_scale: float = 8.0
    lognormal_sigma: float = 0.0   # per-channel K/V scale ~ LogNormal(0, sigma) when > 0
    layers: int = 1
    mt: bool = False
    turn_appends: Tuple[int, ...] = ()   # new prompt tokens appended at each later turn
    seed: int = 1000

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_turns(self) -> int:
        return 1 + len(self.turn_appends)

    def turn_context(self, turn: int) -> int:
        """Cumulative context length seen by stage 1 at the start of `turn`."""
        s = self.S
        for i in range(turn):
            s += self.steps + self.turn_appends[i]
        return s

    def cap(self) -> int:
        """Rows needed in a full (uncompacted) cache for the whole workload."""
        return self.turn_context(self.n_turns - 1) + self.steps


WORKLOADS: Dict[str, Workload] = {
    # Llama3.1-8B-shaped single layer, 4K prompt, c = 16, needles.
    "needle_b1_4k": Workload("needle_b1_4k", B=1, Hq=32, Hkv=8, D=128, S=4096, t=256, blk=16, k1=32,
                             steps=8, n_needles=8, outliers=4, seed=1001),
    # Headline: batch 8, 32K context, budget 1024 (c = 32).
    "b8_32k": Workload("b8_32k", B=8, Hq=32, Hkv=8, D=128, S=32768, t=1024, blk=16, k1=32,
                       steps=64, outliers=4, seed=1002),
    # Extreme compression: 109,000-token prompt, budget 256 (~426x), 16 needles.
    "needle_b1_109k": Workload("needle_b1_109k", B=1, Hq=32, Hkv=8, D=128, S=109000, t=256, blk=16,
                               k1=16, steps=128, n_needles=16, outliers=4, seed=1003),
    # Llama3.1-70B-shaped 4-layer stack, batch 32, 32K, budget 2048, block 32.
    "l70b_b32_32k": Workload("l70b_b32_32k", B=32, Hq=64, Hkv=8, D=128, S=32768, t=2048, blk=32,
                             k1=64, steps=32, lognormal_sigma=0.5, layers=4, seed=1004),
    # Multi-turn (MT): Mistral-7B-shaped, batch 4, turns of 16K, +4K, +4K, budget 512.
    "mt_b4_16k": Workload("mt_b4_16k", B=4, Hq=32, Hkv=8, D=128, S=16384, t=512, blk=16, k1=32,
                          steps=32, mt=True, turn_appends=(4096, 4096), seed=1005),
}


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (for reduced-size parity cases)."""
    d = dict(wl.__dict__)
    d.update(kw)
    return Workload(**d)


# ---------------------------------------------------------------------------
# Streams
# ---------------------------------------------------------------------------

_TAGS = {"k": 1, "v": 2, "qobs": 3, "qdec": 4, "knew": 5, "vnew": 6, "outl": 7, "scale": 8,
         "needle": 9}


def _rng(wl: Workload, layer: int, tag: str, *ids: int) -> np.random.Generator:
    ss = np.random.SeedSequence([wl.seed, layer, _TAGS[tag], *[int(i) + 1 for i in ids]])
    return np.random.Generator(np.random.PCG64(ss))


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def outlier_channels(wl: Workload, layer: int, hk: int) -> np.ndarray:
    if wl.outliers <= 0:
        return np.zeros(0, dtype=np.int64)
    r = _rng(wl, layer, "outl", hk)
    return np.sort(r.choice(wl.D, size=wl.outliers, replace=False))


def channel_scale(wl: Workload, layer: int, hk: int) -> Optional[np.ndarray]:
    if wl.lognormal_sigma <= 0:
        return None
    r = _rng(wl, layer, "scale", hk)
    return np.exp(wl.lognormal_sigma * _normal(r, (wl.D,)).astype(np.float64)).astype(np.float32)


def _key_transform(wl: Workload, layer: int, hk: int, x: np.ndarray) -> np.ndarray:
    ch = outlier_channels(wl, layer, hk)
    if ch.size:
        x[..., ch] *= np.float32(wl.outlier_scale)
    s = channel_scale(wl, layer, hk)
    if s is not None:
        x *= s
    return x


def _value_transform(wl: Workload, layer: int, hk: int, x: np.ndarray) -> np.ndarray:
    s = channel_scale(wl, layer, hk)
    if s is not None:
        x *= s
    return x


def _query_transform(wl: Workload, layer: int, hk: int, x: np.ndarray) -> np.ndarray:
    ch = outlier_channels(wl, layer, hk)
    if ch.size:
        x[..., ch] *= np.float32(wl.outlier_scale)
    return x


# --- decode-time inputs (small) -------------------------------------------


def q_decode(wl: Workload, layer: int = 0, turn: int = 0) -> np.ndarray:
    """Decode queries, bf16 bits [steps, B, Hq, D]."""
    out = np.empty((wl.steps, wl.B, wl.Hq, wl.D), dtype=np.uint16)
    for b in range(wl.B):
        for hq in range(wl.Hq):
            hk = hq // wl.G
            x = _normal(_rng(wl, layer, "qdec", turn, b, hq), (wl.steps, wl.D))
            out[:, b, hq] = f32_to_bf16_bits(_query_transform(wl, layer, hk, x))
    return out


def kv_new(wl: Workload, layer: int = 0, turn: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Keys and values appended at each decode step, bf16 bits [steps, B, Hkv, D]."""
    kn = np.empty((wl.steps, wl.B, wl.Hkv, wl.D), dtype=np.uint16)
    vn = np.empty_like(kn)
    for b in range(wl.B):
        for hk in range(wl.Hkv):
            xk = _normal(_rng(wl, layer, "knew", turn, b, hk), (wl.steps, wl.D))
            xv = _normal(_rng(wl, layer, "vnew", turn, b, hk), (wl.steps, wl.D))
            kn[:, b, hk] = f32_to_bf16_bits(_key_transform(wl, layer, hk, xk))
            vn[:, b, hk] = f32_to_bf16_bits(_value_transform(wl, layer, hk, xv))
    return kn, vn


def needle_positions(wl: Workload, layer: int, b: int) -> np.ndarray:
    """Token positions (inside the first-turn prefix, before the window) of the needles."""
    if wl.n_needles <= 0:
        return np.zeros(0, dtype=np.int64)
    r = _rng(wl, layer, "needle", b)
    return np.sort(r.choice(wl.S - wl.W, size=wl.n_needles, replace=False))


def needle_step(wl: Workload, i: int) -> int:
    """Decode step whose query needle i answers (i mod steps)."""
    return i % wl.steps


def needle_directions(wl: Workload, layer: int, qdec_bits: np.ndarray, b: int, hk: int) -> np.ndarray:
    """Unit direction of needle i = the group-summed decode query of step i mod steps, float64 [n_needles, D]."""
    steps = [needle_step(wl, i) for i in range(wl.n_needles)]
    q = bf16_bits_to_f64(qdec_bits[steps, b, hk * wl.G:(hk + 1) * wl.G]).sum(axis=1)
    return q / np.linalg.norm(q, axis=-1, keepdims=True)


# --- prompt-time inputs (large) -------------------------------------------


def kv_slice(wl: Workload, layer: int, b: int, hk: int, qdec_bits: Optional[np.ndarray] = None,
             lo: int = 0, hi: Optional[int] = None, turn: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Prompt keys/values of one (batch row, KV head), bf16 bits [rows, D].

    For turn 0 the rows are the prompt positions [0, S).  For later turns of a
    multi-turn workload the rows are that turn's newly appended prompt tokens.
    Needle keys (turn 0 only) need the decode queries `qdec_bits`.
    """
    n = wl.S if turn == 0 else wl.turn_appends[turn - 1]
    hi = n if hi is None else hi
    xk = _normal(_rng(wl, layer, "k", turn, b, hk), (n, wl.D))[lo:hi]
    xv = _normal(_rng(wl, layer, "v", turn, b, hk), (n, wl.D))[lo:hi]
    xk = _key_transform(wl, layer, hk, xk)
    xv = _value_transform(wl, layer, hk, xv)
    if turn == 0 and wl.n_needles > 0:
        assert qdec_bits is not None, "needle keys need the decode queries"
        dirs = needle_directions(wl, layer, qdec_bits, b, hk)
        alpha = 8.0 * math.sqrt(wl.D)
        for i, p in enumerate(needle_positions(wl, layer, b)):
            if lo <= p < hi:
                xk[p - lo] = (alpha * dirs[i]).astype(np.float32)
    return f32_to_bf16_bits(xk), f32_to_bf16_bits(xv)


def q_obs(wl: Workload, layer: int = 0, qdec_bits: Optional[np.ndarray] = None, turn: int = 0) -> np.ndarray:
    """Observation-window queries (the last W prompt tokens), bf16 bits [B, Hq, W, D].

    With needles, every window query gets sqrt(D) * (sum of the needle
    directions of its group) added, so the prompt tail "asks about" them.
    """
    out = np.empty((wl.B, wl.Hq, wl.W, wl.D), dtype=np.uint16)
    for b in range(wl.B):
        for hq in range(wl.Hq):
            hk = hq // wl.G
            x = _query_transform(wl, layer, hk, _normal(_rng(wl, layer, "qobs", turn, b, hq), (wl.W, wl.D)))
            if turn == 0 and wl.n_needles > 0:
                assert qdec_bits is not None
                bias = math.sqrt(wl.D) * needle_directions(wl, layer, qdec_bits, b, hk).sum(axis=0)
                x = (x.astype(np.float64) + bias).astype(np.float32)
            out[b, hq] = f32_to_bf16_bits(x)
    return out


def _workers() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def kv_full(wl: Workload, layer: int = 0, qdec_bits: Optional[np.ndarray] = None, turn: int = 0,
            out_k: Optional[np.ndarray] = None, out_v: Optional[np.ndarray] = None,
            row0: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Whole prompt K/V for a turn, bf16 bits.

    Without `out_k`/`out_v` returns new [B, Hkv, rows, D] arrays.  With them,
    writes rows [row0, row0 + rows) of caller arrays shaped [B, Hkv, cap, D].
    """
    n = wl.S if turn == 0 else wl.turn_appends[turn - 1]
    if out_k is None:
        out_k = np.empty((wl.B, wl.Hkv, n, wl.D), dtype=np.uint16)
        out_v = np.empty_like(out_k)
        row0 = 0

    def one(bh):
        b, hk = divmod(bh, wl.Hkv)
        k, v = kv_slice(wl, layer, b, hk, qdec_bits, turn=turn)
        out_k[b, hk, row0:row0 + n] = k
        out_v[b, hk, row0:row0 + n] = v

    with ThreadPoolExecutor(_workers()) as ex:
        list(ex.map(one, range(wl.B * wl.Hkv)))
    return out_k, out_v


@dataclass
class LayerInputs:
    """Everything one layer of a single-turn workload consumes (bf16 bits)."""

    k: np.ndarray          # [B, Hkv, S, D]
    v: np.ndarray
    q_obs: np.ndarray      # [B, Hq, W, D]
    q_dec: np.ndarray      # [steps, B, Hq, D]
    k_new: np.ndarray      # [steps, B, Hkv, D]
    v_new: np.ndarray
    needles: List[np.ndarray] = field(default_factory=list)   # per batch row


def layer_inputs(wl: Workload, layer: int = 0) -> LayerInputs:
    qd = q_decode(wl, layer)
    k, v = kv_full(wl, layer, qd)
    kn, vn = kv_new(wl, layer)
    return LayerInputs(k=k, v=v, q_obs=q_obs(wl, layer, qd), q_dec=qd, k_new=kn, v_new=vn,
                       needles=[needle_positions(wl, layer, b) for b in range(wl.B)])


def small_random(rng_seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """Plain N(0, scale^2) bf16 bits of any shape (for unit and edge-case tests)."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([rng_seed, 77])))
    return f32_to_bf16_bits(_normal(r, shape) * np.float32(scale))
