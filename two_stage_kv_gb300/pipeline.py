"""Device buffers and call sequences of the two-stage path, on top of the C ABI.

`Layer` owns the caches of one attention layer of a single-turn workload:
stage-1 eviction (rkv_snap_evict), KT build, then per decode step an append
(rkv_append_kv) and an HSA step (rkv_hsa_decode).  `MTLayer` keeps the full
cache and runs RocketKV-MT: per turn, stage 1 in mask mode writes the kept
rows straight into the candidate index rows, the KT cache is built over them,
and each decode step appends to the full cache and to the candidate rows.
All arithmetic runs in the CUDA library; this module only allocates buffers
(torch) and passes pointers.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

from . import rkv
from .synth import Workload


def bf16_tensor(bits, device) -> torch.Tensor:
    """uint16 bf16 bit patterns (numpy) -> bf16 tensor on `device`."""
    t = torch.from_numpy(bits.view("int16")).view(torch.bfloat16)
    return t.to(device, non_blocking=False)


def nblk_capacity(tokens: int, blk: int) -> int:
    """KT capacity in blocks for `tokens` candidates, rounded up to a multiple of 8
    (the decode kernel gathers KT rows in 16-byte pieces)."""
    return -(-(-(-tokens // blk)) // 8) * 8


@dataclass
class Budget:
    r: float
    B1: int
    k2: int


def budget(wl: Workload, S: Optional[int] = None) -> Budget:
    r, B1, k2 = rkv.rkv_budget_split(S if S is not None else wl.S, wl.t, wl.blk, wl.W)
    return Budget(r, B1, k2)


class Layer:
    """Single-turn state of one layer: prompt caches in, compacted caches + KT out."""

    def __init__(self, wl: Workload, k: torch.Tensor, v: torch.Tensor, q_obs: torch.Tensor,
                 device="cuda", n_sink: int = 0):
        self.wl = wl
        self.dims = (wl.B, wl.Hq, wl.Hkv, wl.D)
        self.k, self.v, self.q_obs = k, v, q_obs          # [B,Hkv,S,D], [B,Hq,W,D]
        self.cap_in = k.shape[2]
        self.bud = budget(wl)
        self.scale = 1.0 / math.sqrt(wl.D)
        self.n_sink = n_sink
        B, Hkv, D = wl.B, wl.Hkv, wl.D
        self.cap = self.bud.B1 + wl.steps
        self.nblk_cap = nblk_capacity(self.cap, wl.blk)
        self.kc = torch.empty(B, Hkv, self.cap, D, dtype=torch.bfloat16, device=device)
        self.vc = torch.empty_like(self.kc)
        self.keep = torch.empty(B, Hkv, self.bud.B1, dtype=torch.int32, device=device)
        self.kt = torch.empty(B, Hkv, 2, D, self.nblk_cap, dtype=torch.bfloat16, device=device)
        self.pooled = torch.empty(B, Hkv, max(wl.S - wl.W, 1), dtype=torch.float32, device=device)
        self.ws_bytes = rkv.rkv_snap_evict_workspace(self.dims, wl.S, wl.W)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty(B, wl.Hq, D, dtype=torch.float32, device=device)
        self.sel_blocks = torch.empty(B, Hkv, self.bud.k2, dtype=torch.int32, device=device)
        self.sel_channels = torch.empty(B, Hkv, wl.k1, dtype=torch.int32, device=device)
        self.n = 0

    def stage1(self, stream=None, pooled: bool = True):
        wl = self.wl
        rkv.rkv_snap_evict(self.dims, self.q_obs, wl.W, self.k, self.v, self.cap_in, wl.S, wl.P, self.n_sink,
                           self.bud.B1, self.scale, self.keep, self.bud.B1, self.kc, self.vc, self.cap,
                           self.pooled if pooled else None, self.ws, self.ws_bytes, stream)
        self.n = self.bud.B1

    def build_kt(self, stream=None):
        rkv.rkv_build_kt(self.dims, self.kc, self.cap, self.n, None, 0, self.wl.blk, self.kt, self.nblk_cap, stream)

    def stage1_select(self, stream=None, pooled: bool = True):
        """Stage 1 in mask mode: only the keep list (and optionally the pooled scores)."""
        wl = self.wl
        rkv.rkv_snap_evict(self.dims, self.q_obs, wl.W, self.k, self.v, self.cap_in, wl.S, wl.P, self.n_sink,
                           self.bud.B1, self.scale, self.keep, self.bud.B1, None, None, 0,
                           self.pooled if pooled else None, self.ws, self.ws_bytes, stream)

    def compact_kt(self, stream=None):
        """Compaction of the kept rows with the KT cache built on the way (after stage1_select)."""
        rkv.rkv_compact_kt(self.dims, self.k, self.v, self.cap_in, self.keep, self.bud.B1, self.bud.B1, self.kc,
                           self.vc, self.cap, self.wl.blk, self.kt, self.nblk_cap, stream)
        self.n = self.bud.B1

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        rkv.rkv_append_kv(self.dims, k_new, v_new, self.kc, self.vc, self.cap, self.n, self.n, None, 0, self.kt,
                          self.nblk_cap, self.wl.blk, stream)
        self.n += 1

    def decode(self, q: torch.Tensor, stream=None, selections: bool = True, out: Optional[torch.Tensor] = None):
        wl = self.wl
        rkv.rkv_hsa_decode(self.dims, q, self.kc, self.vc, self.cap, self.n, self.kt, self.nblk_cap, wl.blk, wl.k1,
                           self.bud.k2, self.scale, self.out if out is None else out,
                           self.sel_blocks if selections else None, self.sel_channels if selections else None,
                           stream)

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None,
             selections: bool = True, out: Optional[torch.Tensor] = None):
        """One decode step with the append fused into the HSA launch."""
        wl = self.wl
        rkv.rkv_hsa_decode(self.dims, q, self.kc, self.vc, self.cap, self.n, self.kt, self.nblk_cap, wl.blk, wl.k1,
                           self.bud.k2, self.scale, self.out if out is None else out,
                           self.sel_blocks if selections else None, self.sel_channels if selections else None,
                           k_new, v_new, stream)
        self.n += 1

    # -- e4m3 (FP8) storage of the compacted cache -------------------------------

    def enable_fp8(self, k_scale: torch.Tensor, v_scale: torch.Tensor):
        """Allocate e4m3 code caches; k_scale / v_scale are [B, Hkv] fp32 (value = code * scale)."""
        wl = self.wl
        B, Hkv, D = wl.B, wl.Hkv, wl.D
        dev = self.kc.device
        self.k_scale, self.v_scale = k_scale, v_scale
        self.nblk_cap8 = -(-nblk_capacity(self.cap, wl.blk) // 16) * 16
        self.kc8 = torch.empty(B, Hkv, self.cap, D, dtype=torch.uint8, device=dev)
        self.vc8 = torch.empty_like(self.kc8)
        self.kt8 = torch.empty(B, Hkv, 2, D, self.nblk_cap8, dtype=torch.uint8, device=dev)

    def compact_kt_fp8(self, stream=None):
        rkv.rkv_compact_kt_fp8(self.dims, self.k, self.v, self.cap_in, self.keep, self.bud.B1, self.bud.B1,
                               self.k_scale, self.v_scale, self.kc8, self.vc8, self.cap, self.wl.blk, self.kt8,
                               self.nblk_cap8, stream)
        self.n = self.bud.B1

    def step_fp8(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None,
                 selections: bool = True, out: Optional[torch.Tensor] = None):
        """One decode step over the e4m3 cache with the append fused in."""
        wl = self.wl
        rkv.rkv_hsa_decode_fp8(self.dims, q, self.kc8, self.vc8, self.cap, self.n, self.k_scale, self.v_scale,
                               self.kt8, self.nblk_cap8, wl.blk, wl.k1, self.bud.k2, self.scale,
                               self.out if out is None else out, self.sel_blocks if selections else None,
                               self.sel_channels if selections else None, k_new, v_new, stream)
        self.n += 1

    def reset_decode(self):
        """Forget appended tokens (the next stage1() re-creates the compacted caches)."""
        self.n = self.bud.B1


class MTLayer:
    """RocketKV-MT state: the full cache stays resident; stage 2 reads it through idx.

    reading="candidates": stage-2 blocks run over the candidate sequence (the
    stage-1 survivors, then the decoded tokens) read through idx.
    reading="full_blocks": stage-2 blocks are fixed runs of blk rows of the full
    cache; a survivor mask over the turn's prompt rows marks the candidates.
    """

    def __init__(self, wl: Workload, device="cuda", reading: str = "candidates"):
        if reading not in ("candidates", "full_blocks"):
            raise ValueError(reading)
        self.reading = reading
        self.wl = wl
        self.dims = (wl.B, wl.Hq, wl.Hkv, wl.D)
        B, Hkv, D = wl.B, wl.Hkv, wl.D
        self.cap = wl.cap()
        self.k = torch.empty(B, Hkv, self.cap, D, dtype=torch.bfloat16, device=device)
        self.v = torch.empty_like(self.k)
        self.budgets = [budget(wl, wl.turn_context(t)) for t in range(wl.n_turns)]
        self.idx_cap = max(b.B1 for b in self.budgets) + wl.steps
        self.nblk_cap = nblk_capacity(self.idx_cap, wl.blk)
        self.idx = torch.zeros(B, Hkv, self.idx_cap, dtype=torch.int32, device=device)
        if reading == "full_blocks":
            self.nblk_cap = nblk_capacity(self.cap, wl.blk)
            self.mask_ld = (self.cap + 31) // 32
            self.mask = torch.zeros(B, Hkv, self.mask_ld, dtype=torch.int32, device=device)
        self.n_prompt = 0
        self.kt = torch.empty(B, Hkv, 2, D, self.nblk_cap, dtype=torch.bfloat16, device=device)
        S_max = wl.turn_context(wl.n_turns - 1)
        self.ws_bytes = rkv.rkv_snap_evict_workspace(self.dims, S_max, wl.W)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.pooled = torch.empty(B, Hkv, S_max - wl.W, dtype=torch.float32, device=device)
        self.out = torch.empty(B, wl.Hq, D, dtype=torch.float32, device=device)
        self.k2 = max(b.k2 for b in self.budgets)
        self.sel_blocks = torch.empty(B, Hkv, self.k2, dtype=torch.int32, device=device)
        self.sel_channels = torch.empty(B, Hkv, wl.k1, dtype=torch.int32, device=device)
        self.scale = 1.0 / math.sqrt(wl.D)
        self.rows = 0      # rows of the full cache in use
        self.n = 0         # candidates of the current turn
        self.turn = -1

    def add_prompt(self, k: torch.Tensor, v: torch.Tensor):
        """Append a turn's new prompt tokens [B, Hkv, T, D] to the full cache (a plain copy)."""
        T = k.shape[2]
        self.k[:, :, self.rows:self.rows + T].copy_(k)
        self.v[:, :, self.rows:self.rows + T].copy_(v)
        self.rows += T

    def stage1(self, q_obs: torch.Tensor, stream=None):
        """Stage 1 in mask mode over the whole cumulative cache; kept rows -> idx[:, :, :B1]."""
        self.turn += 1
        bud = self.budgets[self.turn]
        wl = self.wl
        rkv.rkv_snap_evict(self.dims, q_obs, wl.W, self.k, self.v, self.cap, self.rows, wl.P, 0, bud.B1,
                           self.scale, self.idx, self.idx_cap, None, None, 0, self.pooled, self.ws, self.ws_bytes,
                           stream)
        self.n = bud.B1
        self.n_prompt = self.rows
        if self.reading == "full_blocks":
            rkv.rkv_keep_mask(self.dims, self.idx, self.idx_cap, bud.B1, self.n_prompt, self.mask, self.mask_ld,
                              stream)

    def build_kt(self, stream=None):
        if self.reading == "full_blocks":
            rkv.rkv_build_kt_masked(self.dims, self.k, self.cap, self.rows, self.mask, self.mask_ld, self.n_prompt,
                                    self.wl.blk, self.kt, self.nblk_cap, stream)
            return
        rkv.rkv_build_kt(self.dims, self.k, self.cap, self.n, self.idx, self.idx_cap, self.wl.blk, self.kt,
                         self.nblk_cap, stream)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        if self.reading == "full_blocks":
            raise RuntimeError("the full-block reading appends inside step()")
        rkv.rkv_append_kv(self.dims, k_new, v_new, self.k, self.v, self.cap, self.n, self.rows, self.idx,
                          self.idx_cap, self.kt, self.nblk_cap, self.wl.blk, stream)
        self.n += 1
        self.rows += 1

    def _masked(self, q, k_new, v_new, stream):
        wl = self.wl
        k2 = self.budgets[self.turn].k2
        rkv.rkv_hsa_decode_mt_masked(self.dims, q, self.k, self.v, self.cap, self.rows, self.mask, self.mask_ld,
                                     self.n_prompt, self.kt, self.nblk_cap, wl.blk, wl.k1, k2, self.scale, self.out,
                                     self.sel_blocks, self.sel_channels, k_new, v_new, stream)

    def decode(self, q: torch.Tensor, stream=None):
        wl = self.wl
        k2 = self.budgets[self.turn].k2
        if self.reading == "full_blocks":
            self._masked(q, None, None, stream)
            return
        rkv.rkv_hsa_decode_mt(self.dims, q, self.k, self.v, self.cap, self.idx, self.idx_cap, self.n, self.kt,
                              self.nblk_cap, wl.blk, wl.k1, k2, self.scale, self.out, self.sel_blocks,
                              self.sel_channels, stream=stream)

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """One MT decode step with the append (full cache row + candidate index) fused in."""
        wl = self.wl
        k2 = self.budgets[self.turn].k2
        if self.reading == "full_blocks":
            self._masked(q, k_new, v_new, stream)
        else:
            rkv.rkv_hsa_decode_mt(self.dims, q, self.k, self.v, self.cap, self.idx, self.idx_cap, self.n, self.kt,
                                  self.nblk_cap, wl.blk, wl.k1, k2, self.scale, self.out, self.sel_blocks,
                                  self.sel_channels, k_new, v_new, self.rows, stream)
        self.n += 1
        self.rows += 1
