"""CPU oracle for the two-stage compressed decode path (RocketKV).

TEST INFRASTRUCTURE ONLY.  This file is plain, slow, obviously correct
numpy in float64.  It exists so the tests, the smoke check and the
benchmark's CPU baseline can check and time the CUDA library against an
independent statement of the method.  The product path never imports it,
and it shares no code with the CUDA library (the only common module is the
seeded input generator, which draws numbers and holds no method arithmetic).

Sources (cited by page title and section):
  [RKV]  "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV
         Cache Compression" (papercache digest of arXiv:2502.14051, ICML 2025).
         Sections used: "方法细节" (method details) -- SnapKV stage, GQA
         group-level selection, pooling kernel 63, HSA steps 1-3 and
         Algorithm 1, RocketKV-MT, token-budget definition, the adaptive split
         factor r, the split inside HSA with its c = 64 worked example, and
         Table 1 (storage and traffic).
  [GUIDE] "RocketKV Guide: Two-Stage KV Cache Compression for LLMs"
         (aifetchly blog): observation window of 32 tokens, softmax scale
         1/sqrt(D), [batch, heads, seq, head_dim] layout, the KV-size formula.

Readings where the pages are silent or ambiguous (each marked READING below):
  R1 window = the last W prompt tokens' queries; those W tokens are always kept
     and only the prefix [0, S-W) competes for the remaining B1-W slots.
  R2 causal softmax per window row over keys 0..(S-W+w); its denominator
     includes the window keys, only prefix probabilities are summed.
  R3 group aggregation is a sum over the G query heads and W window rows.
  R4 pooling is a max-pool, kernel P, stride 1, window clipped at the ends.
  R5 every top-k keeps the larger value; equal values go to the lower index;
     returned index sets are sorted ascending.
  R6 B1 = floor(S * c**-r) clamped to [min(W+1, S), S]; k2 = floor((t/2)/blk)
     blocks, at least 1 (the even step-2 / step-3 split of the budget).
  R7 sign at zero: a zero group sum takes Kmax (Algorithm 1 tests g_i >= 0);
     with the box form of R8 the choice cannot change a score.
  R8 block score = the maximum of the kept-channel part of qbar . x over the
     block's box Kmin <= x <= Kmax (qbar = group-summed q), i.e. per channel
     the larger of qbar_c * Kmax_c and qbar_c * Kmin_c; no scale or softmax is
     applied to it.
  R9 a partial last block uses only its valid tokens, for both the bounds and
     attention, and competes like any other block.
  R10 multi-turn: stage-2 candidates are the stage-1 survivors (ascending)
     followed by the tokens decoded since; blocks are formed over that
     compacted index sequence and K/V rows are read from the full cache.
  R12 FP8 storage (not on the pages; a storage option of this build): the
     compacted K and V hold e4m3 codes (1 sign, 4 exponent bits with bias 7,
     3 mantissa bits, no infinities, S.1111.111 = NaN, largest 448) of
     x / scale, rounded to nearest even in fp32 and saturated to +-448, with a
     caller-given fp32 scale per (batch, KV head) for K and for V; a row's
     value is code * scale.  The KT bounds are the max / min of the stored
     key codes (exact), and block scores are taken on code values (the
     positive K scale does not change their order).
  R11 multi-turn, the other reading (built beside R10): blocks are the fixed
     runs of blk rows of the full cache itself.  A row is a candidate when
     stage 1 kept it (prompt rows [0, n_prompt)) or when it was decoded after
     that prompt (rows >= n_prompt).  Kmax/Kmin of a block run over its
     candidate rows only; a block without candidates scores -inf; the block
     holding the newest row is always chosen (it scores +inf) when it holds a
     candidate; attention covers the candidate rows of the chosen blocks.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# Budget split   [RKV] "方法细节": token budget, adaptive split factor r,
#                split inside HSA, worked example (c = 64), Table 1.
# ---------------------------------------------------------------------------


def split_factor(c: float, r_override: Optional[float] = None) -> float:
    """r = min(0.2 + 0.06 * log2(c), 0.8), kept inside [0.2, 0.8]  [RKV, adaptive split]."""
    if r_override is not None and r_override >= 0:
        return float(r_override)
    r = min(0.2 + 0.06 * math.log2(c), 0.8)
    return max(r, 0.2)


def budget_split(S: int, t: int, blk: int, W: int = 32,
                 r_override: Optional[float] = None) -> Tuple[float, int, int]:
    """(r, B1, k2): stage-1 keep count and stage-2 block count for prompt S, budget t.

    c = S / t is the total compression.  Stage 1 compresses by c**r, so it keeps
    B1 = floor(S / c**r) tokens (READING R6).  The budget t is the KV-pair
    traffic of HSA steps 2 and 3, split evenly, so step 3 reads t/2 tokens,
    i.e. k2 = floor((t/2)/blk) blocks.
    """
    c = S / t
    r = split_factor(c, r_override)
    B1 = int(math.floor(S * c ** (-r)))
    B1 = max(min(W + 1, S), min(B1, S))
    k2 = max(1, (t // 2) // blk)
    return r, B1, k2


def stage_factors(c: float, r: float) -> Tuple[float, float]:
    """Compression of stage 1 (c**r) and of stage 2 (c**(1-r))."""
    return c ** r, c ** (1.0 - r)


def hsa_internal_split(c: float, r: float) -> Tuple[int, float]:
    """Split of stage 2's c**(1-r) between sequence and head dims  [RKV, split inside HSA].

    Page size = ceil(c**((1-r)/2)); the head dimension gets c**(1-r) / page.
    """
    c2 = c ** (1.0 - r)
    page = int(math.ceil(c2 ** 0.5))
    return page, c2 / page


def table1_storage_traffic(c: float, r: float) -> Dict[str, Tuple[float, float]]:
    """Normalised (storage, traffic) per method at compression c  [RKV, Table 1]."""
    return {
        "Full-KV": (1.0, 1.0),
        "DuoAttention": (1.0 / c, 1.0 / c),
        "SnapKV": (1.0 / c, 1.0 / c),
        "Quest": (1.0 + 1.0 / c, 1.0 / c),
        "SparQ": (2.0, 1.0 / c),
        "RocketKV": (1.0 / c ** r + 2.0 / c ** ((1.0 + r) / 2.0), 1.0 / c),
        "RocketKV-MT": (1.0 + 2.0 / c ** ((1.0 + r) / 2.0), 1.0 / c),
    }


def kv_cache_bytes(layers: int, n_kv_heads: int, head_dim: int, seq: int, bytes_per: int,
                   batch: int = 1) -> int:
    """2 * L * H_kv * D * S * bytes (K and V) per sequence, times batch  [GUIDE, KV size]."""
    return 2 * layers * n_kv_heads * head_dim * seq * bytes_per * batch


# ---------------------------------------------------------------------------
# Generic top-k  (READING R5)
# ---------------------------------------------------------------------------


def topk_lowest_index(values: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values; among equal values the lower index wins.

    Returned sorted ascending.  If k >= len(values) every index is returned.
    """
    values = np.asarray(values, dtype=np.float64)
    n = values.shape[0]
    if k >= n:
        return np.arange(n, dtype=np.int64)
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    # lexsort: last key is primary.  Primary = -value ascending, then index ascending.
    order = np.lexsort((np.arange(n), -values))
    return np.sort(order[:k]).astype(np.int64)


def kth_value(values: np.ndarray, k: int) -> float:
    """Value of the k-th largest element (1-based k) under the same ordering."""
    values = np.asarray(values, dtype=np.float64)
    order = np.lexsort((np.arange(values.shape[0]), -values))
    return float(values[order[min(k, values.shape[0]) - 1]])


# ---------------------------------------------------------------------------
# Stage 1: SnapKV eviction  [RKV "方法细节": SnapKV stage, GQA group-level
#          selection, pooling kernel 63]  [GUIDE "Stage 1": window 32, 1/sqrt(D)]
# ---------------------------------------------------------------------------


def snap_scores(q_obs_group: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Aggregated observation-window attention of each prefix key.

    q_obs_group: [G, W, D] float64 -- window queries of the G heads of one group.
    K:           [S, D] float64    -- that group's prompt keys.
    Returns score[j], j < S - W:  sum over heads g and window rows w of
    softmax_j(q_{g,w} . k_j * scale), the softmax over keys 0..S-W+w
    (causal, READING R2), summed over the group (READING R3).
    """
    G, W, D = q_obs_group.shape
    S = K.shape[0]
    Q = q_obs_group.reshape(G * W, D)
    logits = (Q @ K.T) * scale                           # [G*W, S]
    pos = (S - W) + np.tile(np.arange(W), G)             # absolute position of each row
    keep = np.arange(S)[None, :] <= pos[:, None]
    logits = np.where(keep, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    return p[:, : S - W].sum(axis=0)


def max_pool(x: np.ndarray, P: int) -> np.ndarray:
    """1-D max-pool, kernel P (odd), stride 1, window clipped at the ends (READING R4)."""
    n = x.shape[0]
    half = P // 2
    out = np.empty(n, dtype=np.float64)
    for j in range(n):
        out[j] = x[max(0, j - half): min(n, j + half + 1)].max()
    return out


def max_pool_fast(x: np.ndarray, P: int) -> np.ndarray:
    """Same as max_pool, vectorised over the shifts (the loop above is the definition)."""
    n = x.shape[0]
    half = P // 2
    pad = np.full(n + 2 * half, -np.inf)
    pad[half: half + n] = x
    out = pad[0:n].copy()
    for s in range(1, 2 * half + 1):
        np.maximum(out, pad[s: s + n], out=out)
    return out


def snap_keep(q_obs_group: np.ndarray, K: np.ndarray, B1: int, W: int, P: int, scale: float,
              n_sink: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Stage-1 keep set of one GQA group: (keep indices ascending [B1], pooled scores).

    The last W tokens (the observation window) and the first n_sink tokens are
    always kept; the other B1 - W - n_sink slots go to the prefix tokens with
    the highest pooled scores (READING R1, R5).
    """
    S = K.shape[0]
    W = min(W, S)
    if B1 >= S or S - W <= 0:
        return np.arange(S, dtype=np.int64), np.zeros(max(S - W, 0))
    score = snap_scores(q_obs_group[:, -W:, :] if q_obs_group.shape[1] > W else q_obs_group, K, scale)
    pooled = max_pool_fast(score, P)
    n_sink = max(0, min(n_sink, S - W))
    n_top = max(0, B1 - W - n_sink)
    cand = pooled[n_sink:]
    top = topk_lowest_index(cand, n_top) + n_sink
    keep = np.concatenate([np.arange(n_sink), top, np.arange(S - W, S)]).astype(np.int64)
    return keep, pooled


def compact(X: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """Rows of X at the kept positions, in ascending position order (permanent eviction)."""
    return X[keep]


# ---------------------------------------------------------------------------
# KT cache: per-block Kmax / Kmin  [RKV "方法细节": HSA step 1]
# ---------------------------------------------------------------------------


def build_kt(Kc: np.ndarray, n: int, blk: int) -> Tuple[np.ndarray, np.ndarray]:
    """Elementwise max and min of each block of blk consecutive keys.

    Kc: [>= n, D].  Returns Kmax, Kmin as [D, nblk] (channel-major: [RKV] HSA
    step 1 keeps the bounds per head dimension); a partial last block uses
    only its valid rows (READING R9).
    """
    D = Kc.shape[1]
    nblk = (n + blk - 1) // blk
    kmax = np.empty((D, nblk))
    kmin = np.empty((D, nblk))
    for b in range(nblk):
        rows = Kc[b * blk: min(n, (b + 1) * blk)]
        kmax[:, b] = rows.max(axis=0)
        kmin[:, b] = rows.min(axis=0)
    return kmax, kmin


def kt_append(kmax: np.ndarray, kmin: np.ndarray, n: int, k_new: np.ndarray,
              blk: int) -> Tuple[np.ndarray, np.ndarray]:
    """Fold key number n (0-based) into the KT cache (the auxiliary store is
    updated whenever a new key is generated, [RKV] HSA step 1)."""
    b = n // blk
    D = k_new.shape[0]
    if b >= kmax.shape[1]:
        kmax = np.concatenate([kmax, np.empty((D, b + 1 - kmax.shape[1]))], axis=1)
        kmin = np.concatenate([kmin, np.empty((D, b + 1 - kmin.shape[1]))], axis=1)
    if n % blk == 0:
        kmax[:, b] = k_new
        kmin[:, b] = k_new
    else:
        kmax[:, b] = np.maximum(kmax[:, b], k_new)
        kmin[:, b] = np.minimum(kmin[:, b], k_new)
    return kmax, kmin


# ---------------------------------------------------------------------------
# Stage 2: Hybrid Sparse Attention  [RKV "方法细节": HSA steps 2-3, Algorithm 1]
# ---------------------------------------------------------------------------


def hsa_channels(q_group: np.ndarray, k1: int) -> Tuple[np.ndarray, np.ndarray]:
    """i1 = argtopk(sum_g |q_g|, k1) (ascending) and the group-summed q.

    q_group: [G, D].  Summing |q| and q over the group makes every head of the
    group take the same selection (Algorithm 1).
    """
    a = np.abs(q_group).sum(axis=0)
    qbar = q_group.sum(axis=0)
    return topk_lowest_index(a, k1), qbar


def hsa_block_scores(qbar: np.ndarray, i1: np.ndarray, kmax: np.ndarray, kmin: np.ndarray) -> np.ndarray:
    """Block scores of HSA step 2 (READING R8): for block b, the largest value
    that the linear form  sum_{c in i1} qbar_c * x_c  takes over the block's
    bounding box  Kmin[c, b] <= x_c <= Kmax[c, b].

    The box holds every key of the block, so the score bounds qbar . k (kept
    channels only) from above for each of them ([RKV] HSA step 2: the
    Kmax/Kmin bound of the attention score).  A linear form over a box is
    maximised channel by channel, each channel at whichever end of its
    interval gives the larger product; at qbar_c = 0 both ends give 0, so the
    sign convention of Algorithm 1 (READING R7) cannot change a score.
    """
    g = qbar[i1][:, None]                                      # [k1, 1]
    return np.maximum(g * kmax[i1, :], g * kmin[i1, :]).sum(axis=0)


def attention(q_group: np.ndarray, Ks: np.ndarray, Vs: np.ndarray, scale: float) -> np.ndarray:
    """Exact softmax attention of each head over the given keys/values  [RKV HSA step 3]."""
    logits = (q_group @ Ks.T) * scale              # [G, T]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    return (p @ Vs) / p.sum(axis=1, keepdims=True)


def block_tokens(i2: np.ndarray, n: int, blk: int) -> np.ndarray:
    """Valid token positions (ascending) covered by the selected blocks."""
    if i2.size == 0:
        return np.zeros(0, dtype=np.int64)
    t = (i2[:, None] * blk + np.arange(blk)[None, :]).reshape(-1)
    return t[t < n]


def hsa_decode(q_group: np.ndarray, Kc: np.ndarray, Vc: np.ndarray, n: int, kmax: np.ndarray,
               kmin: np.ndarray, blk: int, k1: int, k2: int, scale: float) -> Dict[str, np.ndarray]:
    """One HSA decode step of one GQA group over the first n compacted tokens
    ([RKV] HSA steps 2-3, Algorithm 1).

    The kept channels i1 carry the largest group mass sum_g |q_g|; each block
    is scored by its box bound (hsa_block_scores); the k2 best blocks i2 are
    kept; each head then attends exactly to the valid tokens of those blocks.
    Returns y [G, D] plus the intermediate selections and scores.
    """
    nblk = (n + blk - 1) // blk
    i1, qbar = hsa_channels(q_group, k1)
    s = hsa_block_scores(qbar, i1, kmax[:, :nblk], kmin[:, :nblk])
    i2 = topk_lowest_index(s, k2)
    tok = block_tokens(i2, n, blk)
    y = attention(q_group, Kc[tok], Vc[tok], scale)
    return {"y": y, "i1": i1, "i2": i2, "s": s, "qbar": qbar, "a": np.abs(q_group).sum(axis=0)}


def attention_over_blocks(q_group: np.ndarray, Kc: np.ndarray, Vc: np.ndarray, n: int,
                          i2: np.ndarray, blk: int, scale: float) -> np.ndarray:
    """HSA step 3 alone, over a given block set (used when a tie-exempt block differs)."""
    tok = block_tokens(np.asarray(i2, dtype=np.int64), n, blk)
    return attention(q_group, Kc[tok], Vc[tok], scale)


# ---------------------------------------------------------------------------
# RocketKV-MT  [RKV "方法细节": RocketKV-MT]  (READING R10)
# ---------------------------------------------------------------------------


def build_kt_mt(Kfull: np.ndarray, idx: np.ndarray, n: int, blk: int) -> Tuple[np.ndarray, np.ndarray]:
    """KT over the candidate sequence idx[0:n] (physical rows of the full cache)."""
    return build_kt(Kfull[np.asarray(idx[:n], dtype=np.int64)], n, blk)


def hsa_decode_mt(q_group: np.ndarray, Kfull: np.ndarray, Vfull: np.ndarray, idx: np.ndarray, n: int,
                  kmax: np.ndarray, kmin: np.ndarray, blk: int, k1: int, k2: int,
                  scale: float) -> Dict[str, np.ndarray]:
    """HSA over the full cache restricted to the candidates idx[0:n]: identical
    to hsa_decode on the rows Kfull[idx] (the full history stays in memory)."""
    rows = np.asarray(idx[:n], dtype=np.int64)
    return hsa_decode(q_group, Kfull[rows], Vfull[rows], n, kmax, kmin, blk, k1, k2, scale)


# ---------------------------------------------------------------------------
# RocketKV-MT over the physical cache  [RKV "方法细节": RocketKV-MT]  (READING R11)
# ---------------------------------------------------------------------------


def candidate_rows(keep: np.ndarray, n_prompt: int, n: int) -> np.ndarray:
    """Which of the rows [0, n) stage 2 may attend: the kept prompt rows and
    every row decoded after the prompt (RocketKV-MT limits stage 2 to the
    stage-1 survivors of the input and the tokens generated since)."""
    cand = np.zeros(n, dtype=bool)
    keep = np.asarray(keep, dtype=np.int64)
    cand[keep[keep < min(n_prompt, n)]] = True
    cand[n_prompt:] = True
    return cand


def build_kt_masked(Kfull: np.ndarray, n: int, cand: np.ndarray,
                    blk: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Kmax / Kmin of each run of blk rows of the full cache over its candidate
    rows [D, nblk], and whether the block holds any candidate.  Blocks without
    one keep zeros (they are never scored)."""
    D = Kfull.shape[1]
    nblk = (n + blk - 1) // blk
    kmax = np.zeros((D, nblk))
    kmin = np.zeros((D, nblk))
    has = np.zeros(nblk, dtype=bool)
    for b in range(nblk):
        rows = [r for r in range(b * blk, min(n, (b + 1) * blk)) if cand[r]]
        if rows:
            has[b] = True
            kmax[:, b] = Kfull[rows].max(axis=0)
            kmin[:, b] = Kfull[rows].min(axis=0)
    return kmax, kmin, has


def kt_append_masked(kmax: np.ndarray, kmin: np.ndarray, has: np.ndarray, n: int, k_new: np.ndarray,
                     blk: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Fold decoded row n (always a candidate) into block n // blk: the first
    candidate of a block sets its bounds, later ones widen them."""
    b = n // blk
    D = k_new.shape[0]
    if b >= kmax.shape[1]:
        grow = b + 1 - kmax.shape[1]
        kmax = np.concatenate([kmax, np.zeros((D, grow))], axis=1)
        kmin = np.concatenate([kmin, np.zeros((D, grow))], axis=1)
        has = np.concatenate([has, np.zeros(grow, dtype=bool)])
    if not has[b]:
        kmax[:, b] = k_new
        kmin[:, b] = k_new
        has[b] = True
    else:
        kmax[:, b] = np.maximum(kmax[:, b], k_new)
        kmin[:, b] = np.minimum(kmin[:, b], k_new)
    return kmax, kmin, has


def hsa_decode_mt_masked(q_group: np.ndarray, Kfull: np.ndarray, Vfull: np.ndarray, n: int, cand: np.ndarray,
                         kmax: np.ndarray, kmin: np.ndarray, has: np.ndarray, blk: int, k1: int, k2: int,
                         scale: float) -> Dict[str, np.ndarray]:
    """One HSA step over the blocks of the full cache (READING R11): Algorithm
    1's scores on the candidate-only bounds, blocks without a candidate at
    -inf, the newest row's block at +inf, top-k2 blocks, then attention over
    the candidate rows of those blocks."""
    nblk = (n + blk - 1) // blk
    i1, qbar = hsa_channels(q_group, k1)
    s = hsa_block_scores(qbar, i1, kmax[:, :nblk], kmin[:, :nblk])
    s = np.where(has[:nblk], s, -np.inf)
    tail = (n - 1) // blk
    if has[tail]:
        s[tail] = np.inf
    i2 = topk_lowest_index(s, k2)
    tok = block_tokens(i2, n, blk)
    tok = tok[cand[tok]]
    y = attention(q_group, Kfull[tok], Vfull[tok], scale)
    return {"y": y, "i1": i1, "i2": i2, "s": s, "tok": tok}


# ---------------------------------------------------------------------------
# FP8 (e4m3) storage of the compacted cache  (READING R12)
# ---------------------------------------------------------------------------


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each e4m3 code: exponent field 0 is subnormal (m/8 * 2^-6),
    otherwise (1 + m/8) * 2^(e - 7); S.1111.111 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    val = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, val)


_E4M3_POS = e4m3_decode(np.arange(127, dtype=np.uint8))     # codes 0..126: 0 .. 448, ascending


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code of each value (ties to the even code, i.e. even
    mantissa), magnitudes above 448 saturated to 448, NaN -> 0x7f; the sign
    bit follows the value's sign (a negative value that rounds to zero gives
    0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo = np.abs(a - _E4M3_POS[lo])
    dhi = np.abs(_E4M3_POS[hi] - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


def fp8_quantize(X: np.ndarray, scale: float) -> np.ndarray:
    """Codes of X / scale, the quotient taken in fp32 (READING R12)."""
    q = np.asarray(X, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q.astype(np.float64))


def build_kt_fp8(Kcodes: np.ndarray, n: int, blk: int) -> Tuple[np.ndarray, np.ndarray]:
    """Kmax / Kmin of the key code values of each block, [D, nblk]."""
    return build_kt(e4m3_decode(Kcodes), n, blk)


def hsa_decode_fp8(q_group: np.ndarray, Kcodes: np.ndarray, Vcodes: np.ndarray, n: int, kmax: np.ndarray,
                   kmin: np.ndarray, k_scale: float, v_scale: float, blk: int, k1: int, k2: int,
                   scale: float) -> Dict[str, np.ndarray]:
    """HSA step over an e4m3 cache: Algorithm 1's scores on the code values
    (kmax / kmin from build_kt_fp8), then attention over the selected rows'
    values code * scale."""
    nblk = (n + blk - 1) // blk
    i1, qbar = hsa_channels(q_group, k1)
    s = hsa_block_scores(qbar, i1, kmax[:, :nblk], kmin[:, :nblk])
    i2 = topk_lowest_index(s, k2)
    tok = block_tokens(i2, n, blk)
    Kd = e4m3_decode(Kcodes[tok]) * float(np.float32(k_scale))
    Vd = e4m3_decode(Vcodes[tok]) * float(np.float32(v_scale))
    y = attention(q_group, Kd, Vd, scale)
    return {"y": y, "i1": i1, "i2": i2, "s": s}


# ---------------------------------------------------------------------------
# Whole single-group pipelines (used for small end-to-end checks)
# ---------------------------------------------------------------------------


def pipeline_group(q_obs_group, K, V, q_steps, k_new, v_new, B1, W, P, blk, k1, k2, scale,
                   n_sink: int = 0):
    """Stage 1, KT build, then len(q_steps) decode steps (append, then HSA).

    q_steps [T, G, D]; k_new, v_new [T, D].  Returns keep and per-step results.
    """
    keep, pooled = snap_keep(q_obs_group, K, B1, W, P, scale, n_sink)
    Kc = list(compact(K, keep))
    Vc = list(compact(V, keep))
    n = len(Kc)
    kmax, kmin = build_kt(np.asarray(Kc), n, blk)
    out = []
    for t in range(q_steps.shape[0]):
        kmax, kmin = kt_append(kmax, kmin, n, k_new[t], blk)
        Kc.append(k_new[t])
        Vc.append(v_new[t])
        n += 1
        out.append(hsa_decode(q_steps[t], np.asarray(Kc), np.asarray(Vc), n, kmax, kmin, blk, k1, k2, scale))
    return keep, pooled, out
