"""GPU parity of each entry point against the CPU oracle on small and ragged
shapes (several tiles plus a partial tail), through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import ATOL_OUT, check_topk, max_abs, t2bits, t2f64
from two_stage_kv_gb300 import rkv
from two_stage_kv_gb300.synth import bf16_bits_to_f32, bf16_bits_to_f64, f32_to_bf16_bits, small_random

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)


def _rand(seed, shape, scale=1.0):
    b = small_random(seed, shape, scale)
    return b, _bf16(b)


# ----------------------------------------------------------------- KT cache --


@pytest.mark.parametrize("n,blk,cap_extra", [(300, 16, 5), (64, 16, 0), (1, 16, 3), (1000, 32, 7), (77, 8, 1),
                                              (129, 128, 0)])
def test_build_kt_bit_exact(n, blk, cap_extra):
    B, Hq, Hkv, D = 2, 8, 2, 128
    cap = n + cap_extra
    kb, k = _rand(11 + n, (B, Hkv, cap, D))
    nblk = -(-n // blk)
    kt = torch.full((B, Hkv, 2, D, nblk + 3), float("nan"), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_build_kt((B, Hq, Hkv, D), k, cap, n, None, 0, blk, kt, nblk + 3)
    torch.cuda.synchronize()
    got = t2f64(kt)
    kf = bf16_bits_to_f64(kb)
    for b in range(B):
        for h in range(Hkv):
            kmax, kmin = oracle.build_kt(kf[b, h], n, blk)
            assert np.array_equal(got[b, h, 0, :, :nblk], kmax)
            assert np.array_equal(got[b, h, 1, :, :nblk], kmin)
    # blocks past nblk are untouched
    assert torch.isnan(kt[..., nblk:].float()).all()


@pytest.mark.parametrize("B1,blk,cap", [(300, 16, 1000), (1, 16, 50), (1000, 32, 3000), (77, 8, 200),
                                         (259, 128, 600), (2000, 16, 2100)])
def test_compact_kt_bit_exact(B1, blk, cap):
    """Compaction with the KT cache built on the way equals the oracle's gather of
    the kept rows and its Kmax / Kmin of the compacted keys, bit for bit, and
    writes nothing past B1 rows or ceil(B1 / blk) KT columns."""
    B, Hq, Hkv, D = 2, 8, 2, 128
    kb, k = _rand(21 + B1, (B, Hkv, cap, D))
    vb, v = _rand(22 + B1, (B, Hkv, cap, D))
    rng = np.random.default_rng(B1)
    keep = np.stack([np.stack([np.sort(rng.choice(cap, B1, replace=False)) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32)
    keep_t = torch.from_numpy(keep).to(DEV)
    out_cap = B1 + 5
    nblk = -(-B1 // blk)
    ncap = -(-(nblk + 1) // 8) * 8
    ko = torch.full((B, Hkv, out_cap, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    vo = torch.full_like(ko, float("nan"))
    kt = torch.full((B, Hkv, 2, D, ncap), float("nan"), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_compact_kt((B, Hq, Hkv, D), k, v, cap, keep_t, B1, B1, ko, vo, out_cap, blk, kt, ncap)
    torch.cuda.synchronize()
    kbits, vbits, got = t2bits(ko), t2bits(vo), t2f64(kt)
    kf = bf16_bits_to_f64(kb)
    for b in range(B):
        for h in range(Hkv):
            assert np.array_equal(kbits[b, h, :B1], oracle.compact(kb[b, h], keep[b, h]))
            assert np.array_equal(vbits[b, h, :B1], oracle.compact(vb[b, h], keep[b, h]))
            kmax, kmin = oracle.build_kt(oracle.compact(kf[b, h], keep[b, h]), B1, blk)
            assert np.array_equal(got[b, h, 0, :, :nblk], kmax) and np.array_equal(got[b, h, 1, :, :nblk], kmin)
    assert torch.isnan(ko[:, :, B1:].float()).all() and torch.isnan(vo[:, :, B1:].float()).all()
    assert torch.isnan(kt[..., nblk:].float()).all()


def test_build_kt_mt_rows():
    B, Hq, Hkv, D, full, n, blk = 1, 4, 2, 128, 500, 173, 16
    kb, k = _rand(3, (B, Hkv, full, D))
    rng = np.random.default_rng(5)
    idx = np.stack([np.stack([np.sort(rng.choice(full, n, replace=False)) for _ in range(Hkv)])])
    idx_t = torch.from_numpy(idx.astype(np.int32)).to(DEV)
    nblk = -(-n // blk)
    kt = torch.empty((B, Hkv, 2, D, nblk), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_build_kt((B, Hq, Hkv, D), k, full, n, idx_t, n, blk, kt, nblk)
    got = t2f64(kt)
    kf = bf16_bits_to_f64(kb)
    for h in range(Hkv):
        kmax, kmin = oracle.build_kt_mt(kf[0, h], idx[0, h], n, blk)
        assert np.array_equal(got[0, h, 0], kmax) and np.array_equal(got[0, h, 1], kmin)


def test_append_matches_rebuild():
    B, Hq, Hkv, D, blk = 2, 8, 2, 128, 16
    n0, steps = 45, 40
    cap = n0 + steps
    kb, k = _rand(21, (B, Hkv, cap, D))
    vb, v = _rand(22, (B, Hkv, cap, D))
    nb, knew = _rand(23, (steps, B, Hkv, D))
    mb, vnew = _rand(24, (steps, B, Hkv, D))
    nblk_cap = -(-cap // blk)
    kt = torch.empty((B, Hkv, 2, D, nblk_cap), dtype=torch.bfloat16, device=DEV)
    dims = (B, Hq, Hkv, D)
    rkv.rkv_build_kt(dims, k, cap, n0, None, 0, blk, kt, nblk_cap)
    for s in range(steps):
        rkv.rkv_append_kv(dims, knew[s], vnew[s], k, v, cap, n0 + s, n0 + s, None, 0, kt, nblk_cap, blk)
    torch.cuda.synchronize()
    kexp = kb.copy()
    vexp = vb.copy()
    kexp[:, :, n0:] = nb.transpose(1, 2, 0, 3)
    vexp[:, :, n0:] = mb.transpose(1, 2, 0, 3)
    assert np.array_equal(t2bits(k), kexp) and np.array_equal(t2bits(v), vexp)
    got = t2f64(kt)
    for b in range(B):
        for h in range(Hkv):
            kmax, kmin = oracle.build_kt(bf16_bits_to_f64(kexp[b, h]), cap, blk)
            assert np.array_equal(got[b, h, 0], kmax) and np.array_equal(got[b, h, 1], kmin)


# --------------------------------------------------------------- HSA decode --


def _hsa_case(seed, B, Hq, Hkv, n, blk, k1, k2, cap_extra=3, q_scale=1.0, mt=False, full_rows=None,
              k_scale=1.0, kmod=None, qmod=None):
    D = 128
    G = Hq // Hkv
    dims = (B, Hq, Hkv, D)
    scale = 1 / math.sqrt(D)
    rows = full_rows if mt else n + cap_extra
    kb = small_random(seed, (B, Hkv, rows, D), k_scale)
    if kmod is not None:
        kb = kmod(kb)
    k = _bf16(kb)
    vb, v = _rand(seed + 1, (B, Hkv, rows, D))
    qb = small_random(seed + 2, (B, Hq, D), q_scale)
    if qmod is not None:
        qb = qmod(qb)
    q = _bf16(qb)
    kf, vf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), bf16_bits_to_f64(qb)
    nblk = -(-n // blk)
    ncap = -(-nblk // 8) * 8
    kt = torch.empty((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    sb = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((B, Hkv, k1), -7, dtype=torch.int32, device=DEV)
    if mt:
        rng = np.random.default_rng(seed)
        idx = np.stack([np.stack([np.sort(rng.choice(rows, n, replace=False)) for _ in range(Hkv)])
                        for _ in range(B)]).astype(np.int32)
        idx_t = torch.from_numpy(idx).to(DEV)
        rkv.rkv_build_kt(dims, k, rows, n, idx_t, n, blk, kt, ncap)
        rkv.rkv_hsa_decode_mt(dims, q, k, v, rows, idx_t, n, n, kt, ncap, blk, k1, k2, scale, out, sb, sc)
    else:
        rkv.rkv_build_kt(dims, k, rows, n, None, 0, blk, kt, ncap)
        rkv.rkv_hsa_decode(dims, q, k, v, rows, n, kt, ncap, blk, k1, k2, scale, out, sb, sc)
    torch.cuda.synchronize()
    out_h, sb_h, sc_h = out.cpu().numpy(), sb.cpu().numpy(), sc.cpu().numpy()
    worst, exempt = 0.0, 0
    for b in range(B):
        for h in range(Hkv):
            qg = qf[b, h * G:(h + 1) * G]
            if mt:
                rws = idx[b, h]
                Kc, Vc = kf[b, h][rws], vf[b, h][rws]
            else:
                Kc, Vc = kf[b, h], vf[b, h]
            kmax, kmin = oracle.build_kt(Kc, n, blk)
            res = oracle.hsa_decode(qg, Kc, Vc, n, kmax, kmin, blk, k1, k2, scale)
            assert sc_h[b, h].tolist() == res["i1"].tolist(), "channel set differs"
            k2e = min(k2, nblk)
            exempt += check_topk(sb_h[b, h, :k2e], res["s"], k2, "blocks")
            assert np.all(sb_h[b, h, k2e:] == -1)
            y = res["y"] if np.array_equal(sb_h[b, h, :k2e], res["i2"]) else \
                oracle.attention_over_blocks(qg, Kc, Vc, n, sb_h[b, h, :k2e], blk, scale)
            worst = max(worst, max_abs(out_h[b, h * G:(h + 1) * G], y))
    assert worst <= ATOL_OUT, worst
    return worst, exempt


@pytest.mark.parametrize("B,Hq,Hkv,n,blk,k1,k2", [
    (2, 32, 8, 300, 16, 32, 5),       # ragged tail, G = 4
    (1, 8, 8, 517, 16, 16, 9),        # G = 1
    (1, 64, 8, 1000, 32, 64, 11),     # G = 8, block 32
    (1, 32, 2, 333, 8, 128, 40),      # G = 16, block 8, all channels
    (2, 32, 8, 130, 16, 32, 64),      # k2 >= nblk: full attention
    (1, 32, 8, 1, 16, 32, 4),         # a single token
    (1, 32, 8, 4096, 128, 20, 3),     # block 128
    (1, 32, 8, 20000, 16, 32, 300),   # many blocks, several rounds per CTA
    (1, 32, 8, 700, 1, 32, 40),       # token-level blocks (SparQ-like), gathered rows
    (2, 32, 8, 500, 4, 32, 10),       # block 4, gathered rows
    (1, 64, 8, 333, 12, 64, 7),       # block 12 (not a multiple of 8), G = 8
    (1, 32, 8, 300, 1, 128, 20),      # k1 = D and block 1: exact top-k of qbar . k (Exact-TopK)
    # several staging rounds per CTA (per-warp online softmax, merged once)
    (1, 8, 8, 6000, 16, 16, 300),     # G = 1
    (1, 24, 8, 6000, 16, 32, 300),    # G = 3 (odd group: scalar partial stores)
    (1, 64, 8, 6000, 16, 64, 300),    # G = 8
    (1, 32, 8, 8000, 24, 32, 250),    # block 24: 120-row rounds, zero-filled tail rows
    (2, 40, 8, 8000, 40, 32, 150),    # block 40, G = 5
])
def test_hsa_decode_parity(B, Hq, Hkv, n, blk, k1, k2):
    _hsa_case(100 + n, B, Hq, Hkv, n, blk, k1, k2)


def test_hsa_decode_peaked_attention():
    # large queries make the softmax nearly one-hot: checks the P hi/lo split
    _hsa_case(7, 1, 32, 8, 700, 16, 32, 8, q_scale=6.0)


def test_hsa_decode_all_ties():
    # q = 0: every channel sum and every block score ties, so both selections fall
    # back to the radix path and take the lowest indices; attention is uniform
    _hsa_case(11, 1, 32, 8, 900, 16, 32, 12, qmod=np.zeros_like)


def test_hsa_decode_crowded_boundary_bucket():
    # block 0 holds huge keys and every other block tiny ones: all but one score
    # share a histogram bucket (more members than the pairwise ranking takes),
    # which sends the block selection to the radix path
    def kmod(kb):
        kb = kb.copy()
        kb[:, :, :16, :] = 0x42C8            # bf16 100.0
        return kb
    _hsa_case(12, 1, 32, 8, 700 * 16, 16, 32, 50, k_scale=1e-3, kmod=kmod)


@pytest.mark.parametrize("Hq,k1", [(32, 32), (32, 20), (64, 64)])
def test_hsa_decode_channel_partial_ties(Hq, k1):
    """Queries drawn from {-2, ..., 2}: the group sums of |q| fall in a few values,
    so large groups of channels tie across the k1-th place (the lower channel
    index must win), and some group sums of q are exactly zero (the sign rule
    picks Kmax).  The channel set must equal the oracle's exactly."""
    def qmod(qb):
        r = np.random.default_rng(5 + Hq + k1)
        return f32_to_bf16_bits(r.integers(-2, 3, qb.shape).astype(np.float32))
    _hsa_case(13 + k1, 2, Hq, 8, 900, 16, k1, 12, qmod=qmod)


def test_hsa_decode_split_boundary_bucket():
    """Blocks 10-19 hold the same large keys, so their scores tie exactly and are
    the ten largest, alone in the top histogram bucket; k2 = 5 takes half of that
    bucket, which sends the selection through the pairwise ranking of its
    members.  Ties must go to the lower block index: no tie-band exemption."""
    blk = 16

    def kmod(kb):
        kb = kb.copy()
        big = f32_to_bf16_bits(bf16_bits_to_f32(kb[:, :, 3 * blk:4 * blk, :]) * np.float32(4))
        for j in range(10, 20):
            kb[:, :, j * blk:(j + 1) * blk, :] = big
        return kb
    _, exempt = _hsa_case(14, 1, 32, 8, 700, blk, 32, 5, kmod=kmod)
    assert exempt == 0


@pytest.mark.parametrize("append", [False, True])
def test_hsa_decode_ragged_rows(append):
    """Rows with different candidate counts in one launch: every row matches the
    oracle on its own n (and its own appended token and KT block)."""
    B, Hq, Hkv, D, blk, k1, k2 = 3, 32, 8, 128, 16, 32, 8
    G = Hq // Hkv
    n_rows = [300, 1000, 57]
    n_max, cap = max(n_rows), 1100
    dims = (B, Hq, Hkv, D)
    kb, k = _rand(81, (B, Hkv, cap, D))
    vb, v = _rand(82, (B, Hkv, cap, D))
    qb, q = _rand(83, (B, Hq, D))
    nb_, knew = _rand(84, (B, Hkv, D))
    vnb, vnew = _rand(85, (B, Hkv, D))
    ncap = -(-(-(-(n_max + 1) // blk)) // 8) * 8
    kt = torch.empty((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    for b in range(B):             # each row's KT covers its own candidates
        rkv.rkv_build_kt((1, Hq, Hkv, D), k[b:b + 1], cap, n_rows[b], None, 0, blk, kt[b:b + 1], ncap)
    n_dev = torch.tensor(n_rows, dtype=torch.int32, device=DEV)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    sb = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(D)
    rkv.rkv_hsa_decode_ragged(dims, q, k, v, cap, n_dev, n_max, kt, ncap, blk, k1, k2, scale, out, sb, None,
                              knew if append else None, vnew if append else None)
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags() == 0
    kf, vf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), bf16_bits_to_f64(qb)
    out_h, sb_h, kt_h = out.cpu().numpy(), sb.cpu().numpy(), t2f64(kt)
    worst = 0.0
    for b in range(B):
        n = n_rows[b] + (1 if append else 0)
        for h in range(Hkv):
            Kc, Vc = kf[b, h, :n].copy(), vf[b, h, :n].copy()
            if append:
                Kc[-1] = bf16_bits_to_f64(nb_)[b, h]
                Vc[-1] = bf16_bits_to_f64(vnb)[b, h]
                assert np.array_equal(t2bits(k[b, h, n - 1]), nb_[b, h])   # the row was persisted
            kmax, kmin = oracle.build_kt(Kc, n, blk)
            nblk = kmax.shape[1]
            assert np.array_equal(kt_h[b, h, 0, :, :nblk], kmax) and np.array_equal(kt_h[b, h, 1, :, :nblk], kmin)
            qg = qf[b, h * G:(h + 1) * G]
            res = oracle.hsa_decode(qg, Kc, Vc, n, kmax, kmin, blk, k1, k2, scale)
            k2e = min(k2, nblk)
            check_topk(sb_h[b, h, :k2e], res["s"], k2, f"row {b} blocks")
            assert np.all(sb_h[b, h, k2e:] == -1)
            y = oracle.attention_over_blocks(qg, Kc, Vc, n, sb_h[b, h, :k2e], blk, scale)
            worst = max(worst, max_abs(out_h[b, h * G:(h + 1) * G], y))
    assert worst <= ATOL_OUT, worst


def test_hsa_decode_ragged_length_out_of_range_flagged():
    B, Hq, Hkv, D, blk = 2, 32, 8, 128, 16
    cap, n_max = 400, 300
    dims = (B, Hq, Hkv, D)
    _, k = _rand(91, (B, Hkv, cap, D))
    _, v = _rand(92, (B, Hkv, cap, D))
    _, q = _rand(93, (B, Hq, D))
    ncap = 24
    kt = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_build_kt(dims, k, cap, n_max, None, 0, blk, kt, ncap)
    n_dev = torch.tensor([200, 5000], dtype=torch.int32, device=DEV)     # 5000 > n_max: clamped
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    rkv.rkv_hsa_decode_ragged(dims, q, k, v, cap, n_dev, n_max, kt, ncap, blk, 32, 4, 0.1, out)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_read_device_flags()
    assert "0x2" in str(e.value)
    assert torch.isfinite(out).all()


def _page_table(rng, B, nblk_row, extra):
    """A random block table [B, nblk_row] over num_pages = B * nblk_row + extra pages (all distinct)."""
    num_pages = B * nblk_row + extra
    return rng.permutation(num_pages)[:B * nblk_row].reshape(B, nblk_row).astype(np.int32), num_pages


@pytest.mark.parametrize("blk", [16, 4])
def test_compact_kt_paged_matches_dense(blk):
    B, Hq, Hkv, D, cap, B1 = 2, 8, 2, 128, 900, 333
    dims = (B, Hq, Hkv, D)
    _, k = _rand(101, (B, Hkv, cap, D))
    _, v = _rand(102, (B, Hkv, cap, D))
    rng = np.random.default_rng(7)
    keep = np.stack([np.stack([np.sort(rng.choice(cap, B1, replace=False)) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32)
    keep_t = torch.from_numpy(keep).to(DEV)
    nblk = -(-B1 // blk)
    ncap = -(-nblk // 8) * 8
    bt, num_pages = _page_table(rng, B, nblk, 5)
    bt_t = torch.from_numpy(bt).to(DEV)
    ko = torch.zeros((B, Hkv, nblk * blk, D), dtype=torch.bfloat16, device=DEV)
    vo = torch.zeros_like(ko)
    ktd = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    kp = torch.zeros((num_pages, Hkv, blk, D), dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    ktp = torch.zeros_like(ktd)
    rkv.rkv_compact_kt(dims, k, v, cap, keep_t, B1, B1, ko, vo, nblk * blk, blk, ktd, ncap)
    rkv.rkv_compact_kt_paged(dims, k, v, cap, keep_t, B1, B1, kp, vp, num_pages, bt_t, nblk, blk, ktp, ncap)
    torch.cuda.synchronize()
    assert torch.equal(ktd, ktp)
    for b in range(B):
        for j in range(nblk):
            r = min(blk, B1 - j * blk)
            assert torch.equal(kp[bt[b, j], :, :r], ko[b, :, j * blk:j * blk + r])
            assert torch.equal(vp[bt[b, j], :, :r], vo[b, :, j * blk:j * blk + r])


@pytest.mark.parametrize("blk,append", [(16, False), (16, True), (4, True)])
def test_hsa_decode_paged_equals_dense(blk, append):
    """Paged pools addressed through a block table give bit-identical results to the
    dense caches (same rows, same order), with per-row lengths and the fused append
    landing in slot n % blk of page block_table[b, n / blk]."""
    B, Hq, Hkv, D, k1, k2 = 3, 32, 8, 128, 32, 8
    n_rows = [300, 611, 57]
    n_max = max(n_rows)
    nblk_row = -(-(n_max + 1) // blk)
    cap = nblk_row * blk
    dims = (B, Hq, Hkv, D)
    _, k = _rand(111, (B, Hkv, cap, D))
    _, v = _rand(112, (B, Hkv, cap, D))
    _, q = _rand(113, (B, Hq, D))
    _, knew = _rand(114, (B, Hkv, D))
    _, vnew = _rand(115, (B, Hkv, D))
    rng = np.random.default_rng(11)
    bt, num_pages = _page_table(rng, B, nblk_row, 3)
    bt_t = torch.from_numpy(bt).to(DEV)
    kp = torch.zeros((num_pages, Hkv, blk, D), dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    for b in range(B):
        for j in range(nblk_row):
            kp[bt[b, j]] = k[b, :, j * blk:(j + 1) * blk]
            vp[bt[b, j]] = v[b, :, j * blk:(j + 1) * blk]
    ncap = -(-nblk_row // 8) * 8
    ktd = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    for b in range(B):
        rkv.rkv_build_kt((1, Hq, Hkv, D), k[b:b + 1], cap, n_rows[b], None, 0, blk, ktd[b:b + 1], ncap)
    ktp = ktd.clone()
    n_dev = torch.tensor(n_rows, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(D)
    od = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    op = torch.empty_like(od)
    sd = torch.empty((B, Hkv, k2), dtype=torch.int32, device=DEV)
    sp = torch.empty_like(sd)
    kn_, vn_ = (knew, vnew) if append else (None, None)
    rkv.rkv_hsa_decode_ragged(dims, q, k, v, cap, n_dev, n_max, ktd, ncap, blk, k1, k2, scale, od, sd, None, kn_, vn_)
    rkv.rkv_hsa_decode_paged(dims, q, kp, vp, num_pages, bt_t, nblk_row, n_dev, n_max, ktp, ncap, blk, k1, k2, scale,
                             op, sp, None, kn_, vn_)
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags() == 0
    assert torch.equal(sd, sp) and torch.equal(od, op) and torch.equal(ktd, ktp)
    if append:
        for b in range(B):
            n = n_rows[b]
            assert torch.equal(kp[bt[b, n // blk], :, n % blk], k[b, :, n])
            assert torch.equal(vp[bt[b, n // blk], :, n % blk], v[b, :, n])


def test_hsa_decode_bounded_wait_runs_out():
    """The timeout path of the bounded waits, without a fault: the block-score
    barrier of every CTA is told to expect 16 bytes that no copy delivers and
    each wait is shortened to 20 us.  The wait runs out, the kernel goes on
    with the scores it received (all of them arrived), finishes, and reports
    bit 0 of the device error word; the results equal a normal run's, and the
    next normal launch on the same context is clean."""
    B, Hq, Hkv, D, n, blk, k1, k2 = 2, 32, 8, 128, 3000, 16, 32, 8
    dims = (B, Hq, Hkv, D)
    _, k = _rand(141, (B, Hkv, n, D))
    _, v = _rand(142, (B, Hkv, n, D))
    _, q = _rand(143, (B, Hq, D))
    ncap = -(-(-(-n // blk)) // 8) * 8
    kt = torch.empty((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_build_kt(dims, k, n, n, None, 0, blk, kt, ncap)
    scale = 1 / math.sqrt(D)

    def run():
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
        sb = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=DEV)
        rkv.rkv_hsa_decode(dims, q, k, v, n, n, kt, ncap, blk, k1, k2, scale, out, sb, None)
        torch.cuda.synchronize()
        return out, sb

    assert rkv.rkv_read_device_flags() == 0
    ref_out, ref_sb = run()
    assert rkv.rkv_read_device_flags() == 0
    rkv.rkv_debug_set_wait(20_000, 16)
    try:
        out, sb = run()
        with pytest.raises(rkv.RkvError) as e:
            rkv.rkv_read_device_flags()
        assert e.value.status == 5 and "0x1" in str(e.value)
    finally:
        rkv.rkv_debug_set_wait(0, 0)
    assert torch.isfinite(out).all()
    assert torch.equal(sb, ref_sb) and torch.equal(out, ref_out)
    out2, sb2 = run()
    assert rkv.rkv_read_device_flags() == 0
    assert torch.equal(out2, ref_out) and torch.equal(sb2, ref_sb)


def _kt_bits(Kc, n, blk, ncap):
    """The oracle's Kmax / Kmin of Kc[:n] as bf16 bits [2, D, ncap] (exact: max and
    min of bf16 values are bf16 values); columns past the last block are zero."""
    kmax, kmin = oracle.build_kt(Kc, n, blk)
    out = np.zeros((2, Kc.shape[1], ncap), dtype=np.uint16)
    out[0, :, :kmax.shape[1]] = f32_to_bf16_bits(kmax.astype(np.float32))
    out[1, :, :kmin.shape[1]] = f32_to_bf16_bits(kmin.astype(np.float32))
    return out


@pytest.mark.parametrize("blk,append,n_rows", [
    (16, False, [300, 611, 57, 4000]),
    (16, True, [300, 611, 57, 4000]),
    (4, False, [300, 611, 57, 1500]),
    (4, True, [301, 612, 58, 1500]),
    (32, True, [2047, 31, 5000, 64]),
])
def test_hsa_decode_paged_oracle(blk, append, n_rows):
    """Paged pools against the oracle directly: each batch row's logical sequence
    (rows 0 .. n_b-1, plus the appended token) is scattered into pages of blk rows
    through a shuffled block table; the KT cache comes from the oracle; every
    unused page slot holds large random rows, so a wrong page or slot would
    change the result.  i1 exact, i2 within the tie band, outputs within 2e-3,
    the appended row in slot n % blk of its page and its KT column bit-exact."""
    B, Hq, Hkv, D, k1, k2 = len(n_rows), 32, 8, 128, 32, 12
    G = Hq // Hkv
    n_max = max(n_rows)
    nblk_row = -(-(n_max + 1) // blk)
    dims = (B, Hq, Hkv, D)
    kb = small_random(121 + blk, (B, Hkv, nblk_row * blk, D))
    vb = small_random(122 + blk, (B, Hkv, nblk_row * blk, D))
    qb, q = _rand(123 + blk, (B, Hq, D))
    knb, knew = _rand(124 + blk, (B, Hkv, D))
    vnb, vnew = _rand(125 + blk, (B, Hkv, D))
    rng = np.random.default_rng(13 + blk)
    bt, num_pages = _page_table(rng, B, nblk_row, 7)
    kpb = small_random(126 + blk, (num_pages, Hkv, blk, D), 50.0)     # garbage everywhere first
    vpb = small_random(127 + blk, (num_pages, Hkv, blk, D), 50.0)
    for b in range(B):
        for j in range(-(-n_rows[b] // blk)):
            r = min(blk, n_rows[b] - j * blk)
            kpb[bt[b, j], :, :r] = kb[b, :, j * blk:j * blk + r]
            vpb[bt[b, j], :, :r] = vb[b, :, j * blk:j * blk + r]
    kp, vp = _bf16(kpb), _bf16(vpb)
    ncap = -(-nblk_row // 8) * 8
    kf, vf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), bf16_bits_to_f64(qb)
    ktb = np.stack([np.stack([_kt_bits(kf[b, h], n_rows[b], blk, ncap) for h in range(Hkv)]) for b in range(B)])
    kt = _bf16(ktb)
    n_dev = torch.tensor(n_rows, dtype=torch.int32, device=DEV)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    sb = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((B, Hkv, k1), -7, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(D)
    rkv.rkv_hsa_decode_paged(dims, q, kp, vp, num_pages, torch.from_numpy(bt).to(DEV), nblk_row, n_dev, n_max, kt,
                             ncap, blk, k1, k2, scale, out, sb, sc, knew if append else None,
                             vnew if append else None)
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags() == 0
    out_h, sb_h, sc_h, kt_h = out.cpu().numpy(), sb.cpu().numpy(), sc.cpu().numpy(), t2f64(kt)
    kp_h, vp_h = t2bits(kp), t2bits(vp)
    worst = 0.0
    for b in range(B):
        n = n_rows[b] + (1 if append else 0)
        for h in range(Hkv):
            Kc, Vc = kf[b, h, :n].copy(), vf[b, h, :n].copy()
            if append:
                Kc[-1] = bf16_bits_to_f64(knb)[b, h]
                Vc[-1] = bf16_bits_to_f64(vnb)[b, h]
                pg, sl = bt[b, n_rows[b] // blk], n_rows[b] % blk
                assert np.array_equal(kp_h[pg, h, sl], knb[b, h]) and np.array_equal(vp_h[pg, h, sl], vnb[b, h])
            kmax, kmin = oracle.build_kt(Kc, n, blk)
            nblk = kmax.shape[1]
            assert np.array_equal(kt_h[b, h, 0, :, :nblk], kmax) and np.array_equal(kt_h[b, h, 1, :, :nblk], kmin)
            qg = qf[b, h * G:(h + 1) * G]
            res = oracle.hsa_decode(qg, Kc, Vc, n, kmax, kmin, blk, k1, k2, scale)
            assert sc_h[b, h].tolist() == res["i1"].tolist(), f"row {b} head {h}: channel set differs"
            k2e = min(k2, nblk)
            check_topk(sb_h[b, h, :k2e], res["s"], k2, f"row {b} head {h} blocks")
            assert np.all(sb_h[b, h, k2e:] == -1)
            y = res["y"] if np.array_equal(sb_h[b, h, :k2e], res["i2"]) else \
                oracle.attention_over_blocks(qg, Kc, Vc, n, sb_h[b, h, :k2e], blk, scale)
            worst = max(worst, max_abs(out_h[b, h * G:(h + 1) * G], y))
    assert worst <= ATOL_OUT, worst


@pytest.mark.parametrize("blk,B1", [(16, 333), (4, 333), (32, 2500)])
def test_compact_kt_paged_oracle(blk, B1):
    """Paged compaction against the oracle: page block_table[b, i / blk] slot i % blk
    holds k[b, h, keep[b, h, i]] (bit for bit), the KT cache equals the oracle's
    Kmax / Kmin of the compacted keys, and pages outside the table keep their
    canary contents."""
    B, Hq, Hkv, D, cap = 2, 8, 2, 128, 3000
    dims = (B, Hq, Hkv, D)
    kb, k = _rand(131 + blk, (B, Hkv, cap, D))
    vb, v = _rand(132 + blk, (B, Hkv, cap, D))
    rng = np.random.default_rng(17 + blk)
    keep = np.stack([np.stack([np.sort(rng.choice(cap, B1, replace=False)) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32)
    nblk = -(-B1 // blk)
    ncap = -(-(nblk + 1) // 8) * 8
    bt, num_pages = _page_table(rng, B, nblk, 5)
    kp = torch.full((num_pages, Hkv, blk, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    vp = torch.full_like(kp, float("nan"))
    kt = torch.full((B, Hkv, 2, D, ncap), float("nan"), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_compact_kt_paged(dims, k, v, cap, torch.from_numpy(keep).to(DEV), B1, B1, kp, vp, num_pages,
                             torch.from_numpy(bt).to(DEV), nblk, blk, kt, ncap)
    torch.cuda.synchronize()
    kp_h, vp_h, kt_h = t2bits(kp), t2bits(vp), t2f64(kt)
    kf = bf16_bits_to_f64(kb)
    for b in range(B):
        for h in range(Hkv):
            kc, vc = oracle.compact(kb[b, h], keep[b, h]), oracle.compact(vb[b, h], keep[b, h])
            for i in range(B1):
                assert np.array_equal(kp_h[bt[b, i // blk], h, i % blk], kc[i])
                assert np.array_equal(vp_h[bt[b, i // blk], h, i % blk], vc[i])
            kmax, kmin = oracle.build_kt(oracle.compact(kf[b, h], keep[b, h]), B1, blk)
            assert np.array_equal(kt_h[b, h, 0, :, :nblk], kmax) and np.array_equal(kt_h[b, h, 1, :, :nblk], kmin)
    unused = np.setdiff1d(np.arange(num_pages), bt.reshape(-1))
    assert torch.isnan(kp[torch.from_numpy(unused).to(DEV)].float()).all()


def test_hsa_decode_exact_topk_pin():
    """k1 = D and block 1: the block score is qbar . k_j exactly, so the chosen tokens
    are the plain top-k2 of qbar . k (lowest index on ties) and the output is
    attention over them (the pages' Exact-TopK special case)."""
    B, Hq, Hkv, D, n, k2 = 1, 32, 8, 128, 400, 24
    G = Hq // Hkv
    dims = (B, Hq, Hkv, D)
    kb, k = _rand(61, (B, Hkv, n, D))
    vb, v = _rand(62, (B, Hkv, n, D))
    qb, q = _rand(63, (B, Hq, D))
    ncap = -(-n // 8) * 8
    kt = torch.empty((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    sb = torch.empty((B, Hkv, k2), dtype=torch.int32, device=DEV)
    rkv.rkv_build_kt(dims, k, n, n, None, 0, 1, kt, ncap)
    rkv.rkv_hsa_decode(dims, q, k, v, n, n, kt, ncap, 1, D, k2, 1 / math.sqrt(D), out, sb, None)
    torch.cuda.synchronize()
    kf, vf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), bf16_bits_to_f64(qb)
    out_h, sb_h = out.cpu().numpy(), sb.cpu().numpy()
    for h in range(Hkv):
        qbar = qf[0, h * G:(h + 1) * G].sum(axis=0)
        s = kf[0, h] @ qbar
        check_topk(sb_h[0, h], s, k2, "exact top-k tokens")
        y = oracle.attention(qf[0, h * G:(h + 1) * G], kf[0, h][sb_h[0, h]], vf[0, h][sb_h[0, h]], 1 / math.sqrt(D))
        assert max_abs(out_h[0, h * G:(h + 1) * G], y) <= ATOL_OUT


@pytest.mark.parametrize("n,blk,k2", [(250, 16, 6), (97, 8, 20), (600, 32, 4), (300, 4, 12), (150, 1, 30)])
def test_hsa_decode_mt_parity(n, blk, k2):
    _hsa_case(300 + n, 2, 32, 8, n, blk, 32, k2, mt=True, full_rows=3 * n + 11)


def test_hsa_decode_mt_equals_compacted():
    """MT over (full cache, idx) gives bit-identical results to the compacted path."""
    B, Hq, Hkv, D, full, n, blk, k1, k2 = 2, 32, 8, 128, 900, 300, 16, 32, 7
    dims = (B, Hq, Hkv, D)
    kb, k = _rand(41, (B, Hkv, full, D))
    vb, v = _rand(42, (B, Hkv, full, D))
    _, q = _rand(43, (B, Hq, D))
    rng = np.random.default_rng(44)
    idx = np.stack([np.stack([np.sort(rng.choice(full, n, replace=False)) for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    idx_t = torch.from_numpy(idx).to(DEV)
    kc = torch.stack([torch.stack([k[b, h, idx_t[b, h].long()] for h in range(Hkv)]) for b in range(B)]).contiguous()
    vc = torch.stack([torch.stack([v[b, h, idx_t[b, h].long()] for h in range(Hkv)]) for b in range(B)]).contiguous()
    nblk = -(-n // blk)
    ncap = -(-nblk // 8) * 8
    kt1 = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    kt2 = torch.zeros_like(kt1)
    rkv.rkv_build_kt(dims, k, full, n, idx_t, n, blk, kt1, ncap)
    rkv.rkv_build_kt(dims, kc, n, n, None, 0, blk, kt2, ncap)
    o1 = torch.empty(B, Hq, D, device=DEV)
    o2 = torch.empty_like(o1)
    s1 = torch.empty(B, Hkv, k2, dtype=torch.int32, device=DEV)
    s2 = torch.empty_like(s1)
    rkv.rkv_hsa_decode_mt(dims, q, k, v, full, idx_t, n, n, kt1, ncap, blk, k1, k2, 0.1, o1, s1, None)
    rkv.rkv_hsa_decode(dims, q, kc, vc, n, n, kt2, ncap, blk, k1, k2, 0.1, o2, s2, None)
    torch.cuda.synchronize()
    assert torch.equal(kt1, kt2) and torch.equal(s1, s2) and torch.equal(o1, o2)


def test_hsa_decode_deterministic():
    B, Hq, Hkv, D, n, blk = 4, 32, 8, 128, 3000, 16
    dims = (B, Hq, Hkv, D)
    _, k = _rand(51, (B, Hkv, n, D))
    _, v = _rand(52, (B, Hkv, n, D))
    _, q = _rand(53, (B, Hq, D))
    ncap = -(-(-(-n // blk)) // 8) * 8
    kt = torch.empty((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_build_kt(dims, k, n, n, None, 0, blk, kt, ncap)
    outs = []
    for _ in range(3):
        o = torch.empty(B, Hq, D, device=DEV)
        rkv.rkv_hsa_decode(dims, q, k, v, n, n, kt, ncap, blk, 32, 32, 0.1, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


# ----------------------------------------------------------------- stage 1 --


def _snap_case(seed, B, Hq, Hkv, S, W, P, B1, n_sink=0, cap_extra=5, q_scale=1.0, compact=True, qmod=None):
    D = 128
    G = Hq // Hkv
    dims = (B, Hq, Hkv, D)
    cap = S + cap_extra
    scale = 1 / math.sqrt(D)
    kb, k = _rand(seed, (B, Hkv, cap, D))
    vb, v = _rand(seed + 1, (B, Hkv, cap, D))
    qb, q = _rand(seed + 2, (B, Hq, W, D), q_scale)
    if qmod is not None:
        qb = qmod(qb, kb)
        q = _bf16(qb)
    keep = torch.full((B, Hkv, B1 + 2), -5, dtype=torch.int32, device=DEV)
    ko = torch.empty((B, Hkv, B1 + 1, D), dtype=torch.bfloat16, device=DEV) if compact else None
    vo = torch.empty_like(ko) if compact else None
    L = max(S - W, 0)
    pooled = torch.empty((B, Hkv, max(L, 1)), dtype=torch.float32, device=DEV)
    ws_bytes = rkv.rkv_snap_evict_workspace(dims, S, W)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
    rkv.rkv_snap_evict(dims, q, W, k, v, cap, S, P, n_sink, B1, scale, keep, B1 + 2, ko, vo, B1 + 1,
                       pooled, ws, ws_bytes)
    torch.cuda.synchronize()
    keep_h = keep.cpu().numpy()
    kf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(qb)
    exempt = 0
    for b in range(B):
        for h in range(Hkv):
            ref, pooled_o = oracle.snap_keep(qf[b, h * G:(h + 1) * G], kf[b, h, :S], B1, W, P, scale, n_sink)
            got = keep_h[b, h, :B1]
            assert np.all(keep_h[b, h, B1:] == -5)
            if B1 >= S or L == 0:
                assert got.tolist() == list(range(S))
                continue
            # pooled scores (fp32 accumulation of probabilities)
            pg = pooled[b, h, :L].cpu().numpy().astype(np.float64)
            assert np.max(np.abs(pg - pooled_o) / np.maximum(np.abs(pooled_o), 1e-30)) < 1e-4
            ns = min(n_sink, L)
            assert got[:ns].tolist() == list(range(ns))
            assert got[B1 - min(W, S):].tolist() == list(range(S - min(W, S), S))
            exempt += check_topk(got[ns:B1 - min(W, S)] - ns, pooled_o[ns:], B1 - min(W, S) - ns, "keep")
            if compact:
                assert np.array_equal(t2bits(ko[b, h, :B1]), kb[b, h][got])
                assert np.array_equal(t2bits(vo[b, h, :B1]), vb[b, h][got])
    return exempt


@pytest.mark.parametrize("B,Hq,Hkv,S,W,P,B1,sink", [
    (1, 32, 8, 4096, 32, 63, 1209, 0),      # the 4K workload's shape
    (2, 32, 8, 5000, 32, 63, 700, 0),       # ragged S
    (1, 64, 8, 3000, 32, 63, 500, 0),       # G * W = 256 rows (two row groups)
    (2, 128, 8, 2600, 32, 63, 400, 0),      # G * W = 512 rows: both passes reload Q inside a CTA
    (1, 8, 8, 2100, 32, 7, 300, 4),         # G = 1, pool 7, sinks
    (1, 24, 8, 1500, 32, 1, 100, 0),        # G = 3 (96 rows), no pooling
    (1, 32, 8, 200, 32, 63, 200, 0),        # B1 == S: keep all
    (1, 32, 8, 20, 32, 63, 20, 0),          # prompt shorter than the window
    (1, 32, 8, 70000, 32, 63, 900, 0),      # long prompt, many chunks
    (1, 32, 8, 32768, 32, 63, 1024, 0),     # the 32K batch-8 workload's rows: pool + select over a cluster of 4
    (2, 32, 8, 20000, 32, 63, 700, 4),      # cluster of 3, sinks, ragged last CTA
    (1, 32, 8, 12000, 32, 63, 36, 4),       # cluster, keep count with no prefix slot (window and sinks only)
    (1, 32, 8, 65000, 32, 63, 2000, 0),     # cluster of 8
    (1, 32, 8, 100000, 32, 63, 1500, 4),    # cluster of 13 where the GPU allows more than 8, else pool and select apart
    (1, 32, 8, 5000, 32, 65, 700, 0),       # pool 65: pool and select as separate kernels
    (1, 48, 8, 2500, 32, 63, 300, 0),       # G * W = 192: pass 1 with 256 rows per CTA, 64 of them past the group
    (2, 64, 8, 3000, 20, 63, 400, 2),       # W = 20, G * W = 160: the same with a window off 32, sinks
])
def test_snap_evict_parity(B, Hq, Hkv, S, W, P, B1, sink):
    _snap_case(500 + S, B, Hq, Hkv, S, W, P, B1, sink)


@pytest.mark.parametrize("S", [5000, 20000])
def test_snap_evict_all_scores_tied(S):
    """Zero window queries: every prefix key gets the same score, so the pooled
    scores have an empty range and the select takes its radix path (in one CTA,
    or over a cluster for the longer prompt); the kept prefix positions must be
    the lowest ones (no tie-band exemption)."""
    assert _snap_case(31, 2, 32, 8, S, 32, 63, 700, q_scale=0.0) == 0


@pytest.mark.parametrize("S", [5000, 20000])
def test_snap_evict_crowded_boundary_bucket(S):
    """Window queries zero except one row per group, twice key 5: that key's
    score spans the range and every other pooled score lies within a sliver
    of the minimum, so the 1024-bucket histogram puts thousands of candidates
    in the boundary bucket and the select falls back to its radix path."""
    G = 32 // 8

    def qmod(qb, kb):
        qb = np.zeros_like(qb)
        for b in range(qb.shape[0]):
            for h in range(8):
                qb[b, h * G, 0] = f32_to_bf16_bits(bf16_bits_to_f32(kb[b, h, 5]) * np.float32(2.0))
        return qb
    _snap_case(41, 1, 32, 8, S, 32, 63, 700, qmod=qmod)


def test_snap_evict_mask_mode_and_peaked():
    _snap_case(9, 1, 32, 8, 3000, 32, 63, 400, compact=False, q_scale=4.0)


@pytest.mark.parametrize("S_rows,B1_rows,Hq,n_sink,compact", [
    ([2500, 6000, 1111, 4097], [400, 900, 200, 700], 32, 0, True),     # lengths off the 2048-key chunk and W
    ([3000, 20, 5000], [300, 20, 5000], 32, 0, False),                 # a row shorter than W, a row keeping all
    ([7000, 2049, 3333], [1000, 300, 600], 64, 4, True),                # G = 8, sinks
    ([9000, 30000, 300, 16500], [800, 1024, 100, 700], 32, 4, True),   # pool + select over clusters of 4; a
                                                                        # short row leaves CTAs without positions
])
def test_snap_evict_ragged_parity(S_rows, B1_rows, Hq, n_sink, compact):
    """Per-row prompt lengths and keep counts in one launch: every row matches
    the oracle's stage 1 on its own prefix (pooled scores within 1e-4, keep set
    under the tie rule, window and sinks kept, compaction bit-exact), and no
    keep entry or compacted row past a row's own count is written."""
    B, Hkv, D, W, P = len(S_rows), 8, 128, 32, 63
    G = Hq // Hkv
    dims = (B, Hq, Hkv, D)
    S_max, B1_max = max(S_rows), max(B1_rows)
    cap = S_max + 7
    scale = 1 / math.sqrt(D)
    kb, k = _rand(701, (B, Hkv, cap, D))
    vb, v = _rand(702, (B, Hkv, cap, D))
    qb, q = _rand(703, (B, Hq, W, D))
    keep = torch.full((B, Hkv, B1_max + 3), -5, dtype=torch.int32, device=DEV)
    ko = torch.full((B, Hkv, B1_max + 1, D), float("nan"), dtype=torch.bfloat16, device=DEV) if compact else None
    vo = torch.full_like(ko, float("nan")) if compact else None
    Lmax = max(S_max - W, 1)
    pooled = torch.full((B, Hkv, Lmax), float("nan"), dtype=torch.float32, device=DEV)
    ws_bytes = rkv.rkv_snap_evict_workspace(dims, S_max, W)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
    S_dev = torch.tensor(S_rows, dtype=torch.int32, device=DEV)
    B1_dev = torch.tensor(B1_rows, dtype=torch.int32, device=DEV)
    rkv.rkv_snap_evict_ragged(dims, q, W, k, v, cap, S_dev, S_max, P, n_sink, B1_dev, B1_max, scale, keep,
                              B1_max + 3, ko, vo, B1_max + 1, pooled, ws, ws_bytes)
    torch.cuda.synchronize()
    assert rkv.rkv_read_device_flags() == 0
    keep_h = keep.cpu().numpy()
    kf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(qb)
    for b in range(B):
        S, B1 = S_rows[b], min(B1_rows[b], S_rows[b])
        L = max(S - W, 0)
        for h in range(Hkv):
            got = keep_h[b, h, :B1]
            assert np.all(keep_h[b, h, B1:] == -5), f"row {b}: keep written past B1_b"
            if compact:
                assert torch.isnan(ko[b, h, B1:].float()).all() and torch.isnan(vo[b, h, B1:].float()).all()
            if B1 >= S or L == 0:
                assert got.tolist() == list(range(S))
            else:
                ref, pooled_o = oracle.snap_keep(qf[b, h * G:(h + 1) * G], kf[b, h, :S], B1, W, P, scale, n_sink)
                pg = pooled[b, h, :L].cpu().numpy().astype(np.float64)
                assert np.max(np.abs(pg - pooled_o) / np.maximum(np.abs(pooled_o), 1e-30)) < 1e-4, f"row {b} pooled"
                ns = min(n_sink, L)
                assert got[:ns].tolist() == list(range(ns))
                assert got[B1 - W:].tolist() == list(range(S - W, S))
                check_topk(got[ns:B1 - W] - ns, pooled_o[ns:], B1 - W - ns, f"row {b} keep")
            if compact:
                assert np.array_equal(t2bits(ko[b, h, :B1]), kb[b, h][got])
                assert np.array_equal(t2bits(vo[b, h, :B1]), vb[b, h][got])


@pytest.mark.parametrize("page,S_rows,B1_rows,compact", [
    (16, [2500, 6000, 1111], [400, 900, 200], True),
    (64, [4097, 3000], [700, 3000], True),          # the second row keeps everything
    (128, [5000, 2049, 777], [600, 300, 120], False),
    (64, [12000, 3000], [900, 400], True),           # pool + select over a cluster of 2
])
def test_snap_evict_paged_parity(page, S_rows, B1_rows, compact):
    """Stage 1 reading its prompt K/V through a block table: each row's prompt is
    scattered over a shuffled set of pages (unused page slots hold large random
    rows).  Every row matches the oracle on its own prefix (pooled scores within
    1e-4, keep set under the tie rule, compaction bit-exact), and the keep lists
    and pooled scores equal rkv_snap_evict_ragged's over the same rows held
    densely."""
    B, Hq, Hkv, D, W, P = len(S_rows), 32, 8, 128, 32, 63
    G = Hq // Hkv
    dims = (B, Hq, Hkv, D)
    S_max, B1_max = max(S_rows), max(B1_rows)
    npg_row = -(-S_max // page)
    scale = 1 / math.sqrt(D)
    kb = small_random(721 + page, (B, Hkv, npg_row * page, D))
    vb = small_random(722 + page, (B, Hkv, npg_row * page, D))
    qb, q = _rand(723 + page, (B, Hq, W, D))
    rng = np.random.default_rng(page)
    bt, num_pages = _page_table(rng, B, npg_row, 5)
    kpb = small_random(724 + page, (num_pages, Hkv, page, D), 50.0)
    vpb = small_random(725 + page, (num_pages, Hkv, page, D), 50.0)
    for b in range(B):
        for j in range(-(-S_rows[b] // page)):
            r = min(page, S_rows[b] - j * page)
            kpb[bt[b, j], :, :r] = kb[b, :, j * page:j * page + r]
            vpb[bt[b, j], :, :r] = vb[b, :, j * page:j * page + r]
    S_dev = torch.tensor(S_rows, dtype=torch.int32, device=DEV)
    B1_dev = torch.tensor(B1_rows, dtype=torch.int32, device=DEV)
    ws_bytes = rkv.rkv_snap_evict_workspace(dims, S_max, W)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
    Lmax = S_max - W

    def run(paged):
        keep = torch.full((B, Hkv, B1_max + 2), -5, dtype=torch.int32, device=DEV)
        ko = torch.full((B, Hkv, B1_max, D), float("nan"), dtype=torch.bfloat16, device=DEV) if compact else None
        vo = torch.full_like(ko, float("nan")) if compact else None
        pooled = torch.full((B, Hkv, Lmax), float("nan"), dtype=torch.float32, device=DEV)
        if paged:
            rkv.rkv_snap_evict_paged(dims, q, W, _bf16(kpb), _bf16(vpb), num_pages, page,
                                     torch.from_numpy(bt).to(DEV), npg_row, S_dev, S_max, P, 0, B1_dev, B1_max, scale,
                                     keep, B1_max + 2, ko, vo, B1_max, pooled, ws, ws_bytes)
        else:
            rkv.rkv_snap_evict_ragged(dims, q, W, _bf16(kb), _bf16(vb), npg_row * page, S_dev, S_max, P, 0, B1_dev,
                                      B1_max, scale, keep, B1_max + 2, ko, vo, B1_max, pooled, ws, ws_bytes)
        torch.cuda.synchronize()
        assert rkv.rkv_read_device_flags() == 0
        return keep, ko, vo, pooled

    keep, ko, vo, pooled = run(True)
    keep_d, _, _, pooled_d = run(False)
    assert torch.equal(keep, keep_d)
    for b in range(B):
        L = max(S_rows[b] - W, 0)
        if B1_rows[b] < S_rows[b]:              # (a row that keeps everything scores nothing)
            assert torch.equal(pooled[b, :, :L], pooled_d[b, :, :L])
    keep_h = keep.cpu().numpy()
    kf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(qb)
    for b in range(B):
        S, B1 = S_rows[b], min(B1_rows[b], S_rows[b])
        L = S - W
        for h in range(Hkv):
            got = keep_h[b, h, :B1]
            assert np.all(keep_h[b, h, B1:] == -5)
            if B1 >= S:
                assert got.tolist() == list(range(S))
            else:
                ref, pooled_o = oracle.snap_keep(qf[b, h * G:(h + 1) * G], kf[b, h, :S], B1, W, P, scale)
                pg = pooled[b, h, :L].cpu().numpy().astype(np.float64)
                assert np.max(np.abs(pg - pooled_o) / np.maximum(np.abs(pooled_o), 1e-30)) < 1e-4
                assert got[B1 - W:].tolist() == list(range(S - W, S))
                check_topk(got[:B1 - W], pooled_o, B1 - W, f"row {b} keep")
            if compact:
                assert np.array_equal(t2bits(ko[b, h, :B1]), kb[b, h][got])
                assert np.array_equal(t2bits(vo[b, h, :B1]), vb[b, h][got])


def test_snap_evict_ragged_out_of_range_flagged():
    """A prompt length past S_max and a keep count below the window are clamped
    (row 0 to S_max, row 1 to W + 0) and set bit 1 of the device error word."""
    B, Hq, Hkv, D, W, P = 2, 32, 8, 128, 32, 63
    dims = (B, Hq, Hkv, D)
    S_max, B1_max = 3000, 500
    cap = S_max
    _, k = _rand(711, (B, Hkv, cap, D))
    _, q = _rand(712, (B, Hq, W, D))
    keep = torch.full((B, Hkv, B1_max), -5, dtype=torch.int32, device=DEV)
    ws_bytes = rkv.rkv_snap_evict_workspace(dims, S_max, W)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    rkv.rkv_snap_evict_ragged(dims, q, W, k, None, cap, torch.tensor([9000, 2000], dtype=torch.int32, device=DEV),
                              S_max, P, 0, torch.tensor([400, 3], dtype=torch.int32, device=DEV), B1_max, 0.1, keep,
                              B1_max, None, None, 0, None, ws, ws_bytes)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_read_device_flags()
    assert "0x2" in str(e.value)
    keep_h = keep.cpu().numpy()
    assert keep_h[0, :, 400 - W:400].tolist() == [list(range(S_max - W, S_max))] * Hkv
    assert keep_h[1, :, :W].tolist() == [list(range(2000 - W, 2000))] * Hkv and np.all(keep_h[1, :, W:] == -5)


# ------------------------------------------------------------- fused append --


@pytest.mark.parametrize("mt", [False, True])
@pytest.mark.parametrize("n0,blk,k2", [(300, 16, 5), (320, 16, 7), (0, 16, 3), (95, 32, 2), (1000, 8, 40)])
def test_fused_append_equals_separate(mt, n0, blk, k2):
    """HSA with the append fused in == rkv_append_kv followed by HSA: caches,
    candidate rows, KT, selections and outputs all bit-identical."""
    B, Hq, Hkv, D, k1 = 2, 32, 8, 128, 32
    dims = (B, Hq, Hkv, D)
    steps = 3
    cap = n0 + steps + 5 if not mt else 3 * n0 + 40
    _, k = _rand(61 + n0, (B, Hkv, cap, D))
    _, v = _rand(62 + n0, (B, Hkv, cap, D))
    _, qs = _rand(63, (steps, B, Hq, D))
    _, kn = _rand(64, (steps, B, Hkv, D))
    _, vn = _rand(65, (steps, B, Hkv, D))
    ncap = -(-(-(-(n0 + steps) // blk)) // 8) * 8
    idx_cap = n0 + steps
    if mt:
        rng = np.random.default_rng(66)
        rows = np.stack([np.stack([np.sort(rng.choice(2 * n0 + 1, n0, replace=False)) for _ in range(Hkv)])
                         for _ in range(B)]).astype(np.int32)
        idx = torch.zeros((B, Hkv, idx_cap), dtype=torch.int32, device=DEV)
        idx[:, :, :n0] = torch.from_numpy(rows).to(DEV)
    states = []
    for fused in (False, True):
        kk, vv = k.clone(), v.clone()
        kt = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
        ii = idx.clone() if mt else None
        if n0:
            rkv.rkv_build_kt(dims, kk, cap, n0, ii, idx_cap, blk, kt, ncap)
        outs, sels = [], []
        for s in range(steps):
            o = torch.empty(B, Hq, D, device=DEV)
            sb = torch.empty(B, Hkv, k2, dtype=torch.int32, device=DEV)
            n, row = n0 + s, 2 * n0 + 1 + s
            if fused:
                if mt:
                    rkv.rkv_hsa_decode_mt(dims, qs[s], kk, vv, cap, ii, idx_cap, n, kt, ncap, blk, k1, k2, 0.1, o, sb,
                                          None, kn[s], vn[s], row)
                else:
                    rkv.rkv_hsa_decode(dims, qs[s], kk, vv, cap, n, kt, ncap, blk, k1, k2, 0.1, o, sb, None, kn[s],
                                       vn[s])
            else:
                rkv.rkv_append_kv(dims, kn[s], vn[s], kk, vv, cap, n, row if mt else n, ii, idx_cap, kt, ncap, blk)
                if mt:
                    rkv.rkv_hsa_decode_mt(dims, qs[s], kk, vv, cap, ii, idx_cap, n + 1, kt, ncap, blk, k1, k2, 0.1, o,
                                          sb)
                else:
                    rkv.rkv_hsa_decode(dims, qs[s], kk, vv, cap, n + 1, kt, ncap, blk, k1, k2, 0.1, o, sb)
            outs.append(o)
            sels.append(sb)
        torch.cuda.synchronize()
        states.append((kk, vv, kt, ii, outs, sels))
    a, b = states
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    if mt:
        assert torch.equal(a[3], b[3])
    for s in range(steps):
        assert torch.equal(a[5][s], b[5][s]) and torch.equal(a[4][s], b[4][s])


# ----------------------------------------- multi-turn over full-cache blocks --


def _check_blocks_masked(got, s, k2, what):
    """check_topk for scores with +-inf entries: an infinite k-th score admits no tie band."""
    k = min(k2, s.shape[0])
    if np.isfinite(oracle.kth_value(s, k)):
        return check_topk(got, s, k2, what)
    assert got.tolist() == oracle.topk_lowest_index(s, k).tolist(), what
    return 0


@pytest.mark.parametrize("B,Hq,Hkv,n_prompt,n_dec,blk,k1,k2,dens", [
    (2, 32, 8, 300, 0, 16, 32, 5, 0.3),       # G = 4, ragged tail
    (1, 32, 8, 517, 5, 16, 16, 9, 0.2),       # decoded rows share a block with the prompt's last rows
    (1, 64, 8, 1000, 3, 32, 64, 11, 0.5),     # G = 8, block 32
    (1, 32, 2, 333, 1, 8, 128, 40, 0.1),      # G = 16, block 8, all channels
    (1, 32, 8, 700, 2, 1, 32, 40, 0.3),       # token-level blocks, gathered rows
    (1, 32, 8, 333, 4, 12, 32, 7, 0.25),      # block 12, gathered rows
    (2, 32, 8, 130, 0, 16, 32, 64, 0.3),      # k2 >= blocks
    (1, 32, 8, 5000, 0, 16, 32, 30, 0.02),    # mostly empty blocks
    (1, 32, 8, 600, 0, 16, 32, 50, 0.02),     # fewer blocks with candidates than k2
])
def test_hsa_decode_mt_masked_parity(B, Hq, Hkv, n_prompt, n_dec, blk, k1, k2, dens):
    """The multi-turn reading over fixed blocks of the full cache: keep-list mask,
    candidate-only KT (bit-exact) and a few decode steps with the fused append,
    each against the oracle."""
    D, G, steps = 128, Hq // Hkv, 4
    dims = (B, Hq, Hkv, D)
    scale = 1 / math.sqrt(D)
    seed = n_prompt + 7 * blk + k2
    cap = n_prompt + n_dec + steps + 5
    kb, k = _rand(seed, (B, Hkv, cap, D))
    vb, v = _rand(seed + 1, (B, Hkv, cap, D))
    qb = small_random(seed + 2, (steps, B, Hq, D))
    knb = small_random(seed + 3, (steps, B, Hkv, D))
    vnb = small_random(seed + 4, (steps, B, Hkv, D))
    kf, vf, qf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb), bf16_bits_to_f64(qb)
    knf, vnf = bf16_bits_to_f64(knb), bf16_bits_to_f64(vnb)
    rng = np.random.default_rng(seed)
    nkeep = max(1, int(dens * n_prompt))
    keep = np.stack([np.stack([np.sort(rng.choice(n_prompt, nkeep, replace=False)) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32)
    keep_t = torch.from_numpy(keep).to(DEV)
    mask_ld = -(-cap // 32)
    mask = torch.full((B, Hkv, mask_ld), -1, dtype=torch.int32, device=DEV)
    rkv.rkv_keep_mask(dims, keep_t, nkeep, nkeep, n_prompt, mask, mask_ld)
    n = n_prompt + n_dec
    ncap = -(-(-(-cap // blk)) // 8) * 8
    kt = torch.full((B, Hkv, 2, D, ncap), float("nan"), dtype=torch.bfloat16, device=DEV)
    rkv.rkv_build_kt_masked(dims, k, cap, n, mask, mask_ld, n_prompt, blk, kt, ncap)
    torch.cuda.synchronize()
    words = mask.cpu().numpy().view(np.uint32)
    ktg = t2f64(kt)
    state = {}
    for b in range(B):
        for h in range(Hkv):
            cand = oracle.candidate_rows(keep[b, h], n_prompt, cap)
            bits = np.unpackbits(words[b, h, :-(-n_prompt // 32)].view(np.uint8), bitorder="little")[:n_prompt]
            assert bits.astype(bool).tolist() == cand[:n_prompt].tolist(), "mask bits"
            kmax, kmin, has = oracle.build_kt_masked(kf[b, h], n, cand, blk)
            nb = kmax.shape[1]
            assert np.array_equal(ktg[b, h, 0, :, :nb], kmax) and np.array_equal(ktg[b, h, 1, :, :nb], kmin)
            state[(b, h)] = [kmax, kmin, has, cand]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    sb = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((B, Hkv, k1), -7, dtype=torch.int32, device=DEV)
    kn_t, vn_t, q_t = _bf16(knb), _bf16(vnb), _bf16(qb)
    worst, exempt = 0.0, 0
    for s in range(steps):
        fused = s != 2                      # step 2 attends without appending
        rkv.rkv_hsa_decode_mt_masked(dims, q_t[s], k, v, cap, n, mask, mask_ld, n_prompt, kt, ncap, blk, k1, k2,
                                     scale, out, sb, sc, kn_t[s] if fused else None, vn_t[s] if fused else None)
        torch.cuda.synchronize()
        if fused:
            kf[:, :, n] = knf[s]
            vf[:, :, n] = vnf[s]
        n_att = n + (1 if fused else 0)
        out_h, sb_h, sc_h = out.cpu().numpy(), sb.cpu().numpy(), sc.cpu().numpy()
        for (b, h), st in state.items():
            if fused:
                st[0], st[1], st[2] = oracle.kt_append_masked(st[0], st[1], st[2], n, knf[s, b, h], blk)
            qg = qf[s, b, h * G:(h + 1) * G]
            res = oracle.hsa_decode_mt_masked(qg, kf[b, h], vf[b, h], n_att, st[3], st[0], st[1], st[2], blk, k1,
                                              k2, scale)
            assert sc_h[b, h].tolist() == res["i1"].tolist(), "channel set differs"
            k2e = min(k2, res["s"].shape[0])
            exempt += _check_blocks_masked(sb_h[b, h, :k2e], res["s"], k2, f"step {s} blocks")
            assert np.all(sb_h[b, h, k2e:] == -1)
            if np.array_equal(sb_h[b, h, :k2e], res["i2"]):
                y = res["y"]
            else:
                tok = oracle.block_tokens(sb_h[b, h, :k2e], n_att, blk)
                tok = tok[st[3][tok]]
                y = oracle.attention(qg, kf[b, h][tok], vf[b, h][tok], scale)
            worst = max(worst, max_abs(out_h[b, h * G:(h + 1) * G], y))
        n = n_att
    ktg = t2f64(kt)
    for (b, h), st in state.items():
        nb = st[0].shape[1]
        assert np.array_equal(ktg[b, h, 0, :, :nb], st[0]) and np.array_equal(ktg[b, h, 1, :, :nb], st[1])
    assert worst <= ATOL_OUT, worst


def test_hsa_decode_mt_masked_all_candidates_equals_dense():
    """With every prompt row kept, the reading over full-cache blocks scores the
    same blocks as the dense decode; with k2 large enough to take the newest
    block anyway, both return the same blocks and bit-identical outputs."""
    B, Hq, Hkv, D, n, blk, k1 = 2, 32, 8, 128, 640, 16, 32
    k2 = n // blk
    dims = (B, Hq, Hkv, D)
    kb, k = _rand(61, (B, Hkv, n + 8, D))
    vb, v = _rand(62, (B, Hkv, n + 8, D))
    _, q = _rand(63, (B, Hq, D))
    keep = torch.arange(n, dtype=torch.int32, device=DEV).expand(B, Hkv, n).contiguous()
    mask = torch.zeros((B, Hkv, n // 32), dtype=torch.int32, device=DEV)
    rkv.rkv_keep_mask(dims, keep, n, n, n, mask, n // 32)
    ncap = n // blk
    kt1 = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
    kt2 = torch.zeros_like(kt1)
    rkv.rkv_build_kt_masked(dims, k, n + 8, n, mask, n // 32, n, blk, kt1, ncap)
    rkv.rkv_build_kt(dims, k, n + 8, n, None, 0, blk, kt2, ncap)
    o1 = torch.empty(B, Hq, D, device=DEV)
    o2 = torch.empty_like(o1)
    s1 = torch.empty(B, Hkv, k2, dtype=torch.int32, device=DEV)
    s2 = torch.empty_like(s1)
    rkv.rkv_hsa_decode_mt_masked(dims, q, k, v, n + 8, n, mask, n // 32, n, kt1, ncap, blk, k1, k2, 0.1, o1, s1)
    rkv.rkv_hsa_decode(dims, q, k, v, n + 8, n, kt2, ncap, blk, k1, k2, 0.1, o2, s2)
    torch.cuda.synchronize()
    assert torch.equal(kt1, kt2) and torch.equal(s1, s2) and torch.equal(o1, o2)


# --------------------------------------------------- host-resident prompt V --


def test_compact_kt_reads_page_locked_host_v():
    """A prompt V in page-locked host memory is compacted in place (only the kept
    rows cross the host link) with results identical to a device-resident V;
    pageable host memory is refused on the host before any launch."""
    B, Hq, Hkv, D, cap, B1, blk = 2, 8, 2, 128, 1500, 333, 16
    dims = (B, Hq, Hkv, D)
    kb, k = _rand(71, (B, Hkv, cap, D))
    vb, v = _rand(72, (B, Hkv, cap, D))
    rng = np.random.default_rng(73)
    keep = np.stack([np.stack([np.sort(rng.choice(cap, B1, replace=False)) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32)
    keep_t = torch.from_numpy(keep).to(DEV)
    ncap = -(-(-(-B1 // blk)) // 8) * 8
    outs = []
    for vv in (v, v.cpu().pin_memory()):
        ko = torch.zeros((B, Hkv, B1, D), dtype=torch.bfloat16, device=DEV)
        vo = torch.zeros_like(ko)
        kt = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.bfloat16, device=DEV)
        rkv.rkv_compact_kt(dims, k, vv, cap, keep_t, B1, B1, ko, vo, B1, blk, kt, ncap)
        torch.cuda.synchronize()
        outs.append((ko, vo, kt))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    vf = bf16_bits_to_f64(vb)
    got = t2f64(outs[1][1])
    for b in range(B):
        for h in range(Hkv):
            assert np.array_equal(got[b, h], oracle.compact(vf[b, h], keep[b, h]))
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_compact_kt(dims, k, v.cpu(), cap, keep_t, B1, B1, outs[0][0], outs[0][1], B1, blk, outs[0][2], ncap)
    assert e.value.status == 1


# ------------------------------------------------------ e4m3 (FP8) storage --


def _fp8_case(seed, B, Hkv, cap, B1, k_mag=3.0):
    rng = np.random.default_rng(seed)
    kb = small_random(seed, (B, Hkv, cap, 128), k_mag)
    vb = small_random(seed + 1, (B, Hkv, cap, 128))
    keep = np.stack([np.stack([np.sort(rng.choice(cap, B1, replace=False)) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32)
    # per-(b, h) scales, some small enough that the largest keys saturate
    ks = rng.uniform(0.004, 0.05, (B, Hkv)).astype(np.float32)
    vs = rng.uniform(0.002, 0.02, (B, Hkv)).astype(np.float32)
    return kb, vb, keep, ks, vs


@pytest.mark.parametrize("B1,blk", [(300, 16), (1, 16), (1000, 32), (259, 128), (77, 8)])
def test_compact_kt_fp8_bit_exact(B1, blk):
    """e4m3 compaction: codes of row / scale equal the oracle's bit for bit
    (saturated and negative-zero codes included), KT bounds equal the max /
    min of the key codes' values."""
    B, Hq, Hkv, D, cap = 2, 8, 2, 128, 2 * B1 + 37
    kb, vb, keep, ks, vs = _fp8_case(80 + B1, B, Hkv, cap, B1)
    dims = (B, Hq, Hkv, D)
    ncap = -(-(-(-B1 // blk)) // 16) * 16
    ko = torch.zeros((B, Hkv, B1 + 3, D), dtype=torch.uint8, device=DEV)
    vo = torch.zeros_like(ko)
    kt = torch.full((B, Hkv, 2, D, ncap), 0x55, dtype=torch.uint8, device=DEV)
    ks_t, vs_t = torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV)
    rkv.rkv_compact_kt_fp8(dims, _bf16(kb), _bf16(vb), cap, torch.from_numpy(keep).to(DEV), B1, B1, ks_t, vs_t, ko,
                           vo, B1 + 3, blk, kt, ncap)
    torch.cuda.synchronize()
    kog, vog, ktg = ko.cpu().numpy(), vo.cpu().numpy(), kt.cpu().numpy()
    kf, vf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb)
    nblk = -(-B1 // blk)
    sat = 0
    for b in range(B):
        for h in range(Hkv):
            kc = oracle.fp8_quantize(kf[b, h][keep[b, h]], ks[b, h])
            vc = oracle.fp8_quantize(vf[b, h][keep[b, h]], vs[b, h])
            assert np.array_equal(kog[b, h, :B1], kc), "key codes"
            assert np.array_equal(vog[b, h, :B1], vc), "value codes"
            sat += int(np.sum((kc & 0x7F) == 0x7E))
            kmax, kmin = oracle.build_kt_fp8(kc, B1, blk)
            assert np.array_equal(oracle.e4m3_decode(ktg[b, h, 0, :, :nblk]), kmax)
            assert np.array_equal(oracle.e4m3_decode(ktg[b, h, 1, :, :nblk]), kmin)
            assert np.all(ktg[b, h, :, :, nblk:] == 0x55)
    assert np.all(kog[:, :, B1:] == 0)
    if B1 >= 259:
        assert sat > 0, "the case should exercise saturation"


@pytest.mark.parametrize("B,Hq,Hkv,B1,blk,k1,k2", [
    (2, 32, 8, 300, 16, 32, 5),       # G = 4, ragged tail
    (1, 64, 8, 1000, 32, 64, 11),     # G = 8, block 32
    (1, 32, 2, 333, 8, 128, 40),      # G = 16, block 8, all channels
    (2, 32, 8, 130, 16, 32, 64),      # k2 >= blocks: full attention
    (1, 32, 8, 5000, 16, 32, 30),     # several CTAs per pair, KT prefetch
    (1, 32, 8, 20000, 16, 32, 300),   # chunked KT gather, several rounds per CTA
])
def test_hsa_decode_fp8_parity(B, Hq, Hkv, B1, blk, k1, k2):
    """Decode steps over the e4m3 cache (three with the fused append, one
    without) against the oracle on the stored codes: channels exact, blocks by
    the tie rule, outputs within 2e-3; the appended rows' codes and the KT
    bounds after the appends bit-exact."""
    D, G, steps = 128, Hq // Hkv, 4
    dims = (B, Hq, Hkv, D)
    scale = 1 / math.sqrt(D)
    cap_in = B1 + 57
    kb, vb, keep, ks, vs = _fp8_case(90 + B1, B, Hkv, cap_in, B1, k_mag=1.0)
    cap = B1 + steps + 5
    ncap = -(-(-(-cap // blk)) // 16) * 16
    ko = torch.zeros((B, Hkv, cap, D), dtype=torch.uint8, device=DEV)
    vo = torch.zeros_like(ko)
    kt = torch.zeros((B, Hkv, 2, D, ncap), dtype=torch.uint8, device=DEV)
    ks_t, vs_t = torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV)
    rkv.rkv_compact_kt_fp8(dims, _bf16(kb), _bf16(vb), cap_in, torch.from_numpy(keep).to(DEV), B1, B1, ks_t, vs_t,
                           ko, vo, cap, blk, kt, ncap)
    qb = small_random(91 + B1, (steps, B, Hq, D))
    knb = small_random(92 + B1, (steps, B, Hkv, D))
    vnb = small_random(93 + B1, (steps, B, Hkv, D))
    qf, knf, vnf = bf16_bits_to_f64(qb), bf16_bits_to_f64(knb), bf16_bits_to_f64(vnb)
    kf, vf = bf16_bits_to_f64(kb), bf16_bits_to_f64(vb)
    state = {}
    for b in range(B):
        for h in range(Hkv):
            kc = list(oracle.fp8_quantize(kf[b, h][keep[b, h]], ks[b, h]))
            vc = list(oracle.fp8_quantize(vf[b, h][keep[b, h]], vs[b, h]))
            kmax, kmin = oracle.build_kt_fp8(np.array(kc), B1, blk)
            state[(b, h)] = [kc, vc, kmax, kmin]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    sb = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((B, Hkv, k1), -7, dtype=torch.int32, device=DEV)
    q_t, kn_t, vn_t = _bf16(qb), _bf16(knb), _bf16(vnb)
    n, worst, exempt = B1, 0.0, 0
    for s in range(steps):
        fused = s != 1
        rkv.rkv_hsa_decode_fp8(dims, q_t[s], ko, vo, cap, n, ks_t, vs_t, kt, ncap, blk, k1, k2, scale, out, sb, sc,
                               kn_t[s] if fused else None, vn_t[s] if fused else None)
        torch.cuda.synchronize()
        out_h, sb_h, sc_h = out.cpu().numpy(), sb.cpu().numpy(), sc.cpu().numpy()
        n_att = n + (1 if fused else 0)
        for (b, h), st in state.items():
            if fused:
                kcode = oracle.fp8_quantize(knf[s, b, h][None], ks[b, h])[0]
                vcode = oracle.fp8_quantize(vnf[s, b, h][None], vs[b, h])[0]
                st[0].append(kcode)
                st[1].append(vcode)
                st[2], st[3] = oracle.kt_append(st[2], st[3], n, oracle.e4m3_decode(kcode), blk)
            Kc, Vc = np.array(st[0]), np.array(st[1])
            qg = qf[s, b, h * G:(h + 1) * G]
            res = oracle.hsa_decode_fp8(qg, Kc, Vc, n_att, st[2], st[3], ks[b, h], vs[b, h], blk, k1, k2, scale)
            assert sc_h[b, h].tolist() == res["i1"].tolist(), "channel set differs"
            k2e = min(k2, res["s"].shape[0])
            exempt += check_topk(sb_h[b, h, :k2e], res["s"], k2, f"step {s} blocks")
            if np.array_equal(sb_h[b, h, :k2e], res["i2"]):
                y = res["y"]
            else:
                tok = oracle.block_tokens(sb_h[b, h, :k2e], n_att, blk)
                y = oracle.attention(qg, oracle.e4m3_decode(Kc[tok]) * float(ks[b, h]),
                                     oracle.e4m3_decode(Vc[tok]) * float(vs[b, h]), scale)
            worst = max(worst, max_abs(out_h[b, h * G:(h + 1) * G], y))
        n = n_att
    kog, vog, ktg = ko.cpu().numpy(), vo.cpu().numpy(), kt.cpu().numpy()
    for (b, h), st in state.items():
        assert np.array_equal(kog[b, h, :n], np.array(st[0])) and np.array_equal(vog[b, h, :n], np.array(st[1]))
        nb = st[2].shape[1]
        assert np.array_equal(oracle.e4m3_decode(ktg[b, h, 0, :, :nb]), st[2])
        assert np.array_equal(oracle.e4m3_decode(ktg[b, h, 1, :, :nb]), st[3])
    assert worst <= ATOL_OUT, worst
