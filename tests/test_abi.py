"""CPU checks of the C-ABI library: it loads, exports every symbol that
include/rkv.h declares, its host-side budget helper agrees with the oracle,
and argument errors are reported before any GPU work (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

import oracle
from two_stage_kv_gb300 import build, rkv
from two_stage_kv_gb300.synth import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(rkv.LIB_PATH):
        build.build()
    return rkv.lib()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "rkv.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?(rkv_[a-z_0-9]+)\(", text, re.M)))


def test_header_symbols_exported(lib):
    syms = declared_symbols()
    assert len(syms) >= 9
    assert sorted(rkv.EXPORTED) == syms
    for s in syms:
        assert hasattr(lib, s), s
        assert ctypes.cast(getattr(lib, s), ctypes.c_void_p).value


def test_abi_version(lib):
    assert rkv.rkv_abi_version() == 1


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_budget_split_matches_oracle(lib, name):
    wl = WORKLOADS[name]
    for turn in range(wl.n_turns):
        S = wl.turn_context(turn)
        r, B1, k2 = rkv.rkv_budget_split(S, wl.t, wl.blk, wl.W)
        ro, B1o, k2o = oracle.budget_split(S, wl.t, wl.blk, wl.W)
        assert abs(r - ro) < 1e-12 and B1 == B1o and k2 == k2o


def test_budget_split_override_and_errors(lib):
    assert rkv.rkv_budget_split(32768, 1024, 16, 32, 0.3) == (0.3, *oracle.budget_split(32768, 1024, 16, 32, 0.3)[1:])
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_budget_split(0, 1, 16)
    assert e.value.status == 1


D4 = (1, 32, 8, 128)


@pytest.mark.parametrize("call,status", [
    (lambda: rkv.rkv_hsa_decode((1, 32, 8, 64), 16, 16, 16, 100, 10, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 2),
    (lambda: rkv.rkv_hsa_decode((1, 30, 8, 128), 16, 16, 16, 100, 10, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 0, 16, 16, 100, 10, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 0, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 101, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 100, 16, 16, 129, 8, 4, 0.1, 16, stream=0), 2),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 100, 16, 104, 0, 8, 4, 0.1, 16, stream=0), 2),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 100, 16, 3, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 100, 16, 10, 16, 0, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 100, 16, 10, 16, 129, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 16, 16, 16, 100, 100, 16, 10, 16, 8, 0, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode(D4, 8, 16, 16, 100, 100, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_mt(D4, 16, 16, 16, 100, None, 0, 10, 16, 10, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_snap_evict(D4, 16, 32, 16, 16, 100, 100, 64, 0, 50, 0.1, 16, 50, 16, 16, 50, None, 16,
                                1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict(D4, 16, 32, 16, 16, 100, 100, 63, 0, 50, 0.1, 16, 50, 16, 16, 50, None, None,
                                0, stream=0), 3),
    (lambda: rkv.rkv_snap_evict(D4, 16, 32, 16, 16, 100, 100, 63, 0, 20, 0.1, 16, 20, 16, 16, 20, None, 256,
                                1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict(D4, 16, 32, 16, 16, 100, 100, 63, 0, 50, 0.1, 16, 40, 16, 16, 50, None, 256,
                                1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict(D4, 16, 32, 16, 16, 100, 100, 63, 0, 99, 0.1, 16, 99, 16, None, 99, None, 256,
                                1 << 30, stream=0), 1),
    (lambda: rkv.rkv_compact_kt(D4, 16, 16, 100, 16, 50, 50, 16, 16, 50, 16, 16, 6, stream=0), 1),
    (lambda: rkv.rkv_compact_kt(D4, 16, 16, 100, 16, 50, 50, 16, 16, 40, 16, 16, 8, stream=0), 1),
    (lambda: rkv.rkv_compact_kt(D4, 8, 16, 100, 16, 50, 50, 16, 16, 50, 16, 16, 8, stream=0), 1),
    (lambda: rkv.rkv_compact_kt(D4, 16, 16, 100, 16, 50, 50, 16, 16, 50, 16, 16, 0, stream=0), 1),
    (lambda: rkv.rkv_compact_kt(D4, 16, 16, 100, 16, 40, 50, 16, 16, 50, 16, 16, 8, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_ragged(D4, 16, 16, 16, 100, None, 50, 16, 16, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_ragged(D4, 16, 16, 16, 100, 16, 0, 16, 16, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_ragged(D4, 16, 16, 16, 100, 16, 101, 16, 16, 16, 8, 4, 0.1, 16, stream=0), 1),
    # stage 1 per request: per-row arrays required and 4-byte aligned, a keep count that fits every
    # row's window and sinks; pages a power of two in [8, 128] that cover the longest prompt
    (lambda: rkv.rkv_snap_evict_ragged(D4, 16, 32, 16, 16, 100, None, 100, 63, 0, 16, 50, 0.1, 16, 50, 16, 16, 50,
                                       None, 256, 1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict_ragged(D4, 16, 32, 16, 16, 100, 16, 100, 63, 4, 16, 36, 0.1, 16, 50, 16, 16, 50,
                                       None, 256, 1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict_ragged(D4, 16, 32, 16, 16, 100, 18, 100, 63, 0, 16, 50, 0.1, 16, 50, 16, 16, 50,
                                       None, 256, 1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict_paged(D4, 16, 32, 16, 16, 8, 64, None, 2, 16, 100, 63, 0, 16, 50, 0.1, 16, 50,
                                      16, 16, 50, None, 256, 1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict_paged(D4, 16, 32, 16, 16, 8, 48, 16, 4, 16, 100, 63, 0, 16, 50, 0.1, 16, 50,
                                      16, 16, 50, None, 256, 1 << 30, stream=0), 2),
    (lambda: rkv.rkv_snap_evict_paged(D4, 16, 32, 16, 16, 8, 256, 16, 1, 16, 100, 63, 0, 16, 50, 0.1, 16, 50,
                                      16, 16, 50, None, 256, 1 << 30, stream=0), 2),
    (lambda: rkv.rkv_snap_evict_paged(D4, 16, 32, 16, 16, 8, 64, 16, 1, 16, 100, 63, 0, 16, 50, 0.1, 16, 50,
                                      16, 16, 50, None, 256, 1 << 30, stream=0), 1),
    (lambda: rkv.rkv_snap_evict_paged(D4, 16, 32, 16, 16, 0, 64, 16, 2, 16, 100, 63, 0, 16, 50, 0.1, 16, 50,
                                      16, 16, 50, None, 256, 1 << 30, stream=0), 1),
    (lambda: rkv.rkv_build_kt(D4, 16, 10, 20, None, 0, 16, 16, 4, stream=0), 1),
    (lambda: rkv.rkv_build_kt(D4, 16, 100, 100, None, 0, 16, 16, 6, stream=0), 1),
    (lambda: rkv.rkv_append_kv(D4, 16, 16, 16, 16, 100, 10, 11, None, 0, 16, 10, 16, stream=0), 1),
    (lambda: rkv.rkv_append_kv(D4, 16, 16, 16, 16, 100, 160, 160, None, 0, 16, 10, 16, stream=0), 1),
    (lambda: rkv.rkv_append_kv(D4, 16, 16, 16, 16, 100, 10, 10, 16, 10, 16, 10, 16, stream=0), 1),
    # masked multi-turn: NULL / misaligned mask, n_prompt past n, mask rows too short
    (lambda: rkv.rkv_hsa_decode_mt_masked(D4, 16, 16, 16, 100, 90, None, 4, 80, 16, 16, 16, 8, 4, 0.1, 16,
                                          stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_mt_masked(D4, 16, 16, 16, 100, 90, 18, 4, 80, 16, 16, 16, 8, 4, 0.1, 16,
                                          stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_mt_masked(D4, 16, 16, 16, 100, 90, 16, 4, 91, 16, 16, 16, 8, 4, 0.1, 16,
                                          stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_mt_masked(D4, 16, 16, 16, 100, 90, 16, 2, 80, 16, 16, 16, 8, 4, 0.1, 16,
                                          stream=0), 1),
    (lambda: rkv.rkv_keep_mask(D4, None, 50, 50, 100, 16, 4, stream=0), 1),
    (lambda: rkv.rkv_keep_mask(D4, 16, 40, 50, 100, 16, 4, stream=0), 1),
    (lambda: rkv.rkv_keep_mask(D4, 16, 50, 50, 100, 16, 3, stream=0), 1),
    (lambda: rkv.rkv_build_kt_masked(D4, 16, 100, 90, None, 4, 80, 16, 16, 8, stream=0), 1),
    (lambda: rkv.rkv_build_kt_masked(D4, 16, 100, 90, 16, 4, 91, 16, 16, 8, stream=0), 1),
    (lambda: rkv.rkv_build_kt_masked(D4, 16, 100, 90, 16, 2, 80, 16, 16, 8, stream=0), 1),
    # e4m3 storage: NULL / misaligned scales, block size, KT stride
    (lambda: rkv.rkv_hsa_decode_fp8(D4, 16, 16, 16, 100, 90, None, 16, 16, 16, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_fp8(D4, 16, 16, 16, 100, 90, 18, 16, 16, 16, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_hsa_decode_fp8(D4, 16, 16, 16, 100, 90, 16, 16, 16, 16, 12, 8, 4, 0.1, 16, stream=0), 2),
    (lambda: rkv.rkv_hsa_decode_fp8(D4, 16, 16, 16, 100, 90, 16, 16, 16, 8, 16, 8, 4, 0.1, 16, stream=0), 1),
    (lambda: rkv.rkv_compact_kt_fp8(D4, 16, 16, 100, 16, 50, 50, None, 16, 16, 16, 50, 16, 16, 16, stream=0), 1),
    (lambda: rkv.rkv_compact_kt_fp8(D4, 16, 16, 100, 16, 50, 50, 16, 16, 16, 16, 50, 16, 16, 8, stream=0), 1),
    (lambda: rkv.rkv_compact_kt_fp8(D4, 16, 16, 100, 16, 50, 50, 16, 16, 16, 16, 40, 16, 16, 16, stream=0), 1),
])
def test_invalid_arguments_rejected_on_host(lib, call, status):
    # The calls pass made-up addresses that only the host checks may see; with
    # a GPU visible a missing check would hand them to a kernel, so they run on
    # GPU-less hosts only.
    if torch.cuda.is_available():
        pytest.skip("made-up device addresses are only passed on hosts without a GPU")
    with pytest.raises(rkv.RkvError) as e:
        call()
    assert e.value.status == status, str(e.value)
    assert lib.rkv_last_error()


def test_empty_batch_is_a_no_op(lib):
    d0 = (0, 32, 8, 128)
    rkv.rkv_hsa_decode(d0, None, None, None, 0, 0, None, 0, 16, 8, 4, 0.1, None, stream=0)
    rkv.rkv_build_kt(d0, None, 0, 0, None, 0, 16, None, 0, stream=0)
    rkv.rkv_compact_kt(d0, None, None, 0, None, 0, 0, None, None, 0, 16, None, 0, stream=0)
    rkv.rkv_append_kv(d0, None, None, None, None, 0, 0, 0, None, 0, None, 0, 16, stream=0)
    rkv.rkv_snap_evict(d0, None, 32, None, None, 0, 0, 63, 0, 0, 0.1, None, 0, None, None, 0, None, None, 0, stream=0)


def test_workspace_query(lib):
    assert rkv.rkv_snap_evict_workspace((8, 32, 8, 128), 32768, 32) > 8 * 8 * (32768 - 32) * 4
    assert rkv.rkv_snap_evict_workspace((8, 32, 8, 64), 32768, 32) == 0
