"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol the header declares, and the planner's partition is sound."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import mla_synth as syn
import paged_mla_decode_latent_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mla.build()
    return mla.lib()


def header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = header_functions()
    for n in ("mla_decode_plan", "mla_decode_fwd", "mla_decode_combine"):
        assert n in names
    assert set(names) == set(mla.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for n in header_functions():
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", mla.LIB_PATH], capture_output=True,
                         text=True).stdout
    for n in header_functions():
        assert re.search(rf"\bT {n}\b", out), n


def test_plan_struct_layout_matches_header():
    assert ctypes.sizeof(mla.Plan) == 20 * 4 + 4 * 8
    assert mla.Plan.ws_partial_o_offset.offset == 80


def test_status_strings(L):
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert mla.status_string(st) and mla.status_string(st) != "unknown status"
    assert mla.status_string(12345) == "unknown status"


def check_plan_invariants(p, lens):
    lens = np.asarray(lens)
    assert p.chunk_len % p.key_tile == 0 and p.chunk_len >= p.key_tile
    assert p.num_splits == max(1, -(-int(lens.max()) // p.chunk_len))
    assert p.num_splits * p.chunk_len >= lens.max()
    assert (p.num_splits - 1) * p.chunk_len < max(1, lens.max())
    assert p.rows == p.num_heads * p.sq and p.row_blocks == -(-p.rows // 128)
    assert (p.grid_x, p.grid_y, p.grid_z) == (2 * p.row_blocks, len(lens), p.num_splits)
    assert p.ws_status_offset % 256 == 0 and p.workspace_bytes % 256 == 0
    if p.num_splits > 1:
        o_bytes = len(lens) * p.num_splits * p.rows * 512 * 4
        l_bytes = len(lens) * p.num_splits * p.rows * 4
        assert p.ws_partial_o_offset == 0 and p.ws_partial_lse_offset >= o_bytes
        assert p.ws_status_offset >= p.ws_partial_lse_offset + l_bytes
    assert p.workspace_bytes >= p.ws_status_offset + 4


@pytest.mark.parametrize("lens,h,sq,ps,dt,causal", [
    ([64], 16, 1, 1, 0, False),
    ([8192] * 64, 128, 1, 1, 0, False),
    ([23333], 128, 1, 1, 0, False),
    ([4096] * 8, 16, 1, 64, 1, False),
    ([109440] * 8, 16, 1, 64, 1, False),
    ([8192] * 32, 64, 2, 16, 0, True),
    ([8192] * 32, 16, 8, 64, 0, True),
    (list(syn.ragged_lens(64)), 128, 1, 16, 0, False),
    (list(syn.ragged_lens(64)), 128, 1, 16, 1, False),
    ([0, 5, 0], 128, 1, 1, 0, False),
    ([0], 16, 1, 1, 0, False),
])
def test_plan_partition(L, lens, h, sq, ps, dt, causal):
    p = mla.plan(lens, h, sq, ps, dt, causal, num_sms=148)
    check_plan_invariants(p, lens)


def test_plan_uses_device_free_sm_count(L):
    a = mla.plan([1 << 16], 128, 1, 1, num_sms=148)
    b = mla.plan([1 << 16], 128, 1, 1, num_sms=8)
    assert a.num_splits >= b.num_splits


def test_plan_splits_a_single_long_sequence(L):
    # One long sequence on 148 SMs must be split across many pairs.
    p = mla.plan([23333], 128, 1, 1, num_sms=148)
    assert p.num_splits > 8


@pytest.mark.parametrize("args", [
    dict(lens=[10], h=0), dict(lens=[10], h=129), dict(lens=[10], sq=0), dict(lens=[10], sq=17),
    dict(lens=[10], ps=0), dict(lens=[10], dt=2), dict(lens=[-1]), dict(lens=[10], causal=2),
    dict(lens=[10], h=128, sq=9),
])
def test_plan_rejects_bad_arguments(L, args):
    a = dict(lens=[10], h=16, sq=1, ps=1, dt=0, causal=0)
    a.update(args)
    lens = np.asarray(a["lens"], np.int32)
    p = mla.Plan()
    st = L.mla_decode_plan(lens.ctypes.data, len(lens), a["h"], a["sq"], a["ps"], a["dt"],
                           a["causal"], 148, ctypes.byref(p))
    assert st == mla.ERR_INVALID_ARG


def test_fwd_rejects_bad_arguments_before_touching_the_gpu(L):
    p = mla.plan([64], 16, 1, 1, num_sms=148)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    args = [ctypes.byref(p), fake, fake, 64, None, fake, 64, fake, 0.1, fake, fake]
    # null workspace
    assert L.mla_decode_fwd(*args, None, 1 << 20, None) == mla.ERR_WORKSPACE
    # misaligned workspace
    assert L.mla_decode_fwd(*args, ctypes.c_void_p((1 << 20) + 8), 1 << 20, None) == mla.ERR_WORKSPACE
    # too small
    assert L.mla_decode_fwd(*args, fake, 8, None) == mla.ERR_WORKSPACE
    # null q
    bad = list(args)
    bad[1] = None
    assert L.mla_decode_fwd(*bad, fake, 1 << 20, None) == mla.ERR_INVALID_ARG
    # block table too narrow for the plan's longest context
    bad = list(args)
    bad[6] = 8
    assert L.mla_decode_fwd(*bad, fake, 1 << 20, None) == mla.ERR_INVALID_ARG
    # wrong plan version
    q = mla.Plan.from_buffer_copy(p)
    q.version = 99
    bad = list(args)
    bad[0] = ctypes.byref(q)
    assert L.mla_decode_fwd(*bad, fake, 1 << 20, None) == mla.ERR_INVALID_ARG


def test_epilogue_rejects_bad_arguments_before_touching_the_gpu(L):
    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced
    ok = [fake, fake, fake, fake, fake, 4, 8, fake, fake, 4, 16, 0, None, 0, None, None]
    for i, bad in [(0, None), (4, None), (7, None), (8, None), (6, 0), (6, 129), (10, 0),
                   (11, 2), (13, 2), (1, ctypes.c_void_p((1 << 20) + 8))]:
        a = list(ok)
        a[i] = bad
        assert L.mla_decode_epilogue(*a) == mla.ERR_INVALID_ARG, i
    a = list(ok)
    a[11] = mla.KV_FP8_E4M3  # fp8 cache needs kv_scale
    assert L.mla_decode_epilogue(*a) == mla.ERR_INVALID_ARG
    a = list(ok)
    a[5] = 0  # no tokens: nothing to queue
    assert L.mla_decode_epilogue(*a) == mla.OK


@pytest.mark.parametrize("b,h,sq,ps,cap,sms", [(64, 128, 1, 1, 8192, 152), (1, 16, 1, 64, 131072, 148),
                                              (1024, 64, 2, 16, 4096, 152), (3, 128, 2, 1, 100, 8)])
def test_dplan_info_sizes(L, b, h, sq, ps, cap, sms):
    d = mla.dplan_info(b, h, sq, ps, 0, sq > 1, cap, sms)
    rb = -(-(h * sq) // 128)
    assert d.rows == h * sq and d.row_blocks == rb
    assert d.pairs == min(sms // 2, 127) and d.max_parts == 2 * d.pairs + b
    assert d.max_units == rb * d.max_parts
    offs = [d.ws_units_offset, d.ws_seq_offset, d.ws_count_offset, d.ws_partial_o_offset,
            d.ws_partial_lse_offset, d.ws_status_offset]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert d.ws_seq_offset >= d.ws_units_offset + 16 * d.max_units
    assert d.ws_partial_lse_offset >= d.ws_partial_o_offset + 4 * d.max_parts * d.rows * 512
    assert d.workspace_bytes >= d.ws_status_offset + 4


def test_dplan_rejects_bad_arguments(L):
    d = mla.DPlan()
    for args in [(0, 16, 1, 1, 0, 0, 64, 152), (1025, 16, 1, 1, 0, 0, 64, 152),
                 (1, 0, 1, 1, 0, 0, 64, 152), (1, 16, 1, 1, 2, 0, 64, 152),
                 (1, 16, 1, 1, 0, 0, -1, 152)]:
        assert L.mla_decode_dplan_info(*args, ctypes.byref(d)) == mla.ERR_INVALID_ARG
    good = mla.dplan_info(2, 16, 1, 1, 0, False, 64, 152)
    fake = ctypes.c_void_p(1 << 20)
    # no workspace / too small / wrong version
    assert L.mla_decode_plan_device(ctypes.byref(good), fake, None, None, 1 << 30, None) == mla.ERR_WORKSPACE
    assert L.mla_decode_plan_device(ctypes.byref(good), fake, None, fake, 16, None) == mla.ERR_WORKSPACE
    bad = mla.DPlan.from_buffer_copy(good)
    bad.version = 7
    assert L.mla_decode_plan_device(ctypes.byref(bad), fake, None, fake, 1 << 30, None) == mla.ERR_INVALID_ARG
    # padded table narrower than the capacity
    assert L.mla_decode_fwd_dplan(ctypes.byref(good), fake, fake, 8, None, fake, 32, None, 0.1, fake,
                                  fake, fake, 1 << 30, None) == mla.ERR_INVALID_ARG
