"""The decode entry point that allocates nothing (mla_decode_fwd_noalloc).

Some callers cannot allocate device memory: a plugin whose host server owns
every device allocation through its own pool, or a latency-critical loop that
must not call cudaMalloc / cudaFree (they can synchronise the device).  They
call mla_decode_fwd_noalloc with inputs and outputs only; the library takes
its scratch from a fixed 64 MiB device array of its own.  This file checks,
through the C ABI, that two calls in a row give what mla_decode_fwd +
mla_decode_combine give with a caller-owned workspace, bit for bit (the same
plan and kernels run; only the workspace differs), after the scratch was left
holding another plan's partials, and that the result meets the parity
tolerance against the oracle.  It is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import mla_synth as syn
import paged_mla_decode_latent_gb300 as mla
from parity import assert_close, oracle_full, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def call_noalloc(p, t, plan):
    import torch
    L = mla.lib()
    out = torch.full((p.batch, p.sq, p.heads, 512), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((p.batch, p.sq, p.heads), float("nan"), dtype=torch.float32, device="cuda")
    st = L.mla_decode_fwd_noalloc(
        ctypes.byref(plan), ctypes.c_void_p(t["q"].data_ptr()),
        ctypes.c_void_p(t["cache"].data_ptr()), int(t["cache"].shape[0]),
        ctypes.c_void_p(t["scale"].data_ptr()), ctypes.c_void_p(t["bt"].data_ptr()),
        int(t["bt"].stride(0)), ctypes.c_void_p(t["lens"].data_ptr()),
        ctypes.c_float(p.softmax_scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mla.OK, mla.status_string(st)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_noalloc_matches_workspace_entry_point_twice(kv_dtype):
    p = syn.make_problem(3, 1, 128, [3000, 700, 1], 16, kv_dtype, False, seed=21,
                         name="noalloc")
    t = to_device(p)
    plan = mla.plan(p.seq_lens, p.heads, p.sq, p.page_size, p.kv_dtype, p.causal, 148)
    assert plan.num_splits > 1  # the scratch holds split partials
    ref_o, ref_l, _, status = run_gpu(p, t=t, plan=plan)
    assert status == 0
    # Leave other contents in the scratch first: a different batch and split
    # count, so stale partials of another plan sit where this plan reads.
    other = syn.make_problem(2, 2, 64, [5000, 900], 16, kv_dtype, True, seed=22, name="other")
    ot = to_device(other)
    oplan = mla.plan(other.seq_lens, other.heads, other.sq, other.page_size, other.kv_dtype,
                     other.causal, 148)
    assert oplan.num_splits != plan.num_splits
    call_noalloc(other, ot, oplan)
    # Same plan and kernels as the workspace entry point: the same bits.
    for _ in range(2):  # the scratch keeps the previous call's contents
        out, lse = call_noalloc(p, t, plan)
        assert np.array_equal(out, ref_o), "noalloc output differs from the workspace entry point"
        assert np.array_equal(lse, ref_l), "noalloc lse differs from the workspace entry point"
    ref = oracle_full(p)
    assert_close(out, lse, *ref, "noalloc vs oracle")


def test_noalloc_rejects_plans_beyond_its_scratch():
    big = mla.plan([131072] * 64, 128, 1, 16, syn.KV_BF16, False, 148)
    assert big.workspace_bytes > 64 << 20
    L = mla.lib()
    st = L.mla_decode_fwd_noalloc(ctypes.byref(big), None, None, 1, None, None, 1, None,
                                  ctypes.c_float(0.1), None, None, None)
    assert st == mla.ERR_WORKSPACE
