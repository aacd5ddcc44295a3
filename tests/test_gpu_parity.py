"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bits, at sizes the oracle finishes in seconds, then at the full
workload sizes, every row.  Tolerances are in ``parity.py``."""
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


def check(p, num_sms=0, **kw):
    out, lse, plan, status = run_gpu(p, num_sms=num_sms, **kw)
    ref_o, ref_l = oracle_full(p)
    stats = assert_close(out, lse, ref_o, ref_l, p.name)
    assert status == 0, f"device status {status:#x}"
    return out, lse, plan, stats


def test_tiny_config():
    check(syn.tiny())


@pytest.mark.parametrize("batch,ctx", [(1, 21), (3, 64), (2, 200), (3, 1200), (1, 2049), (2, 4160)])
def test_dense_h128(batch, ctx):
    check(syn.dense(batch, ctx, seed=batch * 1000 + ctx))


@pytest.mark.parametrize("ctx", [300, 4096])
def test_fp8_h16_ps64(ctx):
    check(syn.fp8_long(ctx, batch=2, seed=ctx))


@pytest.mark.parametrize("heads,sq", syn.MTP_SHAPES)
@pytest.mark.parametrize("ps", syn.MTP_PAGE_SIZES)
def test_mtp_causal(heads, sq, ps):
    check(syn.mtp(heads, sq, ps, batch=2, ctx=333, seed=heads * 10 + sq + ps))


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_ragged_small(kv_dtype):
    lens = syn.ragged_lens(6, hi=3000, seed=3)
    check(syn.make_problem(6, 1, 128, lens, 16, kv_dtype, False, seed=5, name="ragged_small"))


def test_mixed_page_sizes_and_rows():
    # H*Sq = 96 (not a power of two), odd page size, non-causal MTP.
    check(syn.make_problem(3, 3, 32, [77, 130, 5], 5, syn.KV_BF16, False, seed=9, name="odd"))
    # more than 128 rows: two row blocks
    check(syn.make_problem(2, 2, 128, [150, 64], 16, syn.KV_BF16, True, seed=10, name="rows256"))


def _growing_rope(kv_dtype, factors, batch=64, heads=128, seed=21):
    """The rope dims of tile i's keys (64 keys a tile) scaled by factors[i]:
    each of the early tiles lifts the row maxima by about 7 nats, more than
    the lazy-rescale threshold, so O is rescaled in several tiles while the
    MMAs of the tiles before may still be in flight.  The value dims stay
    N(0, 1), so the outputs keep their usual size; batch 64 fills the GPU."""
    ctx = 64 * len(factors)
    p = syn.make_problem(batch, 1, heads, [ctx] * batch, 1, syn.KV_BF16, False, seed=seed,
                         name=f"growing_rope_{kv_dtype}")
    x = syn.bf16_bits_to_f32(p.cache.reshape(-1, syn.D_QK)).copy()
    f = np.ones(x.shape[0], np.float32)
    for b in range(batch):
        f[p.block_table[b, :ctx]] = np.repeat(np.asarray(factors, np.float32), 64)
    x[:, syn.D_V:] *= f[:, None]
    if kv_dtype == syn.KV_BF16:
        p.cache = syn.f32_to_bf16_bits(x).reshape(p.cache.shape)
    else:
        scale = float(np.float32(np.abs(x).max() / syn.E4M3_MAX))
        p.cache = syn.f32_to_e4m3((x / np.float32(scale)).reshape(-1)).reshape(p.cache.shape)
        p.kv_dtype, p.kv_scale = kv_dtype, scale
    return p


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_rescale_while_earlier_pv_in_flight(kv_dtype):
    check(_growing_rope(kv_dtype, [0.2, 6.0, 12.0, 18.0, 24.0, 1.0, 1.0, 1.0]))


def test_split_count_invariance():
    p = syn.dense(2, 3000, seed=11)
    ref_o, ref_l = oracle_full(p)
    outs = []
    for num_sms in (2, 8, 16, 148, 4000):  # 1, 2, 4 and 24 splits
        out, lse, plan, _ = run_gpu(p, num_sms=num_sms)
        assert_close(out, lse, ref_o, ref_l, f"num_sms={num_sms} splits={plan.num_splits}")
        outs.append((plan.num_splits, out, lse))
    assert len({s for s, _, _ in outs}) >= 3
    for _, o, l in outs[1:]:
        assert_close(o, l, outs[0][1], outs[0][2], "split vs split")


@pytest.mark.parametrize("kv_dtype,heads,sq", [(syn.KV_FP8_E4M3, 16, 1), (syn.KV_BF16, 16, 4),
                                               (syn.KV_BF16, 64, 1)])
def test_split_count_invariance_few_rows(kv_dtype, heads, sq):
    """The 128-key-tile kernel (at most 64 rows bf16, 16 fp8) over 1 to many splits."""
    p = syn.make_problem(2, sq, heads, [3001, 2500], 16, kv_dtype, sq > 1, seed=41, name="few_rows")
    ref_o, ref_l = oracle_full(p)
    splits = set()
    for num_sms in (2, 8, 148, 4000):
        out, lse, plan, st = run_gpu(p, num_sms=num_sms)
        assert plan.key_tile == 128 and st == 0
        assert_close(out, lse, ref_o, ref_l, f"num_sms={num_sms} splits={plan.num_splits}")
        splits.add(plan.num_splits)
    assert len(splits) >= 3


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
@pytest.mark.parametrize("heads,sq", [(8, 2), (5, 3), (1, 1), (2, 8), (16, 1)])
def test_key_split_rows(kv_dtype, heads, sq):
    """At most 16 rows: the few-row kernel's key-split form, where the two
    warps of TMEM lane quarter 0 share every 128-key tile and trade row maxima
    and sums.  Causal masks across the query tokens, contexts with partial
    tiles and parts (129, 70, 31), one shorter than Sq, 1 to many splits, and
    outlier rows that make the running max jump."""
    p = syn.make_problem(4, sq, heads, [1000, 129, 70, max(sq - 1, 0)], 16, kv_dtype, sq > 1,
                         seed=50 + 7 * heads + sq, outlier_frac=0.02, name=f"key_split_h{heads}_sq{sq}")
    ref_o, ref_l = oracle_full(p)
    for num_sms in (2, 148, 4000):
        out, lse, plan, st = run_gpu(p, num_sms=num_sms)
        assert plan.key_tile == 128 and st == 0
        assert_close(out, lse, ref_o, ref_l, f"{p.name} splits={plan.num_splits}")


def _random_cases(n=24, seed=2026):
    """Seeded random shapes over both kernels and every few-row form: heads
    1..128, Sq 1..8 (rows up to 384, several 128-row blocks), page sizes
    1..128, bf16 / fp8, causal or not, ragged contexts with empty and
    shorter-than-Sq ones, sometimes outlier rows and poisoned slack."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        heads = int(rng.choice([1, 2, 3, 5, 8, 12, 16, 20, 32, 48, 64, 100, 128]))
        sq = int(rng.integers(1, 9)) if heads * 8 <= 384 else int(rng.integers(1, 384 // heads + 1))
        ps = int(rng.choice([1, 2, 3, 5, 16, 33, 64, 128]))
        batch = int(rng.integers(1, 4))
        lens = [int(x) for x in rng.integers(0, 1800, batch)]
        if rng.random() < 0.3:
            lens[0] = int(rng.integers(0, sq + 1))
        kv = syn.KV_FP8_E4M3 if rng.random() < 0.4 else syn.KV_BF16
        causal = bool(rng.random() < 0.6) and sq > 1
        cases.append((i, heads, sq, ps, lens, kv, causal, 0.02 if rng.random() < 0.5 else 0.0,
                      bool(rng.random() < 0.3)))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: f"case{c[0]}_h{c[1]}_sq{c[2]}_ps{c[3]}")
def test_random_shapes(case):
    i, heads, sq, ps, lens, kv, causal, outliers, poison = case
    p = syn.make_problem(len(lens), sq, heads, lens, ps, kv, causal, seed=300 + i,
                         outlier_frac=outliers, poison=poison, name=f"random{i}")
    check(p)
    if sum(lens) > 0:  # and with a forced split count
        check(p, num_sms=8)


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_rescale_while_earlier_pv_in_flight_few_rows(kv_dtype):
    p = _growing_rope(kv_dtype, [0.2, 0.2, 6.0, 6.0, 12.0, 12.0, 18.0, 18.0, 24.0, 24.0, 1.0, 1.0],
                      heads=16)
    check(p)


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_cuda_graph_replay_matches_eager(kv_dtype):
    """fwd + combine captured into one CUDA graph (the combine's programmatic
    dependent launch included) and replayed give the eager bits."""
    import torch
    p = syn.make_problem(3, 2, 64, [3000, 700, 1], 16, kv_dtype, True, seed=18, name="graph")
    t = to_device(p)
    plan = mla.plan(p.seq_lens, p.heads, p.sq, p.page_size, p.kv_dtype, p.causal, 148)
    assert plan.num_splits > 1  # the combine is part of the graph
    ws = mla.workspace_for(plan)
    eager_o, eager_l, _, status = run_gpu(p, t=t, plan=plan, workspace=ws)
    assert status == 0
    out = torch.full((p.batch, p.sq, p.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.batch, p.sq, p.heads), float("nan"), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        mla.fwd(plan, t["q"], t["cache"], t["scale"], t["bt"], t["lens"], p.softmax_scale, out, lse,
                ws, s)
        mla.combine(plan, t["lens"], out, lse, ws, s)
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert mla.check(plan, ws) == 0
        assert np.array_equal(out.double().cpu().numpy(), eager_o)
        assert np.array_equal(lse.double().cpu().numpy(), eager_l)
    ref_o, ref_l = oracle_full(p)
    assert_close(eager_o, eager_l, ref_o, ref_l, "graph")


@pytest.mark.parametrize("num_sms", [24, 148])
def test_splits_two_row_blocks_empty_sequence(num_sms):
    # 256 rows (two row blocks per sequence), causal, an empty sequence and one
    # shorter than a split, over several splits
    p = syn.make_problem(3, 2, 128, [700, 40, 0], 16, syn.KV_BF16, True, seed=19, name="splits")
    out, lse, plan, status = run_gpu(p, num_sms=num_sms)
    assert plan.num_splits > 1 and status == 0
    ref_o, ref_l = oracle_full(p)
    assert_close(out, lse, ref_o, ref_l, f"splits={plan.num_splits}")


def test_empty_and_short_contexts():
    p = syn.make_problem(4, 1, 128, [0, 70, 1, 0], 1, syn.KV_BF16, False, seed=12, name="empty")
    check(p)
    # causal with ctx < Sq: early tokens see no key at all
    check(syn.make_problem(3, 4, 16, [2, 4, 9], 4, syn.KV_BF16, True, seed=13, name="ctx<sq"))


def test_poisoned_slots_and_table_tail_are_never_read():
    for dt in (syn.KV_BF16, syn.KV_FP8_E4M3):
        p = syn.make_problem(3, 2, 64, [100, 37, 64], 16, dt, True, seed=14, poison=True,
                             extra_pages=5, name="poison")
        check(p)


def test_bad_page_id_sets_status_without_fault():
    p = syn.make_problem(2, 1, 16, [40, 40], 1, syn.KV_BF16, False, seed=15)
    p.block_table[1, 7] = 10 ** 6
    out, lse, plan, status = run_gpu(p)
    assert status & mla.DEVFLAG_BAD_PAGE
    # the sequence with a valid table is unaffected
    ref_o, ref_l = oracle_full(p, b_range=(0, 1))
    assert_close(out[:1], lse[:1], ref_o, ref_l, "valid sequence next to a bad one")


def test_context_beyond_plan_sets_status():
    import torch
    p = syn.make_problem(1, 1, 16, [256], 1, syn.KV_BF16, False, seed=16)
    t = to_device(p)
    plan = mla.plan([64], 16, 1, 1)  # plan covers 64 keys, device says 256
    out, lse, _, status = run_gpu(p, t=t, plan=plan)
    assert status & mla.DEVFLAG_CTX_RANGE
    torch.cuda.synchronize()


@pytest.mark.parametrize("num_sms", [8, 148])
@pytest.mark.parametrize("which", [0, 2])
def test_context_between_max_ctx_and_split_cover(which, num_sms):
    """A device context in (max_ctx, num_splits * chunk_len]: the splits would
    cover it, but the block table is only ceil(max_ctx / page_size) wide, so
    the kernel must flag it and clamp it to max_ctx (on a sequence in the
    middle, and on the last one, whose table ends the allocation).  A negative
    context is flagged and read as empty."""
    import torch
    lens = [1000, 700, 1000]
    p = syn.make_problem(3, 1, 16, lens, 1, syn.KV_BF16, False, seed=16, name="ctx_range")
    assert p.block_table.shape[1] == 1000
    t = to_device(p)
    plan = mla.plan(lens, 16, 1, 1, num_sms=num_sms)  # 1 split, or 16 of 64 keys
    assert plan.max_ctx == 1000 and plan.num_splits * plan.chunk_len >= 1020
    dev = list(lens)
    dev[which] = 1020
    dev[1 if which == 0 else 0] = -5
    t["lens"] = torch.tensor(dev, dtype=torch.int32, device="cuda")
    out, lse, _, status = run_gpu(p, t=t, plan=plan)
    assert status & mla.DEVFLAG_CTX_RANGE
    # what the kernel reads: the clamped contexts
    q = syn.make_problem(3, 1, 16, lens, 1, syn.KV_BF16, False, seed=16)
    q.seq_lens = np.clip(np.asarray(dev, np.int32), 0, 1000).astype(np.int32)
    ref_o, ref_l = oracle_full(q)
    assert_close(out, lse, ref_o, ref_l, "clamped contexts")


@pytest.mark.parametrize("form", ["128_rows_bf16", "128_rows_fp8", "few_rows_fp8", "few_rows_wide_bf16", "few_rows_narrow_bf16"])
def test_wait_limit_runs_out_without_fault(form):
    """With a 1 us bound every long wait of the pipeline gives up: the call
    reports MLA_ERR_TIMEOUT through the status word, no fault, and the next
    call with the default bound on the same workspace is correct.  For the
    128-row kernels (bf16 and fp8 caches) and each form of the few-row kernel (its key-split
    exchanges and part pipelines included)."""
    import ctypes
    import torch
    p = {"128_rows_bf16": lambda: syn.dense(16, 4096, seed=40),
         "128_rows_fp8": lambda: syn.make_problem(16, 1, 128, [4096] * 16, 1, syn.KV_FP8_E4M3, False,
                                                  seed=46, name="dense_h128_b16_ctx4096_fp8"),
         "few_rows_fp8": lambda: syn.fp8_long(4096, batch=4, seed=41),
         "few_rows_wide_bf16": lambda: syn.mtp(16, 4, 64, batch=4, ctx=4096, seed=42),
         "few_rows_narrow_bf16": lambda: syn.mtp(8, 2, 16, batch=4, ctx=4096, seed=43)}[form]()
    t = to_device(p)
    plan = mla.plan(p.seq_lens, p.heads, p.sq, p.page_size, p.kv_dtype, p.causal)
    ws = mla.workspace_for(plan)
    short = mla.Plan.from_buffer_copy(plan)
    short.wait_limit_us = 1
    out = torch.full((p.batch, p.sq, p.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.batch, p.sq, p.heads), float("nan"), dtype=torch.float32, device="cuda")
    mla.fwd(short, t["q"], t["cache"], t["scale"], t["bt"], t["lens"], p.softmax_scale, out, lse, ws)
    mla.combine(short, t["lens"], out, lse, ws)
    v = ctypes.c_int32(0)
    st = mla.lib().mla_decode_check(ctypes.byref(short), ctypes.c_void_p(ws.data_ptr()),
                                    mla._stream(None), ctypes.byref(v))
    assert st == mla.ERR_TIMEOUT and (v.value & mla.DEVFLAG_TIMEOUT), (st, v.value)
    torch.cuda.synchronize()
    out2, lse2, _, status = run_gpu(p, t=t, plan=plan, workspace=ws)
    assert status == 0
    ref_o, ref_l = oracle_full(p)
    assert_close(out2, lse2, ref_o, ref_l, "after a timed-out call")


@pytest.mark.parametrize("heads", [16, 128])
def test_fp8_query_range_edges(heads):
    """With an fp8 cache the kernels stage q as f16: q scaled by 2^-10 (many
    elements in f16's subnormal range) still meets the tolerance, and one
    element past 65504 sets MLA_DEVFLAG_Q_RANGE."""
    p = syn.make_problem(2, 1, heads, [700, 130], 16, syn.KV_FP8_E4M3, False, seed=44,
                         name="q_small")
    x = syn.bf16_bits_to_f32(p.q_bits) * np.float32(2.0 ** -10)
    p.q_bits = syn.f32_to_bf16_bits(x)
    check(p)
    big = syn.make_problem(1, 1, heads, [300], 16, syn.KV_FP8_E4M3, False, seed=45, name="q_big")
    big.q_bits[0, 0, 3, 17] = syn.f32_to_bf16_bits(np.array([70000.0], np.float32))[0]
    _, _, _, status = run_gpu(big)
    assert status & mla.DEVFLAG_Q_RANGE


def test_run_to_run_determinism():
    p = syn.dense(2, 1500, seed=17)
    t = to_device(p)
    a = run_gpu(p, t=t, num_sms=148)
    b = run_gpu(p, t=t, num_sms=148)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- full workload sizes, every row against the oracle ----

def full_check(p, num_sms=0):
    out, lse, plan, status = run_gpu(p, num_sms=num_sms)
    assert status == 0
    ref_o, ref_l = oracle_full(p)
    assert_close(out, lse, ref_o, ref_l, f"{p.name} splits={plan.num_splits}")
    return plan


def test_full_dense_b64_ctx8192():
    full_check(syn.dense(64, 8192))


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_full_ragged_b64(kv_dtype):
    full_check(syn.ragged(kv_dtype))


def test_full_fp8_long_ctx109440():
    full_check(syn.fp8_long(109440))


@pytest.mark.parametrize("heads,sq,ps", [(16, 8, 64), (64, 2, 1), (32, 4, 16), (16, 4, 64)])
def test_full_mtp_causal(heads, sq, ps):
    full_check(syn.mtp(heads, sq, ps))


@pytest.mark.parametrize("heads,sq,ps", [(16, 1, 64), (8, 2, 16)])
def test_full_mtp_recipe_key_split(heads, sq, ps):
    """The MTP recipe (causal, outlier rows) at 16 rows: the key-split form
    with a bf16 cache at full size."""
    full_check(syn.mtp(heads, sq, ps))


@pytest.mark.parametrize("ctx", [8192, 23333])
def test_full_dense_batch1_many_splits(ctx):
    plan = full_check(syn.dense(1, ctx, seed=ctx))
    assert plan.num_splits >= 48, plan.num_splits


def test_full_dense_b256_ctx8192():
    full_check(syn.dense(256, 8192, seed=256))
