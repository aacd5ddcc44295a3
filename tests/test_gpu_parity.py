"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bits, at sizes the oracle finishes in seconds, then at the full
workload sizes on sampled rows.  Tolerances are in ``parity.py``."""
import numpy as np
import pytest

import mla_synth as syn
import oracle
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


def test_run_to_run_determinism():
    p = syn.dense(2, 1500, seed=17)
    t = to_device(p)
    a = run_gpu(p, t=t, num_sms=148)
    b = run_gpu(p, t=t, num_sms=148)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- full workload sizes, sampled rows checked one by one against the oracle ----

def sampled_check(p, n_rows=12, seed=0):
    out, lse, plan, status = run_gpu(p)
    assert status == 0
    g = np.random.default_rng(seed)
    for _ in range(n_rows):
        b = int(g.integers(p.batch))
        i = int(g.integers(p.sq))
        h = int(g.integers(p.heads))
        ro, rl = oracle.decode_row(p.q_bits, p.cache, p.kv_dtype, p.kv_scale, p.page_size,
                                   p.block_table, p.seq_lens, p.softmax_scale, p.causal, b, i, h)
        assert_close(out[b, i, h][None], lse[b, i, h][None], ro[None], np.array([rl]),
                     f"{p.name} row (b={b}, i={i}, h={h})")
    assert np.all(np.isfinite(out))
    return plan


def test_full_dense_b64_ctx8192_sampled():
    sampled_check(syn.dense(64, 8192))


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_full_ragged_b64_sampled(kv_dtype):
    sampled_check(syn.ragged(kv_dtype))


def test_full_fp8_long_ctx109440_sampled():
    sampled_check(syn.fp8_long(109440), n_rows=6)


def test_full_mtp_causal_sampled():
    sampled_check(syn.mtp(16, 8, 64), n_rows=8)


def test_full_mtp_h64_sq2_ps1_sampled():
    sampled_check(syn.mtp(64, 2, 1), n_rows=8)
