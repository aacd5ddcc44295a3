"""GPU parity of the decode epilogue (q-concat + paged latent-row insert
through slot_mapping) and of the chained decode step (epilogue -> decode ->
merge, programmatic dependent launches), through the C ABI, against the
oracle on the same bits.  q rows and cache bytes are compared bit for bit
(they are copies and fp8 codes); the decode after the insert within the
tolerances of ``parity.py``."""
import numpy as np
import pytest

import mla_synth as syn
import oracle
import paged_mla_decode_latent_gb300 as mla
from parity import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def _bits(seed, shape, sigma=1.0):
    g = np.random.default_rng(seed)
    return syn.f32_to_bf16_bits(g.standard_normal(shape).astype(np.float32) * np.float32(sigma))


def _t16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def run_epilogue(ql, qp, kc, kp, slots, cache, kv_dtype, scale, early, status=None):
    import torch
    T, H, _ = ql.shape
    q_out = torch.zeros((T, H, 576), dtype=torch.bfloat16, device="cuda")
    if kv_dtype == syn.KV_BF16:
        c = torch.from_numpy(cache.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        c = torch.from_numpy(cache).cuda()
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    mla.epilogue(_t16(ql), _t16(qp), _t16(kc), _t16(kp), torch.from_numpy(slots).cuda(), q_out, c,
                 sc, cache_inputs_early=early, status=status)
    torch.cuda.synchronize()
    q_bits = q_out.view(torch.int16).cpu().numpy().view(np.uint16)
    c_bits = (c.view(torch.int16).cpu().numpy().view(np.uint16) if kv_dtype == syn.KV_BF16
              else c.cpu().numpy())
    return q_bits, c_bits


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
@pytest.mark.parametrize("T,H,ps", [(1, 8, 1), (64, 16, 16), (65, 16, 64), (200, 128, 16)])
@pytest.mark.parametrize("early", [0, 1])
def test_epilogue_bit_exact(kv_dtype, T, H, ps, early):
    g = np.random.default_rng(T * 7 + H + ps + early)
    pages = -(-2 * T // ps) + 2
    ql, qp = _bits(1 + T, (T, H, 512)), _bits(2 + T, (T, H, 64))
    kc, kp = _bits(3 + T, (T, 512), 3.0), _bits(4 + T, (T, 64), 3.0)
    kc[0, :4] = syn.f32_to_bf16_bits(np.array([0.0, -0.0, 1e-6, -1e-6], np.float32))
    kc[0, 4:8] = syn.f32_to_bf16_bits(np.array([900.0, -900.0, 5.3, -5.3], np.float32))
    slots = g.choice(pages * ps, size=T, replace=False).astype(np.int64)
    if T > 1:
        slots[g.choice(T, size=max(1, T // 10), replace=False)] = -1
    if kv_dtype == syn.KV_BF16:
        cache = _bits(5 + T, (pages, ps, 576))
        scale = 1.0
    else:
        cache = g.integers(0, 0x7F, (pages, ps, 576)).astype(np.uint8)
        scale = 0.0123
    q_gpu, c_gpu = run_epilogue(ql, qp, kc, kp, slots, cache, kv_dtype, scale, early)
    q_ref, c_ref = oracle.epilogue(ql, qp, kc, kp, slots, cache, kv_dtype, scale)
    assert np.array_equal(q_gpu, q_ref)
    assert np.array_equal(c_gpu, c_ref)


def test_epilogue_slot_beyond_cache_is_flagged_and_skipped():
    import torch
    T, H, ps, pages = 4, 8, 16, 2
    ql, qp = _bits(11, (T, H, 512)), _bits(12, (T, H, 64))
    kc, kp = _bits(13, (T, 512)), _bits(14, (T, 64))
    slots = np.array([3, pages * ps, 5, -1], np.int64)
    cache = _bits(15, (pages, ps, 576))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, c_gpu = run_epilogue(ql, qp, kc, kp, slots, cache, syn.KV_BF16, 1.0, 0, status)
    assert int(status.item()) & mla.DEVFLAG_BAD_PAGE
    ok = slots.copy()
    ok[1] = -1
    _, c_ref = oracle.epilogue(ql, qp, kc, kp, ok, cache, syn.KV_BF16, 1.0)
    assert np.array_equal(c_gpu, c_ref)


def _step_problem(kv_dtype, heads, sq, ps, lens, causal, seed):
    """A decode problem whose last Sq keys of every sequence are the new
    tokens: the epilogue inserts them (their slots come from the sequence's
    block table) and writes q from its two halves."""
    p = syn.make_problem(len(lens), sq, heads, lens, ps, kv_dtype, causal, seed=seed,
                         name=f"step_{kv_dtype}_{heads}x{sq}_ps{ps}")
    T = p.batch * sq
    ql = np.ascontiguousarray(p.q_bits[..., :512].reshape(T, heads, 512))
    qp = np.ascontiguousarray(p.q_bits[..., 512:].reshape(T, heads, 64))
    kc, kp = _bits(seed + 100, (T, 512)), _bits(seed + 101, (T, 64))
    slots = np.empty(T, np.int64)
    for b in range(p.batch):
        for i in range(sq):
            j = int(p.seq_lens[b]) - sq + i
            slots[b * sq + i] = int(p.block_table[b, j // ps]) * ps + j % ps
    return p, ql, qp, kc, kp, slots


def _run_step(p, ql, qp, kc, kp, slots, plan, ws, t=None, graph=False):
    import torch
    t = t or to_device(p)
    q = torch.zeros_like(t["q"])
    out = torch.full((p.batch, p.sq, p.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.batch, p.sq, p.heads), float("nan"), dtype=torch.float32, device="cuda")
    args = (plan, _t16(ql), _t16(qp), _t16(kc), _t16(kp), torch.from_numpy(slots).cuda(), q,
            t["cache"], t["scale"], t["bt"], t["lens"], p.softmax_scale, out, lse, ws)
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            mla.step(*args, stream=torch.cuda.current_stream())
        g.replay()
    else:
        mla.step(*args)
    torch.cuda.synchronize()
    st = mla.check(plan, ws)
    cache = (t["cache"].view(torch.int16).cpu().numpy().view(np.uint16)
             if p.kv_dtype == syn.KV_BF16 else t["cache"].cpu().numpy())
    return (q.view(torch.int16).cpu().numpy().view(np.uint16), cache,
            out.double().cpu().numpy(), lse.double().cpu().numpy(), st)


@pytest.mark.parametrize("kv_dtype,heads,sq,ps,lens,causal", [
    (syn.KV_BF16, 128, 1, 1, [300, 2000, 5], False),
    (syn.KV_BF16, 32, 4, 16, [700, 64, 4000], True),
    (syn.KV_FP8_E4M3, 16, 1, 64, [3000, 129], False),
    (syn.KV_FP8_E4M3, 64, 2, 16, [900, 2], True),
])
def test_step_matches_oracle(kv_dtype, heads, sq, ps, lens, causal):
    p, ql, qp, kc, kp, slots = _step_problem(kv_dtype, heads, sq, ps, lens, causal, seed=50 + sq)
    plan = mla.plan(p.seq_lens, heads, sq, ps, kv_dtype, causal)
    ws = mla.workspace_for(plan)
    q, cache, out, lse, st = _run_step(p, ql, qp, kc, kp, slots, plan, ws)
    assert st == 0
    q_ref, c_ref = oracle.epilogue(ql, qp, kc, kp, slots, p.cache, kv_dtype, p.kv_scale)
    assert np.array_equal(q, q_ref.reshape(q.shape))
    assert np.array_equal(cache, c_ref)
    ref_o, ref_l = oracle.decode(q_ref.reshape(p.q_bits.shape), c_ref, kv_dtype, p.kv_scale, ps,
                                 p.block_table, p.seq_lens, p.softmax_scale, causal)
    assert_close(out, lse, ref_o, ref_l, p.name)


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_step_graph_replay_matches_eager(kv_dtype):
    p, ql, qp, kc, kp, slots = _step_problem(kv_dtype, 64, 2, 16, [2500, 300, 40], True, seed=60)
    plan = mla.plan(p.seq_lens, 64, 2, 16, kv_dtype, True, 148)
    assert plan.num_splits > 1
    ws = mla.workspace_for(plan)
    eager = _run_step(p, ql, qp, kc, kp, slots, plan, ws)
    replay = _run_step(p, ql, qp, kc, kp, slots, plan, ws, graph=True)
    assert eager[4] == 0 and replay[4] == 0
    for a, b in zip(eager[:4], replay[:4]):
        assert np.array_equal(a, b)
