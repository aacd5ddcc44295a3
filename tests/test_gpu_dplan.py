"""GPU parity of the device-planned decode (mla_decode_dplan_info ->
mla_decode_plan_device -> mla_decode_fwd_dplan -> mla_decode_combine_dplan),
through the C ABI, against the oracle: padded and CSR page tables, the
device-written unit list's coverage, and a CUDA graph captured once and
replayed while the context lengths grow past what they were at capture."""
import numpy as np
import pytest

import mla_synth as syn
import oracle
import paged_mla_decode_latent_gb300 as mla
from parity import assert_close, oracle_full, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def csr_of(p):
    """kv_indptr / kv_indices of a problem's block table (each sequence's pages)."""
    n = [-(-int(c) // p.page_size) for c in p.seq_lens]
    indptr = np.zeros(p.batch + 1, np.int32)
    indptr[1:] = np.cumsum(n)
    idx = np.concatenate([p.block_table[b, :n[b]] for b in range(p.batch)] + [np.zeros(1, np.int32)])
    return indptr, idx.astype(np.int32)


def run_dplan(p, d, t=None, ws=None, csr=False, lens=None):
    import torch
    t = t or to_device(p)
    ws = ws if ws is not None else torch.empty(int(d.workspace_bytes), dtype=torch.uint8, device="cuda")
    out = torch.full((p.batch, p.sq, p.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.batch, p.sq, p.heads), float("nan"), dtype=torch.float32, device="cuda")
    lens_d = t["lens"] if lens is None else lens
    if csr:
        indptr, idx = csr_of(p)
        ip, ix = torch.from_numpy(indptr).cuda(), torch.from_numpy(idx).cuda()
        mla.plan_device(d, lens_d, ws, kv_indptr=ip)
        mla.fwd_dplan(d, t["q"], t["cache"], t["scale"], ix, p.softmax_scale, out, lse, ws,
                      kv_indptr=ip)
    else:
        mla.plan_device(d, lens_d, ws)
        mla.fwd_dplan(d, t["q"], t["cache"], t["scale"], t["bt"], p.softmax_scale, out, lse, ws)
    mla.combine_dplan(d, out, lse, ws)
    st = mla.dplan_check(d, ws)
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), st, ws


def info_for(p, capacity=None, num_sms=0):
    cap = int(capacity if capacity is not None else p.block_table.shape[1] * p.page_size)
    return mla.dplan_info(p.batch, p.heads, p.sq, p.page_size, p.kv_dtype, p.causal, cap, num_sms)


def unit_list(d, ws):
    import torch
    torch.cuda.synchronize()
    raw = ws.cpu().numpy()
    counts = raw[d.ws_count_offset:d.ws_count_offset + 16].view(np.int32)
    units = raw[d.ws_units_offset:d.ws_units_offset + 16 * d.max_units].view(np.int32).reshape(-1, 4)
    seq = raw[d.ws_seq_offset:d.ws_seq_offset + 16 * d.batch].view(np.int32).reshape(-1, 4)
    return counts, units[:counts[0]], seq


CASES = [
    ("ragged_bf16", lambda: syn.make_problem(6, 1, 128, syn.ragged_lens(6, hi=9000, seed=4), 16,
                                             syn.KV_BF16, False, seed=31, name="ragged_bf16")),
    ("ragged_fp8", lambda: syn.make_problem(6, 1, 128, syn.ragged_lens(6, hi=9000, seed=5), 16,
                                            syn.KV_FP8_E4M3, False, seed=32, name="ragged_fp8")),
    ("mtp_empty", lambda: syn.make_problem(4, 4, 16, [3000, 0, 2, 700], 16, syn.KV_BF16, True,
                                           seed=33, name="mtp_empty")),
    ("rows256", lambda: syn.make_problem(3, 2, 128, [1500, 64, 9], 1, syn.KV_BF16, True, seed=34,
                                         name="rows256")),
    ("b1_long", lambda: syn.dense(1, 23333, seed=35)),
    ("dense_b3", lambda: syn.dense(3, 1200, seed=36)),
    ("fp8_h16", lambda: syn.fp8_long(20000, batch=3, seed=37)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("csr", [False, True])
def test_dplan_matches_oracle(name, make, csr):
    p = make()
    d = info_for(p)
    out, lse, st, ws = run_dplan(p, d, csr=csr)
    assert st == 0, hex(st)
    ref_o, ref_l = oracle_full(p)
    assert_close(out, lse, ref_o, ref_l, f"{name} csr={csr}")
    # the unit list covers every sequence's keys once per row block
    counts, units, seq = unit_list(d, ws)
    assert 0 < counts[0] <= d.max_units and counts[2] <= d.max_parts
    for b in range(p.batch):
        ctx, part0, n, _ = seq[b]
        assert ctx == p.seq_lens[b] and n >= 1
        mine = units[units[:, 0] == b]
        for rb in range(d.row_blocks):
            r = mine[(mine[:, 1] & 0xFF) == rb]
            r = r[np.argsort(r[:, 2])]
            assert len(r) == n and r[0, 2] == 0 and r[-1, 3] == ctx
            assert np.all(r[1:, 2] == r[:-1, 3])
            assert sorted((r[:, 1] >> 8).tolist()) == list(range(n))
    cut = [(seq[b, 1], seq[b, 2]) for b in range(p.batch) if seq[b, 2] > 1]
    slots = sorted(s for a, n in cut for s in range(a, a + n))
    assert len(slots) == len(set(slots)) and (not slots or slots[-1] < d.max_parts)


def test_dplan_headline_shape_stays_uncut():
    """Batch 64 x 8192 (every sequence within 5/4 of the fair share): one unit
    per sequence, as the host planner's measured choice."""
    import torch
    d = mla.dplan_info(64, 128, 1, 1, syn.KV_BF16, False, 8192, 152)
    ws = torch.empty(int(d.workspace_bytes), dtype=torch.uint8, device="cuda")
    lens = torch.full((64,), 8192, dtype=torch.int32, device="cuda")
    mla.plan_device(d, lens, ws)
    counts, units, seq = unit_list(d, ws)
    assert counts[0] == 64 and np.all(seq[:, 2] == 1)


def test_dplan_context_clamped_to_capacity_and_csr_pages():
    import torch
    p = syn.make_problem(3, 1, 16, [500, 300, 64], 16, syn.KV_BF16, False, seed=38, name="clamp")
    d = info_for(p, capacity=512)
    t = to_device(p)
    lens = torch.tensor([500, 300, 600], dtype=torch.int32, device="cuda")  # 600 > capacity
    out, lse, st, _ = run_dplan(p, d, t=t, lens=lens)
    assert st & mla.DEVFLAG_CTX_RANGE
    # CSR: sequence 2 owns 4 pages (64 keys); 300 > 64 is clamped to its pages
    lens = torch.tensor([500, 300, 300], dtype=torch.int32, device="cuda")
    out, lse, st, _ = run_dplan(p, d, t=t, lens=lens, csr=True)
    assert st & mla.DEVFLAG_CTX_RANGE
    ref_o, ref_l = oracle_full(p)  # the clamped lengths are the problem's own
    assert_close(out, lse, ref_o, ref_l, "csr clamp")


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
def test_graph_replays_while_contexts_grow(kv_dtype):
    """plan_device + fwd + combine captured once with short contexts, then
    replayed 100 times while every context grows (decode steps add keys; the
    last replays are far past the capture's longest context): every replay
    is clean, and replays are checked against the oracle along the way."""
    import torch
    B, H, ps, cap = 8, 128, 16, 6000
    final = syn.ragged_lens(B, lo=200, hi=cap, seed=int(kv_dtype) + 7)
    p = syn.make_problem(B, 1, H, final, ps, kv_dtype, False, seed=39 + int(kv_dtype),
                         name="graph_grow")
    p.block_table = np.pad(p.block_table, ((0, 0), (0, cap // ps - p.block_table.shape[1])))
    d = info_for(p, capacity=cap)
    t = to_device(p)
    ws = torch.empty(int(d.workspace_bytes), dtype=torch.uint8, device="cuda")
    start = np.maximum(final // 8, 1).astype(np.int32)
    lens = torch.from_numpy(start.copy()).cuda()
    out = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, 1, H), dtype=torch.float32, device="cuda")
    mla.plan_device(d, lens, ws)  # warm-up outside the capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        mla.plan_device(d, lens, ws, stream=s)
        mla.fwd_dplan(d, t["q"], t["cache"], t["scale"], t["bt"], p.softmax_scale, out, lse, ws,
                      stream=s)
        mla.combine_dplan(d, out, lse, ws, stream=s)
    checks = {0, 37, 99}
    for k in range(100):
        cur = (start + ((final - start) * k) // 99).astype(np.int32)
        lens.copy_(torch.from_numpy(cur))
        g.replay()
        assert mla.dplan_check(d, ws) == 0
        if k in checks:
            q = syn.Problem(**{**p.__dict__, "seq_lens": cur})
            ref_o, ref_l = oracle.decode(q.q_bits, q.cache, q.kv_dtype, q.kv_scale, ps,
                                         q.block_table, cur, q.softmax_scale, False)
            assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_o, ref_l,
                         f"replay {k} (max ctx {cur.max()}, at capture {start.max()})")
    assert final.max() > 4 * start.max()
