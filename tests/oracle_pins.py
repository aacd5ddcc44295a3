"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each ``pin_*`` function takes an oracle binding (the real one, or a copy with a
planted mistake) and raises AssertionError when the binding disagrees with a
closed form, an invariance, a brute-force count or an independent library
routine.  ``test_oracle_pins.py`` runs them against the real oracle and checks
that every planted mistake trips at least one of them.

The method being pinned: absorbed-form MLA decode, where each 576-wide query
row scores the 576-wide latent rows of its sequence ("[Perf][Kimi-K3] Cut MLA
decode concat/cache epilogue latency", Purpose item 1: "576-wide row"),
gathered through a block table at any page size, with an optional causal
mask over the 1+MTP query tokens ("HK MLA: MI35x m16x8 retune, new m16x4
kernel, page_size + mask support", Summary track 1), a softmax, and the
softmax-weighted sum of the first 512 dims of those rows plus the row's
log-sum-exp.
"""
from __future__ import annotations

import math
import os

import numpy as np

import mla_synth as syn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def _bf16(x):
    return syn.f32_to_bf16_bits(np.asarray(x, np.float32))


def _f(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def layout(rows_bits, ps, perm_seed=0, dtype=np.uint16):
    """Place logical key rows [n, 576] into pages of size ps, in a shuffled
    physical order.  Returns (cache [P, ps, 576], block_table [1, P])."""
    n = rows_bits.shape[0]
    nblk = max(1, -(-n // ps))
    perm = np.random.default_rng(perm_seed).permutation(nblk).astype(np.int32)
    cache = np.zeros((nblk, ps, 576), dtype)
    for p in range(nblk):
        chunk = rows_bits[p * ps:(p + 1) * ps]
        cache[perm[p], :chunk.shape[0]] = chunk
    return cache, perm.reshape(1, nblk)


def run(orc, q_bits, rows_bits, ps=1, perm_seed=0, scale=SCALE, causal=False,
        kv_dtype=syn.KV_BF16, kv_scale=1.0, ctx=None):
    cache, bt = layout(rows_bits, ps, perm_seed,
                       np.uint16 if kv_dtype == syn.KV_BF16 else np.uint8)
    n = rows_bits.shape[0] if ctx is None else ctx
    return orc.decode(q_bits, cache, kv_dtype, kv_scale, ps, bt,
                      np.array([n], np.int32), scale, causal)


def rand_bits(seed, shape, sigma=1.0):
    g = np.random.default_rng(seed)
    return _bf16(g.standard_normal(shape).astype(np.float32) * np.float32(sigma))


# --------------------------------------------------------------- formats ---

def pin_bf16_decode(orc):
    """bf16 decode agrees with torch's bfloat16 -> float64 on random patterns."""
    import torch
    g = np.random.default_rng(1)
    bits = g.integers(0, 1 << 16, 4096, dtype=np.int64).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # drop inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(got, ref)


def pin_e4m3_all_codes(orc):
    """All 256 fp8 E4M3FN codes decode as torch.float8_e4m3fn does."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_e4m3_spec_values(orc):
    """Notable codes against the values the OCP FP8 specification lists."""
    path = os.path.join(GOLDEN, "e4m3_spec_values.txt")
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code, val = line.split()
        got = orc.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            want = float(eval(val, {"__builtins__": {}}))  # noqa: S307 (literal arithmetic)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def pin_e4m3_encode_roundtrip(orc):
    """Every finite E4M3FN value encodes back to its own code (both zeros too)."""
    for c in range(256):
        v = orc.e4m3_to_double(c)
        if math.isnan(v):
            continue
        assert orc.e4m3_encode(v) == c, (hex(c), v)


def pin_e4m3_encode_matches_torch(orc):
    """Nearest-even encoding agrees with torch's float32 -> float8_e4m3fn cast on
    values from 1e-5 to 448 in magnitude, both signs (the cast's range)."""
    import torch
    g = np.random.default_rng(40)
    x = np.concatenate([g.standard_normal(3000).astype(np.float32) * np.float32(sc)
                        for sc in (1e-4, 1e-2, 1.0, 30.0, 200.0)])
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def pin_e4m3_encode_ties_and_saturation(orc):
    """A value halfway between two neighbouring codes takes the even one;
    magnitudes past 448 saturate to 448; NaN stays NaN."""
    vals = [orc.e4m3_to_double(c) for c in range(0x7F)]
    for c in range(0x7E):
        mid = 0.5 * (vals[c] + vals[c + 1])  # exact in binary32 (at most 5 significant bits)
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == want, (hex(c), mid)
        assert orc.e4m3_encode(-mid) == 0x80 | want
    for big in (448.5, 464.0, 480.0, 1e6, 3e38):
        assert orc.e4m3_encode(big) == 0x7E and orc.e4m3_encode(-big) == 0xFE
    assert orc.e4m3_encode(float("nan")) & 0x7F == 0x7F


def _epilogue_inputs(seed, T, H, pages, ps, kv_dtype, n_pad=1):
    g = np.random.default_rng(seed)
    ql = rand_bits(seed + 1, (T, H, 512))
    qp = rand_bits(seed + 2, (T, H, 64))
    kc = rand_bits(seed + 3, (T, 512), sigma=2.0)
    kp = rand_bits(seed + 4, (T, 64), sigma=2.0)
    slots = g.choice(pages * ps, size=T, replace=False).astype(np.int64)
    slots[g.choice(T, size=n_pad, replace=False)] = -1  # padding tokens
    dt = np.uint16 if kv_dtype == syn.KV_BF16 else np.uint8
    cache = g.integers(0, 1 << (16 if dt is np.uint16 else 8), (pages, ps, 576)).astype(dt)
    if dt is np.uint16:
        cache &= np.uint16(0xBFFF)  # finite patterns only
    return ql, qp, kc, kp, slots, cache


def pin_epilogue_bf16_concat_and_insert(orc):
    """bf16: q rows are ql_nope then q_pe; each non-padding token's cache row
    (page slot // ps, offset slot % ps, in a cache of random bits) becomes
    kv_c then k_pe; every other cache element keeps its bits."""
    T, H, P, ps = 7, 3, 5, 4
    ql, qp, kc, kp, slots, cache = _epilogue_inputs(41, T, H, P, ps, syn.KV_BF16)
    q, out = orc.epilogue(ql, qp, kc, kp, slots, cache, syn.KV_BF16)
    assert np.array_equal(q[:, :, :512], ql) and np.array_equal(q[:, :, 512:], qp)
    flat_in, flat_out = cache.reshape(-1, 576), out.reshape(-1, 576)
    touched = np.zeros(P * ps, bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        touched[slots[t]] = True
        assert np.array_equal(flat_out[slots[t], :512], kc[t])
        assert np.array_equal(flat_out[slots[t], 512:], kp[t])
    assert np.array_equal(flat_out[~touched], flat_in[~touched])


def pin_epilogue_inserted_row_decodes_to_itself(orc):
    """The decode of a one-key sequence whose key is the row the epilogue just
    inserted returns that row's value dims and LSE = scale * <q, row>, with q
    the concatenated query row (closed forms of the decode, bf16 and fp8)."""
    T, H, P, ps = 3, 2, 4, 2
    for dt, s in ((syn.KV_BF16, 1.0), (syn.KV_FP8_E4M3, 0.03125)):
        ql, qp, kc, kp, slots, cache = _epilogue_inputs(43, T, H, P, ps, dt, n_pad=0)
        q, out = orc.epilogue(ql, qp, kc, kp, slots, cache, dt, s)
        for t in range(T):
            off = int(slots[t] % ps)
            # the inserted row, alone at offset 0 of a one-page cache
            page = out[slots[t] // ps][off:off + 1]
            page = np.concatenate([page, np.zeros((ps - 1, 576), page.dtype)])[None]
            o, l = orc.decode(q[t][None, None], page, dt, s, ps, np.array([[0]], np.int32),
                              np.array([1], np.int32), SCALE)
            row = np.concatenate([_f(kc[t]), _f(kp[t])])
            if dt == syn.KV_FP8_E4M3:
                row = np.array([orc.e4m3_to_double(int(c)) * s for c in page[0, 0]])
            assert np.array_equal(o[0, 0], np.broadcast_to(row[:512], (H, 512)))
            qrow = np.concatenate([_f(ql[t]), _f(qp[t])], axis=1)
            assert np.allclose(l[0, 0], SCALE * (qrow @ row), rtol=1e-12, atol=1e-12)


def pin_epilogue_fp8_within_rounding(orc):
    """fp8: each inserted code decodes to x / kv_scale within half an E4M3
    spacing at that magnitude (2^-4 relative for normals, 2^-10 absolute in the
    subnormal range), beyond 448 to 448."""
    T, H, P, ps = 6, 1, 4, 4
    ql, qp, kc, kp, slots, cache = _epilogue_inputs(45, T, H, P, ps, syn.KV_FP8_E4M3)
    s = 0.0123
    _, out = orc.epilogue(ql, qp, kc, kp, slots, cache, syn.KV_FP8_E4M3, s)
    flat = out.reshape(-1, 576)
    for t in range(T):
        if slots[t] < 0:
            continue
        x = np.concatenate([_f(kc[t]), _f(kp[t])])
        y = (x.astype(np.float32) / np.float32(s)).astype(np.float64)
        dec = np.array([orc.e4m3_to_double(int(c)) for c in flat[slots[t]]])
        yc = np.clip(y, -448, 448)
        tol = np.where(np.abs(yc) >= 2.0 ** -6, np.abs(yc) * 2.0 ** -4, 2.0 ** -10)
        assert np.all(np.abs(dec - yc) <= tol + 1e-300)
        assert np.all(np.sign(dec[dec != 0]) == np.sign(y[dec != 0]))


def _kvb_weights(seed, H, sigma=1.0 / 22.6):
    return rand_bits(seed, (H, 256, 512), sigma=sigma)


def pin_gather_kv_matches_numpy(orc):
    """gather_kv_b_proj against numpy's fp64 einsum over the logical rows
    (three sequences in shuffled pages of 16, one empty): k = [W_k c, rope],
    v = W_v c, rows packed sequence by sequence."""
    H, lens = 3, [37, 0, 20]
    seqs = [rand_bits(60 + b, (max(n, 1), 576))[:n] for b, n in enumerate(lens)]
    cache, bt, sl = _pool_layout([r if len(r) else np.zeros((1, 576), np.uint16) for r in seqs],
                                 16, seed=61)
    sl = np.array(lens, np.int32)
    w = _kvb_weights(62, H)
    k, v = orc.gather_kv_b_proj(cache, syn.KV_BF16, 1.0, 16, bt, sl, w)
    rows = np.concatenate([_f(r) for r in seqs if len(r)])
    wf = _f(w)
    want_k = np.einsum("hod,td->tho", wf[:, :128], rows[:, :512])
    want_v = np.einsum("hod,td->tho", wf[:, 128:], rows[:, :512])
    assert k.shape == (sum(lens), H, 192) and v.shape == (sum(lens), H, 128)
    assert np.allclose(k[:, :, :128], want_k, rtol=1e-12, atol=1e-12)
    assert np.allclose(v, want_v, rtol=1e-12, atol=1e-12)
    assert np.array_equal(k[:, :, 128:], np.broadcast_to(rows[:, None, 512:], (len(rows), H, 64)))


def pin_gather_kv_selection_weights(orc):
    """Weights that select one latent dim per output (a permutation per head,
    times 2 for the values) give those dims exactly, fp8 cache included
    (code * kv_scale)."""
    H, n, ps = 2, 11, 4
    g = np.random.default_rng(63)
    w = np.zeros((H, 256, 512), np.uint16)
    sel = [g.permutation(512)[:256] for _ in range(H)]
    for h in range(H):
        w[h, np.arange(128), sel[h][:128]] = _bf16([1.0])[0]
        w[h, 128 + np.arange(128), sel[h][128:]] = _bf16([2.0])[0]
    codes = g.integers(0, 0x7F, (n, 576)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11
    cache, bt = layout(codes, ps, perm_seed=4, dtype=np.uint8)
    s = 0.0625
    k, v = orc.gather_kv_b_proj(cache, syn.KV_FP8_E4M3, s, ps, bt, np.array([n], np.int32), w)
    dec = np.array([[orc.e4m3_to_double(int(c)) for c in row] for row in codes]) * s
    for h in range(H):
        assert np.array_equal(k[:, h, :128], dec[:, sel[h][:128]])
        assert np.array_equal(v[:, h], 2.0 * dec[:, sel[h][128:]])
        assert np.array_equal(k[:, h, 128:], dec[:, 512:])


def pin_gather_kv_page_size_invariance(orc):
    """The same logical rows at page sizes 1 and 16 expand to the same bits."""
    rows = rand_bits(64, (50, 576))
    w = _kvb_weights(65, 2)
    res = []
    for ps in (1, 16):
        cache, bt = layout(rows, ps, perm_seed=ps)
        res.append(orc.gather_kv_b_proj(cache, syn.KV_BF16, 1.0, ps, bt, np.array([50], np.int32), w))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


# ---------------------------------------------------------- closed forms ---

def pin_single_key(orc):
    """ctx = 1: the output is that row's first 512 dims; LSE is its scaled score."""
    q = rand_bits(2, (1, 1, 8, 576))
    row = rand_bits(3, (1, 576))
    out, lse = run(orc, q, row)
    assert np.array_equal(out[0, 0], np.broadcast_to(_f(row[0, :512]), (8, 512)))
    want = SCALE * (_f(q[0, 0]) @ _f(row[0]))
    assert np.allclose(lse[0, 0], want, rtol=1e-13, atol=1e-13)


def pin_single_key_fp8(orc):
    """fp8 cache, ctx = 1: output is code * kv_scale, decoded by torch."""
    import torch
    q = rand_bits(4, (1, 1, 4, 576))
    codes = np.random.default_rng(5).integers(0, 256, (1, 576)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30  # no NaN codes
    s = 0.0123
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()[0]
    out, lse = run(orc, q, codes, kv_dtype=syn.KV_FP8_E4M3, kv_scale=s)
    assert np.allclose(out[0, 0], np.broadcast_to(dec[:512] * s, (4, 512)), rtol=1e-15, atol=0)
    want = SCALE * (_f(q[0, 0]) @ (dec * s))
    assert np.allclose(lse[0, 0], want, rtol=1e-12, atol=1e-13)


def pin_zero_query_mean(orc):
    """q = 0: every score is 0, so the output is the mean value row and LSE = ln n."""
    n = 37
    q = np.zeros((1, 1, 3, 576), np.uint16)
    rows = rand_bits(6, (n, 576))
    out, lse = run(orc, q, rows, ps=4)
    mean = _f(rows[:, :512]).mean(axis=0)
    assert np.allclose(out[0, 0], mean, rtol=0, atol=1e-14)
    assert np.allclose(lse[0, 0], math.log(n), rtol=0, atol=1e-14)


def pin_scale_zero_mean(orc):
    """softmax_scale = 0: uniform weights whatever q is."""
    n = 23
    q = rand_bits(7, (1, 1, 2, 576))
    rows = rand_bits(8, (n, 576))
    out, lse = run(orc, q, rows, scale=0.0)
    assert np.allclose(out[0, 0], _f(rows[:, :512]).mean(axis=0), rtol=0, atol=1e-14)
    assert np.allclose(lse[0, 0], math.log(n), rtol=0, atol=1e-14)


def pin_two_keys_logistic(orc):
    """Two keys whose scores differ by a known amount: the weights are the
    logistic function of the difference (scores built from a rope one-hot)."""
    q = np.zeros((1, 1, 1, 576), np.uint16)
    q[0, 0, 0, 520] = _bf16([2.0])[0]
    rows = rand_bits(9, (2, 576))
    rows[:, 512:] = 0
    rows[0, 520] = _bf16([1.0])[0]
    rows[1, 520] = _bf16([-1.5])[0]
    z0, z1 = SCALE * 2.0 * 1.0, SCALE * 2.0 * -1.5
    w1 = 1.0 / (1.0 + math.exp(z0 - z1))
    out, lse = run(orc, q, rows)
    want = w1 * _f(rows[1, :512]) + (1 - w1) * _f(rows[0, :512])
    assert np.allclose(out[0, 0, 0], want, rtol=1e-14, atol=1e-15)
    assert abs(lse[0, 0, 0] - (z0 + math.log1p(math.exp(z1 - z0)))) < 1e-14


def pin_unit_values(orc):
    """Value dims all 1: the weights sum to one, so every output is 1."""
    rows = rand_bits(10, (41, 576))
    rows[:, :512] = _bf16([1.0])[0]
    q = rand_bits(11, (1, 1, 5, 576), sigma=0.3)
    out, _ = run(orc, q, rows, ps=8)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-14)


def pin_empty_context(orc):
    """ctx = 0 gives out = 0, lse = -inf; causal rows with no visible key too."""
    q = rand_bits(12, (1, 2, 3, 576))
    rows = rand_bits(13, (4, 576))
    out, lse = run(orc, q, rows, ctx=0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out, lse = run(orc, q, rows, ctx=1, causal=True)  # ctx < Sq: token 0 sees nothing
    assert np.all(out[0, 0] == 0) and np.all(np.isneginf(lse[0, 0]))
    assert np.array_equal(out[0, 1], np.broadcast_to(_f(rows[0, :512]), (3, 512)))


def pin_causal_admits_exact_count(orc):
    """Causal: query token i admits exactly ctx - Sq + i + 1 keys.  With q = 0
    the weights are uniform, so LSE = ln(visible keys); a marker value at key
    38 shows up in exactly the tokens that may see it."""
    sq, ctx, marker = 4, 40, 38
    q = np.zeros((1, sq, 2, 576), np.uint16)
    rows = np.zeros((ctx, 576), np.uint16)
    rows[marker, 0] = _bf16([1.0])[0]
    out, lse = run(orc, q, rows, ps=16, causal=True)
    for i in range(sq):
        n = ctx - sq + i + 1
        assert np.allclose(lse[0, i], math.log(n), rtol=0, atol=1e-14)
        want = 1.0 / n if marker < n else 0.0
        assert np.allclose(out[0, i, :, 0], want, rtol=0, atol=1e-16)
    out, lse = run(orc, q, rows, ps=16, causal=False)
    assert np.allclose(lse, math.log(ctx), rtol=0, atol=1e-14)


def pin_matches_torch_sdpa(orc):
    """Dense case (page_size 1, identity table) against torch's fp64
    scaled_dot_product_attention, per (token, head) row."""
    import torch
    sq, h, n = 2, 3, 50
    q = rand_bits(14, (1, sq, h, 576))
    rows = rand_bits(15, (n, 576))
    cache = rows.reshape(n, 1, 576)
    bt = np.arange(n, dtype=np.int32).reshape(1, n)
    out, lse = orc.decode(q, cache, syn.KV_BF16, 1.0, 1, bt, np.array([n], np.int32), SCALE, False)
    qt = torch.from_numpy(_f(q[0]).reshape(sq * h, 576))[None, None]
    kt = torch.from_numpy(_f(rows))[None, None]
    vt = kt[..., :512]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=SCALE)[0, 0].numpy()
    assert np.allclose(out[0].reshape(sq * h, 512), ref, rtol=1e-12, atol=1e-13)


def _pool_layout(seqs, ps, seed):
    """Place each sequence's logical key rows (list of [n_b, 576] arrays) into
    pages of size ps drawn from one shuffled pool.  Returns (cache, block_table,
    seq_lens); the rows are known, so expected values need no gather."""
    nblk = [max(1, -(-r.shape[0] // ps)) for r in seqs]
    total = sum(nblk)
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    cache = np.zeros((total, ps, 576), np.uint16)
    bt = np.zeros((len(seqs), max(nblk)), np.int32)
    off = 0
    for b, rows in enumerate(seqs):
        for k in range(nblk[b]):
            page = perm[off + k]
            bt[b, k] = page
            chunk = rows[k * ps:(k + 1) * ps]
            cache[page, :chunk.shape[0]] = chunk
        off += nblk[b]
    return cache, bt, np.array([r.shape[0] for r in seqs], np.int32)


def pin_decode_row_matches_sdpa_causal(orc):
    """decode_row on every (b, i, h) of a causal MTP batch (three sequences,
    Sq = 4, 3 heads, page size 16, shuffled pages, one sequence shorter than
    Sq) against torch's fp64 scaled_dot_product_attention of that query row
    over the logical rows its token may see, keys [0, ctx - Sq + i + 1)."""
    import torch
    sq, h, lens = 4, 3, [40, 17, 3]
    seqs = [rand_bits(30 + b, (n, 576)) for b, n in enumerate(lens)]
    cache, bt, sl = _pool_layout(seqs, 16, seed=33)
    q = rand_bits(34, (len(lens), sq, h, 576))
    for b, n_ctx in enumerate(lens):
        k = torch.from_numpy(_f(seqs[b]))
        for i in range(sq):
            n = max(0, min(n_ctx, n_ctx - sq + i + 1))
            for hh in range(h):
                out, lse = orc.decode_row(q, cache, syn.KV_BF16, 1.0, 16, bt, sl, SCALE, True,
                                          b, i, hh)
                if n == 0:
                    assert np.all(out == 0) and lse == -math.inf, (b, i, hh)
                    continue
                qr = torch.from_numpy(_f(q[b, i, hh]))[None, None, None]
                kk = k[:n][None, None]
                ref = torch.nn.functional.scaled_dot_product_attention(
                    qr, kk, kk[..., :512], scale=SCALE)[0, 0, 0].numpy()
                z = SCALE * (_f(seqs[b][:n]) @ _f(q[b, i, hh]))
                ref_lse = float(np.logaddexp.reduce(z))
                assert np.allclose(out, ref, rtol=1e-12, atol=1e-13), (b, i, hh)
                assert abs(lse - ref_lse) < 1e-12, (b, i, hh)


def pin_decode_row_equals_decode(orc):
    """decode_row gives, bit for bit, the row decode gives for the whole batch
    (causal MTP, Sq = 4, page size 16, ragged contexts)."""
    p = syn.make_problem(3, 4, 3, [53, 6, 21], 16, syn.KV_BF16, True, seed=35)
    args = (p.q_bits, p.cache, p.kv_dtype, p.kv_scale, p.page_size, p.block_table,
            p.seq_lens, p.softmax_scale, p.causal)
    full_o, full_l = orc.decode(*args)
    for b in range(p.batch):
        for i in range(p.sq):
            for hh in range(p.heads):
                o, l = orc.decode_row(*args, b, i, hh)
                assert np.array_equal(o, full_o[b, i, hh]), (b, i, hh)
                assert l == full_l[b, i, hh] or (np.isneginf(l) and np.isneginf(full_l[b, i, hh]))


# ------------------------------------------------------------ invariances ---

def _random_problem_rows(seed, n):
    return rand_bits(seed, (n, 576))


def pin_page_permutation_invariance(orc):
    """The physical page order does not change a single bit of the result."""
    q = rand_bits(16, (1, 1, 4, 576))
    rows = _random_problem_rows(17, 77)
    a = run(orc, q, rows, ps=4, perm_seed=1)
    b = run(orc, q, rows, ps=4, perm_seed=2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_page_size_invariance(orc):
    """The same logical rows at page sizes 1, 16 and 64 give the same bits."""
    q = rand_bits(18, (1, 2, 3, 576))
    rows = _random_problem_rows(19, 150)
    res = [run(orc, q, rows, ps=ps, causal=True) for ps in (1, 16, 64)]
    for o, l in res[1:]:
        assert np.array_equal(o, res[0][0]) and np.array_equal(l, res[0][1])


def pin_page_layout_causal_subset(orc):
    """16 keys in 4 pages of 4, causal over 4 tokens: each token's visible key
    subset read through the page table equals the dense (page_size 1,
    identity table) result, so page and slot cannot be mixed up."""
    q = rand_bits(25, (1, 4, 2, 576))
    rows = _random_problem_rows(26, 16)
    dense = orc.decode(q, rows.reshape(16, 1, 576), syn.KV_BF16, 1.0, 1,
                       np.arange(16, dtype=np.int32).reshape(1, 16), np.array([16], np.int32),
                       SCALE, True)
    paged = run(orc, q, rows, ps=4, perm_seed=3, causal=True)
    assert np.array_equal(dense[0], paged[0]) and np.array_equal(dense[1], paged[1])


def pin_key_order_invariance(orc):
    """Permuting the logical key order leaves the result unchanged (to rounding)."""
    q = rand_bits(20, (1, 1, 4, 576))
    rows = _random_problem_rows(21, 90)
    perm = np.random.default_rng(22).permutation(90)
    a = run(orc, q, rows, ps=1)
    b = run(orc, q, rows[perm], ps=1)
    assert np.allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    assert np.allclose(a[1], b[1], rtol=1e-13, atol=1e-13)


def pin_split_merge_equals_unsplit(orc):
    """Splitting the key range into chunks (one of them empty) and merging the
    chunk results by log-sum-exp equals the unsplit result."""
    p = syn.make_problem(2, 2, 4, [97, 61], 8, syn.KV_BF16, True, seed=23)
    args = (p.q_bits, p.cache, p.kv_dtype, p.kv_scale, p.page_size, p.block_table,
            p.seq_lens, p.softmax_scale, p.causal)
    full_o, full_l = orc.decode(*args)
    bounds = [0, 7, 30, 64, 97, 200]
    parts = [orc.decode(*args, k_range=(bounds[k], bounds[k + 1])) for k in range(len(bounds) - 1)]
    o_parts = np.stack([o.reshape(-1, 512) for o, _ in parts])
    l_parts = np.stack([l.reshape(-1) for _, l in parts])
    assert np.all(np.isneginf(l_parts[-1]))
    mo, ml = orc.lse_merge(o_parts, l_parts)
    assert np.allclose(mo, full_o.reshape(-1, 512), rtol=1e-12, atol=1e-14)
    assert np.allclose(ml, full_l.reshape(-1), rtol=1e-13, atol=1e-13)


def pin_poison_never_read(orc):
    """NaN in slots past ctx and -1 past the last block-table entry change nothing."""
    kw = dict(batch=3, sq=2, heads=4, seq_lens=[19, 40, 7], page_size=16, causal=True, seed=24)
    a = syn.make_problem(poison=False, **kw)
    b = syn.make_problem(poison=True, **kw)
    ra = orc.decode(a.q_bits, a.cache, 0, 1.0, 16, a.block_table, a.seq_lens, SCALE, True)
    rb = orc.decode(b.q_bits, b.cache, 0, 1.0, 16, b.block_table, b.seq_lens, SCALE, True)
    assert np.all(np.isfinite(rb[0])) and np.array_equal(ra[0], rb[0]) and np.array_equal(ra[1], rb[1])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
