"""GPU parity of the cached-prefix expansion (mla_gather_kv_b_proj) through
the C ABI against the oracle on the same bits: keys and values of every
cached token and head, bf16 and fp8 caches, page sizes 1 / 16 / 64, ragged
batches with chunks past a sequence's end, head counts that leave a partial
head group.  Outputs are bf16, so the tolerance is that of ``parity.py``'s
max-abs and Frobenius bounds."""
import numpy as np
import pytest

import mla_synth as syn
import oracle
import paged_mla_decode_latent_gb300 as mla
from parity import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.lib()


def weights(seed, H):
    g = np.random.default_rng(seed)
    w = g.standard_normal((H, 256, 512)).astype(np.float32) / np.float32(np.sqrt(512.0))
    return syn.f32_to_bf16_bits(w)


def check_close(got, ref, what):
    err = np.abs(got - ref)
    big = np.abs(ref) >= 4.0
    half = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8).astype(int))
    assert (err[~big].max() if (~big).any() else 0) <= 1.5e-2, what
    assert ((err - half)[big].max() if big.any() else 0) <= 1.5e-2, what
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= 4e-3, (what, fro)


def run(p, H, seed=0, max_ctx=None):
    import torch
    t = to_device(p)
    w = weights(seed, H)
    wt = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).cuda()
    cu = np.zeros(p.batch + 1, np.int32)
    cu[1:] = np.cumsum(p.seq_lens)
    T = max(int(cu[-1]), 1)
    k = torch.full((T, H, 192), float("nan"), dtype=torch.bfloat16, device="cuda")
    v = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc = int(max_ctx if max_ctx is not None else p.seq_lens.max())
    mla.gather_kv_b_proj(t["cache"], t["scale"], t["bt"], t["lens"], torch.from_numpy(cu).cuda(),
                         mc, wt, k, v, status)
    torch.cuda.synchronize()
    return k.double().cpu().numpy()[:cu[-1]], v.double().cpu().numpy()[:cu[-1]], int(status.item()), w


@pytest.mark.parametrize("kv_dtype", [syn.KV_BF16, syn.KV_FP8_E4M3])
@pytest.mark.parametrize("H,ps,lens", [(12, 1, [300, 1, 129, 0]), (16, 16, [1000, 77]),
                                        (20, 64, [700, 2000, 5]), (128, 16, [200, 130])])
def test_gather_kv_b_proj_matches_oracle(kv_dtype, H, ps, lens):
    p = syn.make_problem(len(lens), 1, 4, lens, ps, kv_dtype, False, seed=H + ps, name="gkv")
    k, v, st, w = run(p, H, seed=H)
    assert st == 0
    rk, rv = oracle.gather_kv_b_proj(p.cache, p.kv_dtype, p.kv_scale, ps, p.block_table,
                                     p.seq_lens, w)
    check_close(k[:, :, :128], rk[:, :, :128], "k nope")
    check_close(v, rv, "v")
    check_close(k[:, :, 128:], rk[:, :, 128:], "k rope")


def test_gather_kv_b_proj_long_context_fp8():
    """The pages' shape: 12 heads (TP8-local), fp8 cache, page size 1, one long
    context that is not a multiple of the 128-token chunk."""
    p = syn.make_problem(1, 1, 4, [32000 + 77], 1, syn.KV_FP8_E4M3, False, seed=70, name="gkv_long")
    k, v, st, w = run(p, 12, seed=71)
    assert st == 0
    rk, rv = oracle.gather_kv_b_proj(p.cache, p.kv_dtype, p.kv_scale, 1, p.block_table, p.seq_lens, w)
    check_close(k, rk, "k")
    check_close(v, rv, "v")
