"""fp64 CPU oracle for paged MLA decode (absorbed form).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``paged_mla_decode_latent_gb300``) never imports,
links or calls it, and it imports nothing from the product library.

The arithmetic lives in ``mla_oracle.c`` (plain C, IEEE double, OpenMP over
query rows).  This module only compiles it with gcc and marshals numpy arrays.
See the header of ``mla_oracle.c`` for the definition it follows and the pages
each step comes from.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariances, brute force, library cross-checks); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "libmla_oracle.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1

_default = None


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``libmla_oracle.so`` next to it."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c99", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime on this host: build single-threaded.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    c_p = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.mla_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.mla_oracle_bf16_to_double.restype = f64
    lib.mla_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.mla_oracle_e4m3_to_double.restype = f64
    lib.mla_oracle_num_threads.argtypes = []
    lib.mla_oracle_num_threads.restype = i32
    lib.mla_oracle_decode_range.argtypes = [
        c_p, c_p, i32, f64, i32, c_p, i64, c_p, i32, i32, i32, i32, f64,
        i32, i32, i64, i64, c_p, c_p]
    lib.mla_oracle_decode_range.restype = None
    lib.mla_oracle_decode_row.argtypes = [
        c_p, c_p, i32, f64, i32, c_p, i64, c_p, i32, i32, i32, f64,
        i32, i32, i32, c_p, c_p]
    lib.mla_oracle_decode_row.restype = None
    lib.mla_oracle_lse_merge.argtypes = [c_p, c_p, i32, i64, c_p, c_p]
    lib.mla_oracle_lse_merge.restype = None
    lib.mla_oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.mla_oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.mla_oracle_epilogue.argtypes = [c_p, c_p, c_p, c_p, c_p, i32, i32, c_p, c_p, i64, i32,
                                        i32, ctypes.c_float]
    lib.mla_oracle_epilogue.restype = None
    lib.mla_oracle_gather_kv_b_proj.argtypes = [c_p, i32, f64, i32, c_p, i64, c_p, c_p, i32, c_p,
                                                i32, c_p, c_p]
    lib.mla_oracle_gather_kv_b_proj.restype = None
    return lib


def _load():
    global _default
    if _default is None:
        build()
        _default = _bind(_LIB)
    return _default


def compile_variant(src_text: str, workdir: str):
    """Compile a modified copy of the oracle source into ``workdir`` and bind it.

    Used only by the tests that check the pins catch planted mistakes; the
    returned object has the same functions as this module.
    """
    import types
    src = os.path.join(workdir, "variant.c")
    lib = os.path.join(workdir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-shared", "-fPIC", "-std=c99", src, "-o", lib, "-lm"],
                   check=True, capture_output=True, text=True)
    bound = _bind(lib)
    ns = types.SimpleNamespace(KV_BF16=KV_BF16, KV_FP8_E4M3=KV_FP8_E4M3)
    for name in ("bf16_to_double", "e4m3_to_double", "decode", "decode_row", "lse_merge",
                 "e4m3_encode", "epilogue", "gather_kv_b_proj"):
        fn = globals()[name]
        ns.__dict__[name] = (lambda f: (lambda *a, **k: f(*a, _lib=bound, **k)))(fn)
    return ns


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use on this host."""
    return int(_load().mla_oracle_num_threads())


def bf16_to_double(bits: int, _lib=None) -> float:
    return float((_lib or _load()).mla_oracle_bf16_to_double(int(bits)))


def e4m3_to_double(code: int, _lib=None) -> float:
    return float((_lib or _load()).mla_oracle_e4m3_to_double(int(code)))


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def decode(q_bits, cache, kv_dtype, kv_scale, page_size, block_table, seq_lens,
           softmax_scale, causal=False, b_range=None, k_range=None, _lib=None):
    """Attention of every query row of sequences ``b_range`` (default: all).

    q_bits      uint16 [B, Sq, H, 576]   bf16 bit patterns
    cache       uint16 (bf16 bits) or uint8 (e4m3 codes) [num_pages, ps, 576]
    block_table int32  [B, max_blocks]
    seq_lens    int32  [B]
    k_range     optional (k_begin, k_end) restriction of every row's keys

    Returns (out [nb, Sq, H, 512] float64, lse [nb, Sq, H] float64).
    """
    lib = _lib or _load()
    q_bits = _c(q_bits, np.uint16)
    B, Sq, H, D = q_bits.shape
    assert D == 576
    cache = _c(cache, np.uint16 if kv_dtype == KV_BF16 else np.uint8)
    assert cache.shape[-1] == 576 and cache.shape[1] == page_size
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    b0, b1 = (0, B) if b_range is None else b_range
    k0, k1 = (0, np.iinfo(np.int64).max) if k_range is None else k_range
    nb = b1 - b0
    out = np.zeros((nb, Sq, H, 512), np.float64)
    lse = np.zeros((nb, Sq, H), np.float64)
    lib.mla_oracle_decode_range(
        q_bits.ctypes.data, cache.ctypes.data, int(kv_dtype), float(kv_scale),
        int(page_size), bt.ctypes.data, int(bt.shape[1]), sl.ctypes.data, B, Sq, H,
        int(bool(causal)), float(softmax_scale), int(b0), int(b1), int(k0), int(k1),
        out.ctypes.data, lse.ctypes.data)
    return out, lse


def decode_row(q_bits, cache, kv_dtype, kv_scale, page_size, block_table, seq_lens,
               softmax_scale, causal, b, i, h, _lib=None):
    """Attention of the single query row (b, i, h): (out [512], lse)."""
    lib = _lib or _load()
    q_bits = _c(q_bits, np.uint16)
    B, Sq, H, _ = q_bits.shape
    cache = _c(cache, np.uint16 if kv_dtype == KV_BF16 else np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.zeros(512, np.float64)
    lse = np.zeros(1, np.float64)
    lib.mla_oracle_decode_row(
        q_bits.ctypes.data, cache.ctypes.data, int(kv_dtype), float(kv_scale),
        int(page_size), bt.ctypes.data, int(bt.shape[1]), sl.ctypes.data, Sq, H,
        int(bool(causal)), float(softmax_scale), int(b), int(i), int(h),
        out.ctypes.data, lse.ctypes.data)
    return out, float(lse[0])


def lse_merge(o_parts, lse_parts, _lib=None):
    """Log-sum-exp merge of S partial results: o_parts [S, rows, 512], lse_parts [S, rows]."""
    lib = _lib or _load()
    o_parts = _c(o_parts, np.float64)
    lse_parts = _c(lse_parts, np.float64)
    S, rows = lse_parts.shape
    out = np.zeros((rows, 512), np.float64)
    lse = np.zeros(rows, np.float64)
    lib.mla_oracle_lse_merge(o_parts.ctypes.data, lse_parts.ctypes.data, int(S), int(rows),
                             out.ctypes.data, lse.ctypes.data)
    return out, lse


def e4m3_encode(y: float, _lib=None) -> int:
    """Nearest fp8 E4M3FN code of the binary32 value y (ties to even, saturating)."""
    return int((_lib or _load()).mla_oracle_e4m3_encode(float(np.float32(y))))


def epilogue(ql_nope, q_pe, kv_c, k_pe, slot_mapping, cache, kv_dtype, kv_scale=1.0,
             _lib=None):
    """The decode epilogue: returns (q [T, H, 576] bf16 bits, the cache after the
    inserts).  ql_nope uint16 [T, H, 512], q_pe uint16 [T, H, 64], kv_c uint16
    [T, 512], k_pe uint16 [T, 64] (bf16 bits), slot_mapping int64 [T], cache
    uint16 / uint8 [P, ps, 576] (copied, not modified)."""
    lib = _lib or _load()
    ql = _c(ql_nope, np.uint16)
    qp = _c(q_pe, np.uint16)
    kc = _c(kv_c, np.uint16)
    kp = _c(k_pe, np.uint16)
    sm = _c(slot_mapping, np.int64)
    T, H, _ = ql.shape
    q = np.zeros((T, H, 576), np.uint16)
    out_cache = np.array(cache, dtype=np.uint16 if kv_dtype == KV_BF16 else np.uint8, copy=True,
                         order="C")
    lib.mla_oracle_epilogue(ql.ctypes.data, qp.ctypes.data, kc.ctypes.data, kp.ctypes.data,
                            sm.ctypes.data, int(T), int(H), q.ctypes.data, out_cache.ctypes.data,
                            int(out_cache.shape[0]), int(out_cache.shape[1]), int(kv_dtype),
                            float(np.float32(kv_scale)))
    return q, out_cache


def gather_kv_b_proj(cache, kv_dtype, kv_scale, page_size, block_table, seq_lens, w_bits,
                     _lib=None):
    """Per-head keys and values of every cached token: (k [T, H, 192], v [T, H, 128])
    in float64, T = sum(seq_lens), rows packed sequence by sequence.  w_bits is
    kv_b_proj as bf16 bits [H, 256, 512] (each head's 128 key rows, then 128
    value rows)."""
    lib = _lib or _load()
    cache = _c(cache, np.uint16 if kv_dtype == KV_BF16 else np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    w = _c(w_bits, np.uint16)
    H = int(w.shape[0])
    assert w.shape[1:] == (256, 512)
    cu = np.zeros(len(sl) + 1, np.int32)
    cu[1:] = np.cumsum(sl)
    T = int(cu[-1])
    k = np.zeros((max(T, 1), H, 192), np.float64)
    v = np.zeros((max(T, 1), H, 128), np.float64)
    lib.mla_oracle_gather_kv_b_proj(cache.ctypes.data, int(kv_dtype), float(kv_scale),
                                    int(page_size), bt.ctypes.data, int(bt.shape[1]),
                                    sl.ctypes.data, cu.ctypes.data, int(len(sl)), w.ctypes.data,
                                    H, k.ctypes.data, v.ctypes.data)
    return k[:T], v[:T]