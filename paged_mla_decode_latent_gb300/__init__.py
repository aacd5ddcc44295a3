"""Paged MLA decode (absorbed form) for GB300 / sm_103a -- thin Python binding.

Every step of the decode runs in ``libmla_decode.so`` (hand-written CUDA for
sm_103a, C ABI declared in ``include/mla_decode.h``).  This module only loads
that library with ctypes and turns torch tensors into pointers and the current
CUDA stream into a ``cudaStream_t``.  There is no CPU or PyTorch fallback: if
the library is missing, every call raises.

Names follow the C ABI: ``plan`` -> ``mla_decode_plan``, ``fwd`` ->
``mla_decode_fwd``, ``combine`` -> ``mla_decode_combine``, ``check`` ->
``mla_decode_check``, ``epilogue`` -> ``mla_decode_epilogue``, ``step`` ->
``mla_decode_step``; the device-planned path: ``dplan_info``, ``plan_device``,
``fwd_dplan`` and ``combine_dplan``; ``gather_kv_b_proj`` ->
``mla_gather_kv_b_proj``.  ``decode`` is plan + fwd + combine with freshly
allocated outputs and workspace, for convenience.
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmla_decode.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1
D_QK = 576
D_V = 512

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_DEVICE_CHECK = -5
ERR_TIMEOUT = -6

DEVFLAG_BAD_PAGE = 0x1
DEVFLAG_CTX_RANGE = 0x2
DEVFLAG_TIMEOUT = 0x4
DEVFLAG_Q_RANGE = 0x8

# Every symbol include/mla_decode.h declares.
EXPORTED_SYMBOLS = ("mla_decode_plan", "mla_decode_fwd", "mla_decode_combine",
                    "mla_decode_check", "mla_decode_dplan_info", "mla_decode_plan_device",
                    "mla_decode_fwd_dplan", "mla_decode_combine_dplan", "mla_decode_epilogue",
                    "mla_decode_step", "mla_gather_kv_b_proj", "mla_decode_fwd_noalloc",
                    "mla_status_string", "mla_decode_version")


class Plan(ctypes.Structure):
    """Mirror of ``mla_decode_plan_t`` (plain old data)."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "version", "batch", "num_heads", "sq", "page_size", "kv_dtype", "causal", "rows",
        "row_tile", "row_blocks", "max_ctx", "key_tile", "chunk_len", "num_splits", "num_sms",
        "cluster_size", "grid_x", "grid_y", "grid_z", "wait_limit_us")] + [
        (n, ctypes.c_int64) for n in (
            "ws_partial_o_offset", "ws_partial_lse_offset", "ws_status_offset", "workspace_bytes")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class DPlan(ctypes.Structure):
    """Mirror of ``mla_decode_dplan_t`` (plain old data)."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "version", "batch", "num_heads", "sq", "page_size", "kv_dtype", "causal", "rows",
        "row_blocks", "ctx_capacity", "num_sms", "pairs", "max_parts", "max_units",
        "min_chunk_keys", "key_tile", "wait_limit_us", "reserved0")] + [
        (n, ctypes.c_int64) for n in (
            "ws_units_offset", "ws_seq_offset", "ws_count_offset", "ws_partial_o_offset",
            "ws_partial_lse_offset", "ws_status_offset", "workspace_bytes")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class MLADecodeError(RuntimeError):
    def __init__(self, status, where):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    from . import _build
    return _build.build(force=force, verbose=verbose)


def lib():
    """The loaded ``libmla_decode.so``; raises if it was never built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run paged_mla_decode_latent_gb300.build() "
                           "(needs nvcc); there is no fallback implementation")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    P = ctypes.POINTER(Plan)
    L.mla_decode_plan.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, P]
    L.mla_decode_plan.restype = ctypes.c_int
    L.mla_decode_fwd.argtypes = [P, vp, vp, i64, vp, vp, i64, vp, f32, vp, vp, vp,
                                 ctypes.c_size_t, vp]
    L.mla_decode_fwd.restype = ctypes.c_int
    L.mla_decode_combine.argtypes = [P, vp, vp, ctypes.c_size_t, vp, vp, vp]
    L.mla_decode_combine.restype = ctypes.c_int
    L.mla_decode_fwd_noalloc.argtypes = [P, vp, vp, i64, vp, vp, i64, vp, f32, vp, vp, vp]
    L.mla_decode_fwd_noalloc.restype = ctypes.c_int
    D = ctypes.POINTER(DPlan)
    L.mla_decode_dplan_info.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, D]
    L.mla_decode_dplan_info.restype = ctypes.c_int
    L.mla_decode_plan_device.argtypes = [D, vp, vp, vp, ctypes.c_size_t, vp]
    L.mla_decode_plan_device.restype = ctypes.c_int
    L.mla_decode_fwd_dplan.argtypes = [D, vp, vp, i64, vp, vp, i64, vp, f32, vp, vp, vp,
                                       ctypes.c_size_t, vp]
    L.mla_decode_fwd_dplan.restype = ctypes.c_int
    L.mla_decode_combine_dplan.argtypes = [D, vp, ctypes.c_size_t, vp, vp, vp]
    L.mla_decode_combine_dplan.restype = ctypes.c_int
    L.mla_gather_kv_b_proj.argtypes = [vp, i64, i32, i32, vp, vp, i64, vp, vp, i32, i32, vp, i32,
                                       vp, vp, vp, vp]
    L.mla_gather_kv_b_proj.restype = ctypes.c_int
    L.mla_decode_epilogue.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, vp, i64, i32, i32, vp,
                                      i32, vp, vp]
    L.mla_decode_epilogue.restype = ctypes.c_int
    L.mla_decode_step.argtypes = [P, vp, vp, vp, vp, vp, i32, vp, vp, i64, vp, vp, i64, vp, f32,
                                  vp, vp, vp, ctypes.c_size_t, vp]
    L.mla_decode_step.restype = ctypes.c_int
    L.mla_decode_check.argtypes = [P, vp, vp, ctypes.POINTER(i32)]
    L.mla_decode_check.restype = ctypes.c_int
    L.mla_status_string.argtypes = [ctypes.c_int]
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_decode_version.argtypes = []
    L.mla_decode_version.restype = ctypes.c_char_p
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def version() -> str:
    return lib().mla_decode_version().decode()


def _raise(st, where):
    if st != OK:
        raise MLADecodeError(st, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def plan(seq_lens_host, num_heads: int, sq: int, page_size: int, kv_dtype: int = KV_BF16,
         causal: bool = False, num_sms: int = 0) -> Plan:
    """``mla_decode_plan`` on host context lengths (list / numpy / CPU tensor)."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32).reshape(-1))
    p = Plan()
    st = lib().mla_decode_plan(lens.ctypes.data, int(lens.size), int(num_heads), int(sq),
                               int(page_size), int(kv_dtype), int(bool(causal)), int(num_sms),
                               ctypes.byref(p))
    _raise(st, "mla_decode_plan")
    return p


def fwd(p: Plan, q, kv_cache, kv_scale, block_table, seq_lens, softmax_scale: float, out, lse,
        workspace, stream=None) -> None:
    """``mla_decode_fwd``.  Tensors are CUDA tensors in the layouts of the C ABI."""
    st = lib().mla_decode_fwd(
        ctypes.byref(p), _ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]), _ptr(kv_scale),
        _ptr(block_table), int(block_table.stride(0)), _ptr(seq_lens), float(softmax_scale),
        _ptr(out), _ptr(lse), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _stream(stream))
    _raise(st, "mla_decode_fwd")


def combine(p: Plan, seq_lens, out, lse, workspace, stream=None) -> None:
    """``mla_decode_combine`` (no-op when the plan has one split)."""
    st = lib().mla_decode_combine(
        ctypes.byref(p), _ptr(seq_lens), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(out), _ptr(lse), _stream(stream))
    _raise(st, "mla_decode_combine")


def dplan_info(batch: int, num_heads: int, sq: int, page_size: int, kv_dtype: int = KV_BF16,
               causal: bool = False, ctx_capacity: int = 0, num_sms: int = 0) -> DPlan:
    """``mla_decode_dplan_info``: sizes of the device-planned decode."""
    d = DPlan()
    st = lib().mla_decode_dplan_info(int(batch), int(num_heads), int(sq), int(page_size),
                                     int(kv_dtype), int(bool(causal)), int(ctx_capacity),
                                     int(num_sms), ctypes.byref(d))
    _raise(st, "mla_decode_dplan_info")
    return d


def _ws_bytes(workspace):
    return int(workspace.numel() * workspace.element_size())


def plan_device(d: DPlan, seq_lens, workspace, kv_indptr=None, stream=None) -> None:
    """``mla_decode_plan_device``: the partition, computed on the GPU."""
    st = lib().mla_decode_plan_device(ctypes.byref(d), _ptr(seq_lens), _ptr(kv_indptr),
                                      _ptr(workspace), _ws_bytes(workspace), _stream(stream))
    _raise(st, "mla_decode_plan_device")


def fwd_dplan(d: DPlan, q, kv_cache, kv_scale, block_table, softmax_scale: float, out, lse,
              workspace, kv_indptr=None, stream=None) -> None:
    """``mla_decode_fwd_dplan``; block_table is kv_indices when kv_indptr is given."""
    stride = int(block_table.stride(0)) if block_table.dim() == 2 else 1
    st = lib().mla_decode_fwd_dplan(
        ctypes.byref(d), _ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]), _ptr(kv_scale),
        _ptr(block_table), stride, _ptr(kv_indptr), float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), _ws_bytes(workspace), _stream(stream))
    _raise(st, "mla_decode_fwd_dplan")


def combine_dplan(d: DPlan, out, lse, workspace, stream=None) -> None:
    """``mla_decode_combine_dplan``."""
    st = lib().mla_decode_combine_dplan(ctypes.byref(d), _ptr(workspace), _ws_bytes(workspace),
                                        _ptr(out), _ptr(lse), _stream(stream))
    _raise(st, "mla_decode_combine_dplan")


def dplan_check(d: DPlan, workspace, stream=None) -> int:
    """Device status bits of the last device-planned call (blocks until the stream drains)."""
    import torch
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    off = int(d.ws_status_offset)
    return int(workspace[off:off + 4].view(torch.int32).item())


def gather_kv_b_proj(kv_cache, kv_scale, block_table, seq_lens, cu_seqlens, max_ctx: int, w_kv_b,
                     k_out, v_out, status, stream=None) -> None:
    """``mla_gather_kv_b_proj``: k_out [T, H, 192], v_out [T, H, 128] bf16 from the
    paged latent and kv_b_proj w_kv_b [H, 256, 512] bf16."""
    import torch
    fp8 = kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    st = lib().mla_gather_kv_b_proj(
        _ptr(kv_cache), int(kv_cache.shape[0]), int(kv_cache.shape[1]),
        KV_FP8_E4M3 if fp8 else KV_BF16, _ptr(kv_scale), _ptr(block_table),
        int(block_table.stride(0)), _ptr(seq_lens), _ptr(cu_seqlens), int(seq_lens.numel()),
        int(max_ctx), _ptr(w_kv_b), int(w_kv_b.shape[0]), _ptr(k_out), _ptr(v_out), _ptr(status),
        _stream(stream))
    _raise(st, "mla_gather_kv_b_proj")


def epilogue(ql_nope, q_pe, kv_c, k_pe, slot_mapping, q_out, kv_cache, kv_scale=None,
             cache_inputs_early: bool = False, status=None, stream=None) -> None:
    """``mla_decode_epilogue``: q_out = ql_nope || q_pe; cache[slot] = kv_c || k_pe
    (bf16, or e4m3 codes of x / kv_scale for a uint8 / float8 cache)."""
    import torch
    T, H, _ = ql_nope.shape
    fp8 = kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    st = lib().mla_decode_epilogue(
        _ptr(ql_nope), _ptr(q_pe), _ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping), int(T), int(H),
        _ptr(q_out), _ptr(kv_cache), int(kv_cache.shape[0]), int(kv_cache.shape[1]),
        KV_FP8_E4M3 if fp8 else KV_BF16, _ptr(kv_scale), int(bool(cache_inputs_early)),
        _ptr(status), _stream(stream))
    _raise(st, "mla_decode_epilogue")


def step(p: Plan, ql_nope, q_pe, kv_c, k_pe, slot_mapping, q, kv_cache, kv_scale, block_table,
         seq_lens, softmax_scale: float, out, lse, workspace, cache_inputs_early: bool = False,
         stream=None) -> None:
    """``mla_decode_step``: epilogue, fwd and combine chained by programmatic launches."""
    st = lib().mla_decode_step(
        ctypes.byref(p), _ptr(ql_nope), _ptr(q_pe), _ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping),
        int(bool(cache_inputs_early)), _ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]),
        _ptr(kv_scale), _ptr(block_table), int(block_table.stride(0)), _ptr(seq_lens),
        float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream(stream))
    _raise(st, "mla_decode_step")


def check(p: Plan, workspace, stream=None) -> int:
    """``mla_decode_check``: device status bits (blocks until the stream drains)."""
    v = ctypes.c_int32(0)
    st = lib().mla_decode_check(ctypes.byref(p), _ptr(workspace), _stream(stream), ctypes.byref(v))
    if st not in (OK, ERR_DEVICE_CHECK, ERR_TIMEOUT):
        _raise(st, "mla_decode_check")
    return int(v.value)


def workspace_for(p: Plan, device="cuda"):
    import torch
    return torch.empty(max(int(p.workspace_bytes), 256), dtype=torch.uint8, device=device)


def decode(q, kv_cache, block_table, seq_lens, seq_lens_host=None, kv_scale=None,
           softmax_scale: float | None = None, causal: bool = False, p: Plan | None = None,
           workspace=None, stream=None):
    """plan + fwd + combine; returns (out bf16 [B,Sq,H,512], lse fp32 [B,Sq,H])."""
    import torch
    B, Sq, H, D = q.shape
    assert D == D_QK
    kv_dtype = KV_FP8_E4M3 if kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn) else KV_BF16
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(192.0)
    if p is None:
        host = seq_lens_host if seq_lens_host is not None else seq_lens.cpu()
        p = plan(host, H, Sq, int(kv_cache.shape[1]), kv_dtype, causal)
    if workspace is None:
        workspace = workspace_for(p, q.device)
    out = torch.empty((B, Sq, H, D_V), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Sq, H), dtype=torch.float32, device=q.device)
    fwd(p, q, kv_cache, kv_scale, block_table, seq_lens, softmax_scale, out, lse, workspace, stream)
    combine(p, seq_lens, out, lse, workspace, stream)
    return out, lse
