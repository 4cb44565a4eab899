"""ctypes binding of libdsa.so: argument marshalling only.

Every step of the hot path runs in the CUDA kernels behind the C ABI
(``include/dsa.h``).  This module turns torch CUDA tensors into device
pointers, allocates the scratch workspace the library asks for (unless the
caller passes one) and forwards the current torch stream.  There is no CPU
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import _build

MAX_STAGES = 8
BF16, F32, BF16_FP8KV = 0, 1, 2   # dsa_dtype

_c_int = ctypes.c_int
_vp = ctypes.c_void_p


class DecodeShape(ctypes.Structure):
    _fields_ = [("B", _c_int), ("T_max", _c_int), ("T_q", _c_int), ("H_q", _c_int),
                ("H_kv", _c_int), ("D", _c_int), ("dtype", _c_int)]


class HipCfg(ctypes.Structure):
    _fields_ = [("n_stages", _c_int), ("chunk", _c_int * MAX_STAGES),
                ("keep", _c_int * MAX_STAGES), ("n_sink", _c_int), ("n_stream", _c_int)]


class HipDebug(ctypes.Structure):
    _fields_ = [("stage_idx", _vp * MAX_STAGES), ("stage_cnt", _vp * MAX_STAGES),
                ("chunk_score", _vp * MAX_STAGES), ("rep", _vp * MAX_STAGES),
                ("rep_score", _vp * MAX_STAGES)]


class PrefillShape(ctypes.Structure):
    _fields_ = [("B", _c_int), ("S", _c_int), ("H_q", _c_int), ("H_kv", _c_int), ("D", _c_int)]


class VsCfg(ctypes.Structure):
    _fields_ = [("last_q", _c_int), ("n_vertical", _c_int), ("n_slash", _c_int), ("block", _c_int)]


class VsDebug(ctypes.Structure):
    _fields_ = [("vsum", _vp), ("ssum", _vp)]


class MixedCfg(ctypes.Structure):
    _fields_ = [("head_pattern", _vp), ("vs", VsCfg), ("n_global", _c_int), ("n_local", _c_int),
                ("k_b", _c_int)]


PATTERN_VERTICAL_SLASH, PATTERN_A_SHAPE, PATTERN_BLOCK_SPARSE = 0, 1, 2
_PATTERN_NAMES = {"vertical_slash": 0, "vs": 0, "a_shape": 1, "block_sparse": 2}


class BsDebug(ctypes.Structure):
    _fields_ = [("q_pool", _vp), ("k_pool", _vp), ("scores", _vp)]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", _c_int), ("total_ms", ctypes.c_double)]


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


_lib = None

# name -> (restype, argtypes)
_SIGNATURES = {
    "dsa_version": (_c_int, []),
    "dsa_last_error": (ctypes.c_char_p, []),
    "dsa_strerror": (ctypes.c_char_p, [_c_int]),
    "dsa_hip_max_chunks": (_c_int, [_vp, _vp, _c_int, ctypes.POINTER(_c_int)]),
    "hip_select_workspace": (_c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_size_t)]),
    "hip_select": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "hip_select_cached": (_c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_uint32, _vp, _vp, _vp, _vp,
                                   ctypes.c_size_t, _vp]),
    "sparse_attn_decode_workspace": (_c_int, [_vp, _c_int, _c_int, _c_int,
                                              ctypes.POINTER(ctypes.c_size_t)]),
    "sparse_attn_decode": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                    ctypes.c_float, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "vs_index_build_workspace": (_c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_size_t)]),
    "vs_index_build": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                ctypes.c_size_t, _vp]),
    "ashape_index_build": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp]),
    "block_sparse_index_build_workspace": (_c_int, [_vp, _c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "block_sparse_index_build": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                          _vp, _vp, ctypes.c_size_t, _vp]),
    "mixed_index_build_workspace": (_c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_size_t)]),
    "mixed_index_build": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                   _vp]),
    "dsa_hip_prefill_max_chunks": (_c_int, [_vp, _vp, _c_int, ctypes.POINTER(_c_int)]),
    "hip_prefill_select_workspace": (_c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_size_t)]),
    "hip_prefill_select": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "hip_prefill_lists": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp]),
    "sparse_attn_prefill": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                     _vp, ctypes.c_float, _vp, _vp, _vp]),
    "sparse_attn_decode_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                            ctypes.c_float, _vp, _vp, _vp, _vp]),
    "dsa_device_error": (_c_int, [ctypes.POINTER(_c_int)]),
    "dsa_set_wait_limit": (_c_int, [ctypes.c_ulonglong]),
    "dsa_profile_enable": (_c_int, [_c_int]),
    "dsa_profile_collect": (_c_int, [_vp, _c_int, ctypes.POINTER(_c_int)]),
}


def device_error() -> int:
    """Read and clear the library's device error words: 0 = none; bit 0 / bit 1: a
    prefill-attention / vertical-slash-estimate CTA gave up a wait; bit 2 (checked
    build): a kernel met out-of-range device-side input."""
    lib = load()
    c = _c_int()
    st = lib.dsa_device_error(ctypes.byref(c))
    if st == -6:   # DSA_ERR_DEVICE_CHECK: the code says what was met
        return c.value
    _check("dsa_device_error", st)
    return c.value


def set_wait_limit(ns: int = 0) -> None:
    """Limit of the tensor-core kernels' bounded waits in nanoseconds (0: the default)."""
    lib = load()
    _check("dsa_set_wait_limit", lib.dsa_set_wait_limit(ctypes.c_ulonglong(ns)))


def profile_enable(on: bool = True) -> None:
    """Bracket every library kernel launch with CUDA events on its stream."""
    load().dsa_profile_enable(1 if on else 0)


def profile_collect() -> dict:
    """Wait for the recorded events; {kernel name: (launches, total ms)}, then clear."""
    lib = load()
    buf = (KernelStat * 64)()
    n = _c_int()
    _check("dsa_profile_collect", lib.dsa_profile_collect(buf, 64, ctypes.byref(n)))
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(min(n.value, 64))}


def library_path() -> str:
    """Path of the library this process loads (the checked build with DSA_CHECKED=1)."""
    return _build.LIB_CHECKED if os.environ.get("DSA_CHECKED") == "1" else _build.LIB


def load(build_if_missing: bool = False):
    """Load libdsa.so (building it first if asked and absent).  With DSA_CHECKED=1 in
    the environment at the first call, the checked build libdsa_checked.so instead (the
    same kernels with device-side input checks compiled in)."""
    global _lib
    if _lib is not None:
        return _lib
    checked = os.environ.get("DSA_CHECKED") == "1"
    path = _build.LIB_CHECKED if checked else _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"{os.path.basename(path)} not built ({path}); run __graft_entry__.build()")
        _build.build(checked=checked)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name, None)
        if fn is None:
            continue  # reported by exported_symbols(); calling it raises AttributeError
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols() -> dict:
    """Which C entry points of the binding the loaded library exports."""
    lib = load()
    return {name: hasattr(lib, name) for name in _SIGNATURES}


def _check(fn: str, status: int):
    if status != 0:
        msg = _lib.dsa_last_error().decode(errors="replace")
        raise DsaError(fn, status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _workspace(nbytes: int, device, ws):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError(f"workspace too small: {nbytes} bytes needed")
        return ws
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- decode

@dataclass
class HipConfig:
    chunk: tuple
    keep: tuple
    n_sink: int
    n_stream: int

    def c(self) -> HipCfg:
        cfg = HipCfg()
        cfg.n_stages = len(self.chunk)
        for i, (c, k) in enumerate(zip(self.chunk, self.keep)):
            cfg.chunk[i] = int(c)
            cfg.keep[i] = int(k)
        cfg.n_sink = int(self.n_sink)
        cfg.n_stream = int(self.n_stream)
        return cfg


def _is_fp8(t: torch.Tensor) -> bool:
    return t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None)


def decode_shape(q: torch.Tensor, k: torch.Tensor) -> DecodeShape:
    """q bf16 / fp32 with k of the same type, or q bf16 with k FP8 E4M3 (a uint8 or
    float8_e4m3fn tensor of codes)."""
    B, T_q, H_q, D = q.shape
    T_max, H_kv = k.shape[1], k.shape[2]
    if _is_fp8(k):
        if q.dtype != torch.bfloat16:
            raise TypeError("FP8 keys and values need a bfloat16 query")
        return DecodeShape(B, T_max, T_q, H_q, H_kv, D, BF16_FP8KV)
    if k.dtype != q.dtype:
        raise TypeError(f"k ({k.dtype}) must have the type of q ({q.dtype})")
    return DecodeShape(B, T_max, T_q, H_q, H_kv, D, _dtype_code(q))


def hip_select_workspace_bytes(q, k, cfg: HipConfig) -> int:
    lib = load()
    n = ctypes.c_size_t()
    shape, c = decode_shape(q, k), cfg.c()
    _check("hip_select_workspace", lib.hip_select_workspace(ctypes.byref(shape), ctypes.byref(c),
                                                             ctypes.byref(n)))
    return n.value


def hip_max_chunks(q, k, cfg: HipConfig, stage: int) -> int:
    lib = load()
    n = _c_int()
    shape, c = decode_shape(q, k), cfg.c()
    _check("dsa_hip_max_chunks", lib.dsa_hip_max_chunks(ctypes.byref(shape), ctypes.byref(c),
                                                         stage, ctypes.byref(n)))
    return n.value


def hip_select(q, k, kv_len, cfg: HipConfig, *, debug: bool = False, out=None, workspace=None,
               stream=None):
    """Run all pruning stages; returns (sel_idx [B, keep[-1]], sel_cnt [B][, debug dict])."""
    return _hip_select(q, k, kv_len, cfg, None, debug, out, workspace, stream)


def hip_select_cached(q, k, kv_len, cfg: HipConfig, refresh: int, *, out, workspace,
                      debug: bool = False, stream=None):
    """Recompute only the pruning stages whose bit is set in `refresh` (InfiniteHiP,
    section 3.4 "Sparse Attention Mask Caching"); the others keep the lists they left in
    `workspace` / `out` on an earlier call, so both must persist between calls.
    Returns like hip_select (debug tensors of skipped stages stay at their fill)."""
    if out is None or workspace is None:
        raise ValueError("hip_select_cached needs the persistent out buffers and workspace")
    return _hip_select(q, k, kv_len, cfg, int(refresh), debug, out, workspace, stream)


def refresh_mask(step: int, n_refresh) -> int:
    """Stages to recompute at decoding step `step` (counted from 0) when stage i is
    refreshed every n_refresh[i] steps (InfiniteHiP, section 3.4): bit i is set iff
    step % n_refresh[i] == 0, so step 0 recomputes every stage."""
    m = 0
    for i, r in enumerate(n_refresh):
        if int(r) <= 0:
            raise ValueError("refresh intervals must be positive")
        if step % int(r) == 0:
            m |= 1 << i
    return m


class HipSelectCache:
    """Decoding-loop helper for mask caching: owns the workspace and the selection
    buffers, keeps the step counter and recomputes, on each call, the stages whose
    refresh interval divides it.  Shapes and config are fixed at construction."""

    def __init__(self, q, k, cfg: HipConfig, n_refresh):
        if len(n_refresh) != len(cfg.chunk):
            raise ValueError("one refresh interval per pruning stage")
        refresh_mask(0, n_refresh)
        self.cfg = cfg
        self.n_refresh = tuple(int(r) for r in n_refresh)
        B = q.shape[0]
        self.sel_idx = torch.empty(B, cfg.keep[-1], dtype=torch.int32, device=q.device)
        self.sel_cnt = torch.empty(B, dtype=torch.int32, device=q.device)
        self.workspace = _workspace(hip_select_workspace_bytes(q, k, cfg), q.device, None)
        self.step = 0

    def mask(self, step=None) -> int:
        return refresh_mask(self.step if step is None else step, self.n_refresh)

    def __call__(self, q, k, kv_len, *, debug: bool = False, stream=None):
        m = self.mask()
        self.step += 1
        return hip_select_cached(q, k, kv_len, self.cfg, m, out=(self.sel_idx, self.sel_cnt),
                                 workspace=self.workspace, debug=debug, stream=stream)


def _hip_select(q, k, kv_len, cfg, refresh, debug, out, workspace, stream):
    lib = load()
    _need_cuda(q, k, kv_len)
    shape, c = decode_shape(q, k), cfg.c()
    B = shape.B
    dev = q.device
    if out is None:
        sel_idx = torch.empty(B, cfg.keep[-1], dtype=torch.int32, device=dev)
        sel_cnt = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        sel_idx, sel_cnt = out
    dbg = None
    dbg_t = None
    if debug:
        dbg = HipDebug()
        dbg_t = {"stage_idx": [], "stage_cnt": [], "chunk_score": [], "rep": [], "rep_score": []}
        for i in range(len(cfg.chunk)):
            mc = hip_max_chunks(q, k, cfg, i)
            t = {
                "stage_idx": torch.full((B, cfg.keep[i]), -7, dtype=torch.int32, device=dev),
                "stage_cnt": torch.full((B,), -7, dtype=torch.int32, device=dev),
                "chunk_score": torch.full((B, max(mc, 1)), float("nan"), device=dev),
                "rep": torch.full((B, shape.H_q, max(mc, 1)), -7, dtype=torch.int32, device=dev),
                "rep_score": torch.full((B, shape.H_q, max(mc, 1)), float("nan"), device=dev),
            }
            for key, v in t.items():
                dbg_t[key].append(v)
                getattr(dbg, key)[i] = v.data_ptr()
    nbytes = hip_select_workspace_bytes(q, k, cfg)
    ws = _workspace(nbytes, dev, workspace)
    dbg_p = ctypes.byref(dbg) if dbg else None
    if refresh is None:
        st = lib.hip_select(_ptr(q), _ptr(k), _ptr(kv_len), ctypes.byref(shape), ctypes.byref(c),
                            _ptr(sel_idx), _ptr(sel_cnt), dbg_p, _ptr(ws),
                            ctypes.c_size_t(ws.numel()), _stream(stream))
    else:
        st = lib.hip_select_cached(_ptr(q), _ptr(k), _ptr(kv_len), ctypes.byref(shape),
                                   ctypes.byref(c), refresh, _ptr(sel_idx), _ptr(sel_cnt),
                                   dbg_p, _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    _check("hip_select" if refresh is None else "hip_select_cached", st)
    if debug:
        return sel_idx, sel_cnt, dbg_t
    return sel_idx, sel_cnt


def sparse_attn_decode_workspace_bytes(q, k, max_sel: int, n_sink: int, n_stream: int) -> int:
    lib = load()
    n = ctypes.c_size_t()
    shape = decode_shape(q, k)
    _check("sparse_attn_decode_workspace",
           lib.sparse_attn_decode_workspace(ctypes.byref(shape), max_sel, n_sink, n_stream,
                                            ctypes.byref(n)))
    return n.value


def sparse_attn_decode(q, k, v, kv_len, sel_idx, sel_cnt, *, n_sink: int, n_stream: int,
                       scale: float | None = None, out=None, lse=None, want_lse: bool = True,
                       workspace=None, stream=None):
    """Attention over sink + selected + window keys; returns (out, lse or None)."""
    lib = load()
    _need_cuda(q, k, v, kv_len, sel_idx, sel_cnt)
    shape = decode_shape(q, k)
    max_sel = sel_idx.shape[1] if sel_idx is not None else 0
    if scale is None:
        scale = shape.D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(shape.B, shape.T_q, shape.H_q, dtype=torch.float32, device=q.device)
    nbytes = sparse_attn_decode_workspace_bytes(q, k, max_sel, n_sink, n_stream)
    ws = _workspace(nbytes, q.device, workspace)
    st = lib.sparse_attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_len), _ptr(sel_idx),
                                _ptr(sel_cnt), max_sel, n_sink, n_stream, ctypes.c_float(scale),
                                ctypes.byref(shape), _ptr(out), _ptr(lse), _ptr(ws),
                                ctypes.c_size_t(ws.numel()), _stream(stream))
    _check("sparse_attn_decode", st)
    return out, lse


def sparse_attn_decode_noalloc(q, k, v, kv_len, sel_idx, sel_cnt, *, n_sink: int, n_stream: int,
                               scale: float | None = None, out=None, lse=None,
                               want_lse: bool = True, stream=None):
    """sparse_attn_decode whose split-K scratch is the library's built-in device array.

    For callers that must not allocate device memory when they call: nothing is
    allocated here either when `out` (and `lse`, or want_lse=False) are given.
    Calls that overlap on the GPU share the one array and must be serialised.
    """
    lib = load()
    _need_cuda(q, k, v, kv_len, sel_idx, sel_cnt)
    shape = decode_shape(q, k)
    max_sel = sel_idx.shape[1] if sel_idx is not None else 0
    if scale is None:
        scale = shape.D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(shape.B, shape.T_q, shape.H_q, dtype=torch.float32, device=q.device)
    st = lib.sparse_attn_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_len), _ptr(sel_idx),
                                        _ptr(sel_cnt), max_sel, n_sink, n_stream,
                                        ctypes.c_float(scale), ctypes.byref(shape), _ptr(out),
                                        _ptr(lse), _stream(stream))
    _check("sparse_attn_decode_noalloc", st)
    return out, lse


# ----------------------------------------------------------------------------- prefill

def prefill_shape(q: torch.Tensor, k: torch.Tensor) -> PrefillShape:
    B, S, H_q, D = q.shape
    return PrefillShape(B, S, H_q, k.shape[2], D)


def vs_index_build_workspace_bytes(q, k, last_q, n_vertical, n_slash, block=64) -> int:
    lib = load()
    n = ctypes.c_size_t()
    shape = prefill_shape(q, k)
    cfg = VsCfg(last_q, n_vertical, n_slash, block)
    _check("vs_index_build_workspace",
           lib.vs_index_build_workspace(ctypes.byref(shape), ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def vs_index_build(q, k, *, last_q: int = 64, n_vertical: int, n_slash: int, block: int = 64,
                   debug: bool = False, out: dict | None = None, workspace=None, stream=None):
    """Vertical-slash index and its tile/column lists; returns a dict of tensors."""
    lib = load()
    _need_cuda(q, k)
    shape = prefill_shape(q, k)
    B, S, H_q = shape.B, shape.S, shape.H_q
    nq = (S + block - 1) // block
    dev = q.device
    if out is None:
        out = {
            "vertical": torch.empty(B, H_q, n_vertical, dtype=torch.int32, device=dev),
            "slash": torch.empty(B, H_q, n_slash, dtype=torch.int32, device=dev),
            "blk_cnt": torch.empty(B, H_q, nq, dtype=torch.int32, device=dev),
            "blk_idx": torch.empty(B, H_q, nq, nq, dtype=torch.int32, device=dev),
            "col_cnt": torch.empty(B, H_q, nq, dtype=torch.int32, device=dev),
            "col_idx": torch.empty(B, H_q, nq, max(n_vertical, 1), dtype=torch.int32, device=dev),
        }
    dbg = None
    if debug:
        out["vsum"] = torch.empty(B, H_q, S, dtype=torch.float32, device=dev)
        out["ssum"] = torch.empty(B, H_q, S, dtype=torch.float32, device=dev)
        dbg = VsDebug(out["vsum"].data_ptr(), out["ssum"].data_ptr())
    cfg = VsCfg(last_q, n_vertical, n_slash, block)
    ws = _workspace(vs_index_build_workspace_bytes(q, k, last_q, n_vertical, n_slash, block),
                    dev, workspace)
    st = lib.vs_index_build(_ptr(q), _ptr(k), ctypes.byref(shape), ctypes.byref(cfg),
                            _ptr(out["vertical"]), _ptr(out["slash"]), _ptr(out["blk_cnt"]),
                            _ptr(out["blk_idx"]), _ptr(out["col_cnt"]), _ptr(out["col_idx"]),
                            ctypes.byref(dbg) if dbg else None, _ptr(ws),
                            ctypes.c_size_t(ws.numel()), _stream(stream))
    _check("vs_index_build", st)
    return out


def _block_lists(B, H_q, nq, max_blk, dev, out):
    if out is None:
        out = {
            "blk_cnt": torch.empty(B, H_q, nq, dtype=torch.int32, device=dev),
            "blk_idx": torch.empty(B, H_q, nq, max(max_blk, 1), dtype=torch.int32, device=dev),
            "col_cnt": torch.empty(B, H_q, nq, dtype=torch.int32, device=dev),
        }
    out.setdefault("col_idx", None)
    return out


def ashape_index_build(q, k, *, n_global: int, n_local: int, block: int = 64, max_blk=None,
                       out: dict | None = None, stream=None):
    """A-shape lists (initial blocks + a band ending at the diagonal); q and k give the
    shape only.  Returns a dict with blk_cnt, blk_idx, col_cnt (all 0), col_idx None."""
    lib = load()
    shape = prefill_shape(q, k)
    nq = (shape.S + block - 1) // block
    if max_blk is None:
        max_blk = min(nq, n_global // block + n_local // block)
    out = _block_lists(shape.B, shape.H_q, nq, max_blk, q.device, out)
    _need_cuda(out["blk_cnt"], out["blk_idx"], out["col_cnt"])
    st = lib.ashape_index_build(ctypes.byref(shape), block, n_global, n_local,
                                out["blk_idx"].shape[-1], _ptr(out["blk_cnt"]),
                                _ptr(out["blk_idx"]), _ptr(out["col_cnt"]), _stream(stream))
    _check("ashape_index_build", st)
    return out


def block_sparse_index_build_workspace_bytes(q, k, block: int = 64) -> int:
    lib = load()
    n = ctypes.c_size_t()
    shape = prefill_shape(q, k)
    _check("block_sparse_index_build_workspace",
           lib.block_sparse_index_build_workspace(ctypes.byref(shape), block, ctypes.byref(n)))
    return n.value


def block_sparse_index_build(q, k, *, k_b: int, block: int = 64, max_blk=None,
                             debug: bool = False, out: dict | None = None, workspace=None,
                             stream=None):
    """Block-Sparse lists (mean-pooled block attention, top-k_b key blocks per query
    block).  Returns a dict with blk_cnt, blk_idx, col_cnt (all 0), col_idx None and,
    with debug, the pooled blocks and the block logits."""
    lib = load()
    _need_cuda(q, k)
    shape = prefill_shape(q, k)
    B, S, H_q = shape.B, shape.S, shape.H_q
    nq = (S + block - 1) // block
    if max_blk is None:
        max_blk = min(k_b, nq)
    out = _block_lists(B, H_q, nq, max_blk, q.device, out)
    dbg = None
    if debug:
        dev = q.device
        out["q_pool"] = torch.empty(B, H_q, nq, shape.D, dtype=torch.float32, device=dev)
        out["k_pool"] = torch.empty(B, shape.H_kv, nq, shape.D, dtype=torch.float32, device=dev)
        out["scores"] = torch.full((B, H_q, nq, nq), float("nan"), dtype=torch.float32, device=dev)
        dbg = BsDebug(out["q_pool"].data_ptr(), out["k_pool"].data_ptr(),
                      out["scores"].data_ptr())
    ws = _workspace(block_sparse_index_build_workspace_bytes(q, k, block), q.device, workspace)
    st = lib.block_sparse_index_build(_ptr(q), _ptr(k), ctypes.byref(shape), block, k_b,
                                      out["blk_idx"].shape[-1], _ptr(out["blk_cnt"]),
                                      _ptr(out["blk_idx"]), _ptr(out["col_cnt"]),
                                      ctypes.byref(dbg) if dbg else None, _ptr(ws),
                                      ctypes.c_size_t(ws.numel()), _stream(stream))
    _check("block_sparse_index_build", st)
    return out


def _mixed_cfg(H_q, head_pattern, last_q, n_vertical, n_slash, n_global, n_local, k_b, block):
    pats = [(_PATTERN_NAMES[p] if isinstance(p, str) else int(p)) for p in head_pattern]
    if len(pats) != H_q:
        raise ValueError(f"head_pattern needs {H_q} entries, got {len(pats)}")
    arr = (ctypes.c_uint8 * H_q)(*pats)
    cfg = MixedCfg(ctypes.cast(arr, _vp), VsCfg(last_q, n_vertical, n_slash, block), n_global,
                   n_local, k_b)
    return cfg, arr, pats


def mixed_index_build(q, k, *, head_pattern, last_q: int = 64, n_vertical: int = 1000,
                      n_slash: int = 6096, n_global: int = 1024, n_local: int = 4096,
                      k_b: int = 100, block: int = 64, out: dict | None = None, workspace=None,
                      stream=None):
    """Per-head patterns (head_pattern: one of "vertical_slash", "a_shape",
    "block_sparse" or 0/1/2 per query head) into one set of tile/column lists."""
    lib = load()
    _need_cuda(q, k)
    shape = prefill_shape(q, k)
    B, S, H_q = shape.B, shape.S, shape.H_q
    cfg, arr, pats = _mixed_cfg(H_q, head_pattern, last_q, n_vertical, n_slash, n_global,
                                n_local, k_b, block)
    nq = (S + block - 1) // block
    dev = q.device
    if out is None:
        out = {
            "blk_cnt": torch.empty(B, H_q, nq, dtype=torch.int32, device=dev),
            "blk_idx": torch.empty(B, H_q, nq, nq, dtype=torch.int32, device=dev),
            "col_cnt": torch.empty(B, H_q, nq, dtype=torch.int32, device=dev),
            "col_idx": torch.empty(B, H_q, nq, max(n_vertical, 1), dtype=torch.int32, device=dev),
        }
    n = ctypes.c_size_t()
    _check("mixed_index_build_workspace",
           lib.mixed_index_build_workspace(ctypes.byref(shape), ctypes.byref(cfg), ctypes.byref(n)))
    ws = _workspace(n.value, dev, workspace)
    st = lib.mixed_index_build(_ptr(q), _ptr(k), ctypes.byref(shape), ctypes.byref(cfg),
                               _ptr(out["blk_cnt"]), _ptr(out["blk_idx"]), _ptr(out["col_cnt"]),
                               _ptr(out["col_idx"]), _ptr(ws), ctypes.c_size_t(ws.numel()),
                               _stream(stream))
    del arr
    _check("mixed_index_build", st)
    return out


def mixed_index_build_workspace_bytes(q, k, *, head_pattern, last_q: int = 64,
                                      n_vertical: int = 1000, n_slash: int = 6096,
                                      n_global: int = 1024, n_local: int = 4096, k_b: int = 100,
                                      block: int = 64) -> int:
    lib = load()
    shape = prefill_shape(q, k)
    cfg, arr, _ = _mixed_cfg(shape.H_q, head_pattern, last_q, n_vertical, n_slash, n_global,
                             n_local, k_b, block)
    n = ctypes.c_size_t()
    _check("mixed_index_build_workspace",
           lib.mixed_index_build_workspace(ctypes.byref(shape), ctypes.byref(cfg), ctypes.byref(n)))
    del arr
    return n.value


def hip_prefill_max_chunks(q, k, cfg: HipConfig, stage: int) -> int:
    lib = load()
    n = _c_int()
    shape, c = prefill_shape(q, k), cfg.c()
    _check("dsa_hip_prefill_max_chunks",
           lib.dsa_hip_prefill_max_chunks(ctypes.byref(shape), ctypes.byref(c), stage, ctypes.byref(n)))
    return n.value


def hip_prefill_select_workspace_bytes(q, k, cfg: HipConfig) -> int:
    lib = load()
    n = ctypes.c_size_t()
    shape, c = prefill_shape(q, k), cfg.c()
    _check("hip_prefill_select_workspace",
           lib.hip_prefill_select_workspace(ctypes.byref(shape), ctypes.byref(c), ctypes.byref(n)))
    return n.value


def hip_prefill_select(q, k, cfg: HipConfig, *, debug: bool = False, out=None, workspace=None,
                       stream=None):
    """InfiniteHiP pruning for every 64-row query block of a causal prefill; returns
    (sel_idx [B * n_qblk, keep[-1]], sel_cnt [B * n_qblk][, debug dict]), rows ordered
    b * n_qblk + m."""
    lib = load()
    _need_cuda(q, k)
    shape, c = prefill_shape(q, k), cfg.c()
    R = shape.B * ((shape.S + 63) // 64)
    dev = q.device
    if out is None:
        sel_idx = torch.empty(R, cfg.keep[-1], dtype=torch.int32, device=dev)
        sel_cnt = torch.empty(R, dtype=torch.int32, device=dev)
    else:
        sel_idx, sel_cnt = out
    dbg = dbg_t = None
    if debug:
        dbg = HipDebug()
        dbg_t = {"stage_idx": [], "stage_cnt": [], "chunk_score": [], "rep": [], "rep_score": []}
        for i in range(len(cfg.chunk)):
            mc = max(hip_prefill_max_chunks(q, k, cfg, i), 1)
            t = {
                "stage_idx": torch.full((R, cfg.keep[i]), -7, dtype=torch.int32, device=dev),
                "stage_cnt": torch.full((R,), -7, dtype=torch.int32, device=dev),
                "chunk_score": torch.full((R, mc), float("nan"), device=dev),
                "rep": torch.full((R, shape.H_q, mc), -7, dtype=torch.int32, device=dev),
                "rep_score": torch.full((R, shape.H_q, mc), float("nan"), device=dev),
            }
            for key, v in t.items():
                dbg_t[key].append(v)
                getattr(dbg, key)[i] = v.data_ptr()
    ws = _workspace(hip_prefill_select_workspace_bytes(q, k, cfg), dev, workspace)
    st = lib.hip_prefill_select(_ptr(q), _ptr(k), ctypes.byref(shape), ctypes.byref(c),
                                _ptr(sel_idx), _ptr(sel_cnt), ctypes.byref(dbg) if dbg else None,
                                _ptr(ws), ctypes.c_size_t(ws.numel()), _stream(stream))
    _check("hip_prefill_select", st)
    if debug:
        return sel_idx, sel_cnt, dbg_t
    return sel_idx, sel_cnt


def hip_prefill_lists(q, k, cfg: HipConfig, sel_idx, sel_cnt, *, out: dict | None = None,
                      stream=None):
    """Each query block's sink + selection + window as sparse_attn_prefill lists (the
    same for every head); returns a dict with blk_cnt, blk_idx, col_cnt, col_idx."""
    lib = load()
    _need_cuda(sel_idx, sel_cnt)
    shape, c = prefill_shape(q, k), cfg.c()
    nq = (shape.S + 63) // 64
    max_blk = -(-cfg.n_sink // 64) + -(-cfg.n_stream // 64) + 2
    max_col = cfg.keep[-1] + 126
    dev = sel_idx.device
    if out is None:
        out = {
            "blk_cnt": torch.empty(shape.B, shape.H_q, nq, dtype=torch.int32, device=dev),
            "blk_idx": torch.empty(shape.B, shape.H_q, nq, max_blk, dtype=torch.int32, device=dev),
            "col_cnt": torch.empty(shape.B, shape.H_q, nq, dtype=torch.int32, device=dev),
            "col_idx": torch.empty(shape.B, shape.H_q, nq, max_col, dtype=torch.int32, device=dev),
        }
    st = lib.hip_prefill_lists(ctypes.byref(shape), ctypes.byref(c), _ptr(sel_idx), _ptr(sel_cnt),
                               out["blk_idx"].shape[-1], out["col_idx"].shape[-1],
                               _ptr(out["blk_cnt"]), _ptr(out["blk_idx"]), _ptr(out["col_cnt"]),
                               _ptr(out["col_idx"]), _stream(stream))
    _check("hip_prefill_lists", st)
    return out


def sparse_attn_prefill(q, k, v, blk_cnt, blk_idx, col_cnt, col_idx, *, scale=None,
                        block: int = 64, out=None, lse=None, want_lse: bool = True, stream=None):
    """Causal attention over the listed tiles and columns (col_idx None: no columns);
    returns (out, lse or None)."""
    lib = load()
    _need_cuda(q, k, v, blk_cnt, blk_idx, col_cnt, col_idx)
    shape = prefill_shape(q, k)
    if scale is None:
        scale = shape.D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(shape.B, shape.H_q, shape.S, dtype=torch.float32, device=q.device)
    st = lib.sparse_attn_prefill(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(shape), block,
                                 blk_idx.shape[-1], 0 if col_idx is None else col_idx.shape[-1],
                                 _ptr(blk_cnt),
                                 _ptr(blk_idx), _ptr(col_cnt), _ptr(col_idx),
                                 ctypes.c_float(scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("sparse_attn_prefill", st)
    return out, lse
