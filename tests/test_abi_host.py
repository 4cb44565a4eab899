"""The C-ABI library builds, loads, exports every declared symbol and validates
its arguments on the host (no GPU needed: every call here fails before any launch)."""
import ctypes
import os
import re

import pytest

from dynamic_sparse_attention_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_four_entry_points():
    names = _declared()
    for n in ("hip_select", "sparse_attn_decode", "vs_index_build", "sparse_attn_prefill"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, f"declared in include/dsa.h but not exported: {missing}"


def test_version_and_strerror(lib):
    assert lib.dsa_version() == 1
    assert lib.dsa_strerror(-3) == b"workspace missing or too small"


def _shape(**kw):
    d = dict(B=1, T_max=4096, T_q=1, H_q=32, H_kv=8, D=128, dtype=0)
    d.update(kw)
    return binding.DecodeShape(**d)


def _cfg(chunk=(256, 64, 16, 4), keep=(2048, 1024, 512, 256), n_sink=16, n_stream=64):
    return binding.HipConfig(chunk, keep, n_sink, n_stream).c()


@pytest.mark.parametrize("kw,status", [
    (dict(H_q=30), -1), (dict(D=96), -2), (dict(dtype=5), -2), (dict(B=0), -1),
    (dict(T_q=0), -1), (dict(H_q=256, H_kv=8), -2),
])
def test_bad_shapes_rejected(lib, kw, status):
    n = ctypes.c_size_t()
    s = _shape(**kw)
    c = _cfg()
    assert lib.hip_select_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == status
    assert lib.dsa_last_error()


@pytest.mark.parametrize("chunk,keep", [
    ((0,), (16,)), ((64,), (32,)), ((16, 16), (64, 128)), ((8192,), (8192,)),
])
def test_bad_configs_rejected(lib, chunk, keep):
    n = ctypes.c_size_t()
    s = _shape()
    c = _cfg(chunk, keep)
    assert lib.hip_select_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == -1


def test_workspace_sizes(lib):
    n = ctypes.c_size_t()
    s = _shape(T_max=1 << 20)
    c = _cfg(keep=(32768, 16384, 8192, 4096), n_sink=128, n_stream=1024)
    assert lib.hip_select_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == 0
    # scores for every stage + lists for the first three stages
    assert n.value >= 4 * (4092 + 512 + 1024 + 2048) + 4 * (32768 + 16384 + 8192)
    m = ctypes.c_int()
    assert lib.dsa_hip_max_chunks(ctypes.byref(s), ctypes.byref(c), 0, ctypes.byref(m)) == 0
    assert m.value == (1048576 - 128 - 1024 + 255) // 256
    # bf16 with <= 16 query rows per KV head: the cluster kernel merges in shared memory
    assert lib.sparse_attn_decode_workspace(ctypes.byref(s), 4096, 128, 1024, ctypes.byref(n)) == 0
    assert n.value == 0
    # fp32, or more than 16 rows per KV head: split-K partials in the workspace
    for kw in ({"dtype": 1}, {"T_q": 8}):
        s2 = _shape(T_max=1 << 20, **kw)
        assert lib.sparse_attn_decode_workspace(ctypes.byref(s2), 4096, 128, 1024, ctypes.byref(n)) == 0
        assert n.value > 0


def test_null_and_misaligned_pointers_rejected(lib):
    s = _shape()
    c = _cfg()
    buf = (ctypes.c_char * 64)()
    base = ctypes.addressof(buf)
    mis = ctypes.c_void_p(base + (1 if base % 16 else 2))
    ok = ctypes.c_void_p(base + (-base % 16))
    null = ctypes.c_void_p(0)
    # q NULL
    st = lib.hip_select(null, ok, ok, ctypes.byref(s), ctypes.byref(c), ok, ok, None, ok,
                        ctypes.c_size_t(1 << 30), None)
    assert st == -4
    # q misaligned
    st = lib.hip_select(mis, ok, ok, ctypes.byref(s), ctypes.byref(c), ok, ok, None, ok,
                        ctypes.c_size_t(1 << 30), None)
    assert st == -4
    # workspace too small
    st = lib.hip_select(ok, ok, ok, ctypes.byref(s), ctypes.byref(c), ok, ok, None, ok,
                        ctypes.c_size_t(8), None)
    assert st == -3
    st = lib.sparse_attn_decode(ok, ok, ok, ok, ok, ok, 16, 4, 4, ctypes.c_float(float("nan")),
                                ctypes.byref(s), ok, None, ok, ctypes.c_size_t(1 << 30), None)
    assert st == -1


def test_hip_select_cached_validates_the_refresh_mask(lib):
    s = _shape()
    c = _cfg()   # four stages
    buf = (ctypes.c_char * 64)()
    ok = ctypes.c_void_p(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 16))
    for mask in (1 << 4, 0xFFFFFFFF, 1 << 31):
        st = lib.hip_select_cached(ok, ok, ok, ctypes.byref(s), ctypes.byref(c),
                                   ctypes.c_uint32(mask), ok, ok, None, ok,
                                   ctypes.c_size_t(1 << 30), None)
        assert st == -1
        assert b"refresh mask" in lib.dsa_last_error()
    # a valid mask gets as far as the workspace check (no launch)
    st = lib.hip_select_cached(ok, ok, ok, ctypes.byref(s), ctypes.byref(c), ctypes.c_uint32(0b0110),
                               ok, ok, None, ok, ctypes.c_size_t(8), None)
    assert st == -3


def test_refresh_mask_helper():
    assert binding.refresh_mask(0, (16, 8, 4, 4)) == 0b1111
    assert binding.refresh_mask(4, (16, 8, 4, 4)) == 0b1100
    assert binding.refresh_mask(8, (16, 8, 4, 4)) == 0b1110
    assert binding.refresh_mask(5, (16, 8, 4, 4)) == 0
    assert binding.refresh_mask(48, (96, 24, 8, 8)) == 0b1110
    with pytest.raises(ValueError):
        binding.refresh_mask(3, (4, 0))


def _pshape(**kw):
    d = dict(B=1, S=4096, H_q=8, H_kv=2, D=128)
    d.update(kw)
    return binding.PrefillShape(**d)


def test_pattern_builders_validate_arguments(lib):
    s = _pshape()
    buf = (ctypes.c_char * 64)()
    ok = ctypes.c_void_p(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 16))
    # A-shape: token counts must be multiples of 64, max_blk must hold a row
    assert lib.ashape_index_build(ctypes.byref(s), 64, 100, 256, 64, ok, ok, ok, None) == -1
    assert lib.ashape_index_build(ctypes.byref(s), 64, 128, 256, 5, ok, ok, ok, None) == -1
    assert b"max_blk" in lib.dsa_last_error()
    assert lib.ashape_index_build(ctypes.byref(s), 32, 128, 256, 64, ok, ok, ok, None) == -2
    assert lib.ashape_index_build(ctypes.byref(s), 64, 128, 256, 6, None, ok, ok, None) == -4
    # Block-Sparse: workspace = pooled q and k in fp32
    n = ctypes.c_size_t()
    assert lib.block_sparse_index_build_workspace(ctypes.byref(s), 64, ctypes.byref(n)) == 0
    assert n.value >= 4 * 64 * 128 * (8 + 2)
    assert lib.block_sparse_index_build(ok, ok, ctypes.byref(s), 64, -1, 10, ok, ok, ok, None, ok,
                                        ctypes.c_size_t(1 << 30), None) == -1
    assert lib.block_sparse_index_build(ok, ok, ctypes.byref(s), 64, 100, 50, ok, ok, ok, None, ok,
                                        ctypes.c_size_t(1 << 30), None) == -1
    assert lib.block_sparse_index_build(ok, ok, ctypes.byref(s), 64, 10, 10, ok, ok, ok, None, ok,
                                        ctypes.c_size_t(16), None) == -3
    big = _pshape(S=4 << 20)
    assert lib.block_sparse_index_build(ok, ok, ctypes.byref(big), 64, 10, 10, ok, ok, ok, None, ok,
                                        ctypes.c_size_t(1 << 40), None) == -2


def test_mixed_patterns_validate_arguments(lib):
    s = _pshape(H_q=4, H_kv=2)
    n = ctypes.c_size_t()

    def cfg(pats, **kw):
        arr = (ctypes.c_uint8 * len(pats))(*pats)
        c = binding.MixedCfg(ctypes.cast(arr, ctypes.c_void_p), binding.VsCfg(64, 100, 200, 64),
                             kw.get("n_global", 1024), kw.get("n_local", 4096), kw.get("k_b", 100))
        return c, arr

    c, keep = cfg([1, 1, 1, 1])
    assert lib.mixed_index_build_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == 0
    assert n.value == 0                      # A-shape heads need no scratch
    c, keep = cfg([2, 1, 1, 1])
    assert lib.mixed_index_build_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == 0
    assert n.value >= 4 * 64 * 128 * 6       # pooled q and k
    c, keep = cfg([0, 1, 2, 3])
    assert lib.mixed_index_build_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == -1
    c, keep = cfg([1, 1, 0, 0], n_global=100)
    assert lib.mixed_index_build_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == -1
    c, keep = cfg([0, 0, 0, 0], n_global=100)  # A-shape settings unused: fine
    assert lib.mixed_index_build_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == 0
    big = _pshape(H_q=512, H_kv=8)
    c, keep = cfg([1] * 512)
    assert lib.mixed_index_build_workspace(ctypes.byref(big), ctypes.byref(c), ctypes.byref(n)) == -2


def test_fp8_kv_shapes(lib):
    n = ctypes.c_size_t()
    c = _cfg()
    # bf16 queries over FP8 keys / values: D = 128 only, at most 16 rows per KV head
    s = _shape(dtype=2)
    assert lib.hip_select_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == 0
    assert lib.sparse_attn_decode_workspace(ctypes.byref(s), 4096, 128, 1024, ctypes.byref(n)) == 0
    assert n.value == 0                        # the cluster kernel needs no scratch
    s = _shape(dtype=2, D=64)
    assert lib.hip_select_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == -2
    s = _shape(dtype=2, T_q=8)                 # 4 heads per KV head x 8 rows = 32 > 16
    assert lib.sparse_attn_decode_workspace(ctypes.byref(s), 4096, 128, 1024, ctypes.byref(n)) == -2
    assert b"FP8" in lib.dsa_last_error()
    s = _shape(dtype=3)
    assert lib.hip_select_workspace(ctypes.byref(s), ctypes.byref(c), ctypes.byref(n)) == -2


def test_prefill_rejects_a_non_positive_scale(lib):
    """The prefill kernel orders scores by their raw value: scale <= 0 is an argument
    error, rejected before any launch (there is no second kernel to fall back to)."""
    s = _pshape()
    buf = (ctypes.c_char * 64)()
    ok = ctypes.c_void_p(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 16))
    for bad in (0.0, -1.0, float("inf")):
        st = lib.sparse_attn_prefill(ok, ok, ok, ctypes.byref(s), 64, 4, 4, ok, ok, ok, ok,
                                     ctypes.c_float(bad), ok, None, None)
        assert st == -1
        assert b"scale" in lib.dsa_last_error()
