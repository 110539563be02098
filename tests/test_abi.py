"""CPU checks of the C-ABI library: it builds, loads, exports every declared symbol, and its
host-side logic (shape checks, sizes, argument validation) answers without a GPU."""
import ctypes
import os
import re

import pytest

from quantized_grouped_gemm_gb300 import _lib, build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_path_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_grouped_ffn", "moe_combine", "moe_forward", "moe_pack_weights"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(names) == set(_lib.exported_symbols())


def test_shape_checks(lib):
    ok = _lib.moe_shape(512, 2048, 256, 8, 512, 512, 64)
    assert lib.moe_check_shape(ctypes.byref(ok)) == _lib.MOE_OK
    for bad, rc in [((512, 2048, 128, 8, 512, 512, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((512, 2000, 256, 8, 512, 512, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((512, 2048, 256, 8, 500, 500, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((512, 2048, 256, 8, 192, 192, 64), _lib.MOE_ERR_UNSUPPORTED),   # I % 128 != 0
                    ((512, 2048, 256, 8, 640, 640, 64), _lib.MOE_OK),
                    ((512, 7168 + 256, 256, 8, 512, 512, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((512, 2048, 256, 8, 8192 + 128, 8192 + 128, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((65537, 2048, 256, 8, 512, 512, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((512, 2048, 256, 8, 512, 256, 64), _lib.MOE_ERR_UNSUPPORTED),
                    ((512, 2048, 256, 8, 512, 512, 32), _lib.MOE_ERR_UNSUPPORTED),
                    ((-1, 2048, 256, 8, 512, 512, 64), _lib.MOE_ERR_INVALID_ARG)]:
        s = _lib.moe_shape(*bad)
        assert lib.moe_check_shape(ctypes.byref(s)) == rc, bad
    assert lib.moe_check_shape(None) == _lib.MOE_ERR_INVALID_ARG


def test_sizes(lib):
    s = _lib.moe_shape(4096, 2048, 256, 8, 512, 512, 64)
    ws = lib.moe_workspace_bytes(ctypes.byref(s), None)
    # xs (8T x d bf16) + h (9T x 2I bf16) + weighted rows (9T x d fp32) + fp32 sum (T x d) dominate
    big = 8 * 4096 * 2048 * 2 + 9 * 4096 * 1024 * 2 + 9 * 4096 * 2048 * 4 + 4096 * 2048 * 4
    assert big <= ws < 1.1 * big + (1 << 20)
    # packed bytes = a 256-byte header + checkpoint bytes (0.5625 B per weight, 3 d x I matrices per expert)
    assert lib.moe_packed_bytes(ctypes.byref(s), 256, 512) == 256 + 256 * 3 * 2048 * 512 * 9 // 16
    assert lib.moe_max_tiles(2048, 8, 256, 32) == 16384 // 32 + 256
    bad = _lib.moe_shape(4096, 2048, 256, 8, 500, 500, 64)
    assert lib.moe_workspace_bytes(ctypes.byref(bad), None) == 0


def test_argument_validation_without_gpu(lib):
    s = _lib.moe_shape(16, 512, 256, 8, 128, 128, 64)
    rt = _lib.moe_routing()
    # null routing/workspace pointers are rejected on the host, before any CUDA call
    assert lib.moe_route(ctypes.byref(s), None, None, None, ctypes.byref(rt), None, 0, None, None) == \
        _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_ffn(ctypes.byref(s), None, ctypes.byref(rt), None, None, None, 0, None, None) == \
        _lib.MOE_ERR_INVALID_ARG
    opts = _lib.moe_options(32, 4)   # decode kernels take one token
    assert lib.moe_route(ctypes.byref(s), None, None, None, ctypes.byref(rt), None, 0, ctypes.byref(opts),
                         None) == _lib.MOE_ERR_UNSUPPORTED
    # T = 0 is a no-op that returns before looking at any pointer
    z = _lib.moe_shape(0, 512, 256, 8, 128, 128, 64)
    assert lib.moe_route(ctypes.byref(z), None, None, None, None, None, 0, None, None) == _lib.MOE_OK
    assert lib.moe_error_string(_lib.MOE_ERR_WORKSPACE).decode() != "unknown error"
    assert lib.moe_launch_count() == 0


def _static_scratch_limit():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return int(re.search(r"#define MOE_STATIC_SCRATCH_BYTES (\d+)", src).group(1))


def _static_scratch_needed(d, I, E=256, k=8):
    """Bytes the no-workspace decode call needs, as its header documents (each part rounded up
    to 256): status words, fp32 sum [d], decode scratch, tagged router logits."""
    up = lambda v: (v + 255) // 256 * 256
    return up(256) + up(d * 4) + up(8 * E * 4 + (k + 1) * 2 * I * 4) + up(8 * E * 8)


def test_static_scratch_rejects_what_does_not_fit(lib):
    """The shape and its scratch size are checked before any pointer, so null pointers
    everywhere still give the size error (nothing is launched, no GPU needed)."""
    big = _lib.moe_shape(1, 7168, 256, 8, 8192, 8192, 64)
    assert _static_scratch_needed(7168, 8192) > _static_scratch_limit()
    assert _static_scratch_needed(2048, 512) <= _static_scratch_limit()   # the decode workload fits
    rc = lib.moe_forward_decode_static(ctypes.byref(big), None, None, None, None, None, None, None, None)
    assert rc == _lib.MOE_ERR_WORKSPACE
    two = _lib.moe_shape(2, 1024, 256, 8, 256, 256, 64)
    rc = lib.moe_forward_decode_static(ctypes.byref(two), None, None, None, None, None, None, None, None)
    assert rc == _lib.MOE_ERR_UNSUPPORTED
    # a shape that fits gets to the pointer checks: null pointers are an argument error
    fits = _lib.moe_shape(1, 2048, 256, 8, 512, 512, 64)
    rc = lib.moe_forward_decode_static(ctypes.byref(fits), None, None, None, None, None, None, None, None)
    assert rc == _lib.MOE_ERR_INVALID_ARG


def test_host_routing_option_is_validated(lib):
    """moe_options.host_routing takes 0 or 1; anything else is an argument error (no GPU)."""
    s = _lib.moe_shape(512, 2048, 256, 8, 512, 512, 64)
    for v, ok in ((0, True), (1, True), (2, False), (-1, False)):
        o = _lib.moe_options(32, 1, 0, 0, v)
        n = lib.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(o))
        assert (n > 0) == ok, (v, n)


def test_unfused_dequant_option_sizes_the_workspace(lib):
    """moe_options.unfused_dequant takes 0 or 1; with 1 the prefill workspace also holds every
    expert's weights as bf16 ((E + 1) x 6 MB at d=2048, I=512), decode's does not (no GPU)."""
    s = _lib.moe_shape(512, 2048, 256, 8, 512, 512, 64)
    base = lib.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(_lib.moe_options(32, 1, 0, 0, 0, 0)))
    big = lib.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(_lib.moe_options(32, 1, 0, 0, 0, 1)))
    pairs = (512 // 128) * (2048 // 64) + (2048 // 256) * (512 // 64)
    assert big >= base + 257 * pairs * 32768 and big < base + 257 * pairs * 32768 + 4096
    for v in (2, -1):
        assert lib.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(_lib.moe_options(32, 1, 0, 0, 0, v))) == 0
    s1 = _lib.moe_shape(1, 2048, 256, 8, 512, 512, 64)
    assert (lib.moe_workspace_bytes(ctypes.byref(s1), ctypes.byref(_lib.moe_options(32, 1, 0, 0, 0, 1))) ==
            lib.moe_workspace_bytes(ctypes.byref(s1), None))


def test_deterministic_option_is_validated(lib):
    """moe_options.deterministic takes 0 or 1; anything else is an argument error (no GPU)."""
    s = _lib.moe_shape(4096, 2048, 256, 8, 512, 512, 64)
    for v, ok in ((0, True), (1, True), (2, False), (-1, False)):
        o = _lib.moe_options(32, 1, 0, v)
        n = lib.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(o))
        assert (n > 0) == ok, (v, n)


def test_gemm_rows_option_is_validated(lib):
    """moe_options.gemm_rows takes 0 (default 128) or 16, 32, 64, 128; anything else is an
    argument error.  The workspace does not depend on it (its tile lists are sized for 16)."""
    s = _lib.moe_shape(4096, 2048, 256, 8, 512, 512, 64)
    base = lib.moe_workspace_bytes(ctypes.byref(s), None)
    for v, ok in ((0, True), (16, True), (32, True), (64, True), (128, True), (48, False), (256, False),
                  (-16, False)):
        o = _lib.moe_options(32, 1, 0, 0, 0, 0, v)
        n = lib.moe_workspace_bytes(ctypes.byref(s), ctypes.byref(o))
        assert (n == base) if ok else (n == 0), (v, n)
