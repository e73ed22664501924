"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
function include/mxfp8moe.h declares, sizes its buffers as documented and
rejects bad arguments synchronously (before touching a device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(mxfp8_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_precision_moe_gb300 import _lib, build

    build.build()
    return _lib.load()


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("mxfp8_quantize_2d", "mxfp8_quantize_3d_experts", "mxfp8_grouped_mm_fwd", "mxfp8_grouped_mm_dgrad",
              "mxfp8_grouped_mm_wgrad", "mxfp8_scale_bytes", "mxfp8_check_offsets", "mxfp8_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "mxfp8_precision_moe_gb300", "libmxfp8moe.so"))
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, f"not exported: {missing}"


def test_scale_bytes(lib):
    from mxfp8_precision_moe_gb300 import SCALES_BLOCKED, SCALES_COMPACT

    assert lib.mxfp8_scale_bytes(256, 256, 1, SCALES_COMPACT) == 256 * 8
    # blocked bound: (ceil(rows/128) + G) * 128 * ceil(K/128) * 4
    assert lib.mxfp8_scale_bytes(256, 256, 2, SCALES_BLOCKED) == (2 + 2) * 128 * 2 * 4
    assert lib.mxfp8_scale_bytes(300, 160, 3, SCALES_BLOCKED) == (3 + 3) * 128 * 2 * 4
    assert lib.mxfp8_scale_bytes_colgroups(100, 256, 2) == 128 * (2 + 2) * 4
    assert lib.mxfp8_scale_bytes(10, 33, 1, SCALES_COMPACT) == 0  # K not a multiple of 32


def test_bound_covers_every_split(lib, oracle_lib):
    import numpy as np

    from mxfp8_precision_moe_gb300 import SCALES_BLOCKED

    rng = np.random.default_rng(0)
    for _ in range(200):
        G = int(rng.integers(1, 9))
        sizes = rng.integers(0, 300, G)
        M, K = int(sizes.sum()), int(rng.integers(1, 20)) * 32
        ends = np.cumsum(sizes)
        assert lib.mxfp8_scale_bytes(M, K, G, SCALES_BLOCKED) >= oracle_lib.blocked_rowgroups_bytes(ends, K // 32)
        sz32 = sizes // 32 * 32
        assert lib.mxfp8_scale_bytes_colgroups(K, int(sz32.sum()), G) >= \
            oracle_lib.blocked_colgroups_bytes(K, np.cumsum(sz32))


def test_status_strings(lib):
    for s in range(10):
        assert lib.mxfp8_status_string(s)
    assert lib.mxfp8_status_string(8).decode().startswith("bounded wait")


def test_argument_errors_need_no_device(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    # K not a multiple of 32
    assert lib.mxfp8_quantize_2d(fake, 64, 48, 1, 0, None, 0, fake, fake, None, None, None, None) == 3
    # no direction
    assert lib.mxfp8_quantize_2d(fake, 64, 64, 0, 0, None, 0, fake, fake, None, None, None, None) == 4
    # 32x32 with blocked scales
    assert lib.mxfp8_quantize_2d(fake, 64, 64, 4, 1, None, 0, fake, fake, None, None, None, None) == 4
    # NULL input
    assert lib.mxfp8_quantize_2d(None, 64, 64, 1, 0, None, 0, fake, fake, None, None, None, None) == 1
    # COL with M not a multiple of 32
    assert lib.mxfp8_quantize_2d(fake, 40, 64, 2, 0, None, 0, None, None, fake, fake, None, None) == 3
    # misaligned pointer
    assert lib.mxfp8_quantize_2d(P((1 << 20) + 8), 64, 64, 1, 0, None, 0, fake, fake, None, None, None, None) == 3
    # grouped GEMMs: N not a multiple of 32, too many groups, NULL offsets, wgrad M % 32
    assert lib.mxfp8_grouped_mm_fwd(fake, fake, fake, fake, fake, 2, 64, 48, 64, fake, None, None) == 3
    assert lib.mxfp8_grouped_mm_fwd(fake, fake, fake, fake, fake, 2000, 64, 64, 64, fake, None, None) == 2
    assert lib.mxfp8_grouped_mm_dgrad(fake, fake, fake, fake, None, 2, 64, 64, 64, fake, None, None) == 1
    assert lib.mxfp8_grouped_mm_wgrad(fake, fake, fake, fake, fake, 2, 48, 64, 64, fake, None, None) == 3
    assert lib.mxfp8_quantize_3d_experts(fake, 0, 64, 64, 1, 0, fake, fake, None, None, None, None) == 2


def test_argument_errors_of_the_fused_and_option_calls(lib):
    """The calls added for the SwiGLU expert, the stability variants, the 32x32 weights and the
    two-operand dgrad reject bad arguments before touching a device as well."""
    P = ctypes.c_void_p
    fake = P(1 << 20)
    odd = P((1 << 20) + 8)  # 8-byte aligned only
    q2o = lib.mxfp8_quantize_2d_opts
    # unknown option bit; an option with 32x32 blocks; Hadamard on a copy that is not written
    assert q2o(fake, 64, 64, 3, 1, None, 0, 8, 0, fake, fake, fake, fake, None, None) == 4
    assert q2o(fake, 64, 64, 4, 0, None, 0, 1, 0, fake, fake, None, None, None, None) == 4
    assert q2o(fake, 64, 64, 2, 1, None, 0, 2, 0, None, None, fake, fake, None, None) == 4
    assert q2o(fake, 64, 64, 1, 1, None, 0, 4, 0, fake, fake, None, None, None, None) == 4
    # 3D experts: 32x32 blocks need ROW and/or COL; the transposed copy needs its buffers
    assert lib.mxfp8_quantize_3d_experts(fake, 2, 64, 64, 4, 1, fake, fake, None, None, None, None) == 4
    assert lib.mxfp8_quantize_3d_experts(fake, 2, 64, 64, 4 | 2, 1, None, None, None, fake, None, None) == 1
    # fused gate/up GEMM: (x, xs, wg, wgs, wu, wus, offs, G, M, H, D, h1, h3, hq, hs, hTq, hTs, status, stream)
    sw = lib.mxfp8_grouped_mm_swiglu_fwd
    ok = [fake] * 7
    assert sw(*ok[:4], None, fake, fake, 2, 64, 64, 64, fake, fake, fake, fake, None, None, None, None) == 1
    assert sw(*ok, 2, 64, 64, 64, fake, fake, fake, fake, fake, None, None, None) == 1   # hT_q without hT_s
    assert sw(*ok, 0, 64, 64, 64, fake, fake, fake, fake, None, None, None, None) == 2
    assert sw(*ok, 2, 64, 48, 64, fake, fake, fake, fake, None, None, None, None) == 3   # H % 32
    assert sw(*ok, 2, 40, 64, 64, fake, fake, fake, fake, fake, fake, None, None) == 3   # token-wise, M % 32
    assert sw(*ok, 2, 64, 64, 64, odd, fake, fake, fake, None, None, None, None) == 3
    # fused SwiGLU backward: (dh, h1, h3, M, H, offs, G, 8 outputs, status, stream)
    bw = lib.mxfp8_swiglu_bwd_quantize
    assert bw(fake, fake, None, 64, 64, fake, 2, *[fake] * 8, None, None) == 1
    assert bw(fake, fake, fake, 64, 64, fake, 0, *[fake] * 8, None, None) == 2
    assert bw(fake, fake, fake, 40, 64, fake, 2, *[fake] * 8, None, None) == 3
    assert bw(fake, fake, fake, 64, 64, fake, 2, *[fake] * 7, odd, None, None) == 3
    # two-operand dgrad: (d1, d1s, w1, w1s, d2, d2s, w2, w2s, offs, G, M, N, K, dA, status, stream)
    d2 = lib.mxfp8_grouped_mm_dgrad2
    assert d2(*[fake] * 4, None, fake, fake, fake, fake, 2, 64, 64, 64, fake, None, None) == 1
    assert d2(*[fake] * 4, fake, None, fake, fake, fake, 2, 64, 64, 64, fake, None, None) == 1
    assert d2(*[fake] * 6, odd, fake, fake, 2, 64, 64, 64, fake, None, None) == 3
    assert d2(*[fake] * 9, 2, 64, 48, 64, fake, None, None) == 3                        # contraction N % 32
