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
