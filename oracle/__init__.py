"""CPU oracle for MXFP8 quantization and the block-scaled grouped GEMM.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  The
product package never imports it and shares no code with it.

The arithmetic lives in ``mxfp8_oracle.c`` (plain C, fp64); this module builds
it with gcc, loads it with ctypes and wraps it for numpy arrays.  bf16 tensors
are passed as their uint16 bit patterns.  See the C file's header for the
sources and for which functions are pinned by which tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp8_oracle.c")
_LIB = os.path.join(_HERE, "libmxfp8_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available, never fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", _LIB, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = ctypes.c_double
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f64.restype = ctypes.c_double
        L.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e8m0_to_f64.restype = ctypes.c_double
        L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e8m0_from_amax.argtypes = [ctypes.c_double]
        L.oracle_e8m0_from_amax.restype = ctypes.c_uint8
        L.oracle_quantize_vec.argtypes = [P, I64, I64, P, P]
        L.oracle_quantize_rows.argtypes = [P, I64, I64, P, P]
        L.oracle_quantize_cols.argtypes = [P, I64, I64, P, P]
        L.oracle_quantize_32x32.argtypes = [P, I64, I64, P, P]
        L.oracle_blocked_offset.argtypes = [I64, I64, I64]
        L.oracle_blocked_offset.restype = I64
        L.oracle_blocked_rowgroups.argtypes = [P, I64, I64, P, I64, P]
        L.oracle_blocked_rowgroups.restype = I64
        L.oracle_blocked_colgroups.argtypes = [P, I64, I64, P, I64, P]
        L.oracle_blocked_colgroups.restype = I64
        L.oracle_dot.argtypes = [P, P, P, P, I64]
        L.oracle_dot.restype = ctypes.c_double
        L.oracle_grouped_mm_rows.argtypes = [P, P, P, P, P, I64, I64, I64, I64, P]
        L.oracle_grouped_mm_wgrad.argtypes = [P, P, P, P, P, I64, I64, I64, I64, P]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
        L.oracle_bf16_from_f64.restype = ctypes.c_uint16
        L.oracle_bf16_from_f64_array.argtypes = [P, I64, P]
        L.oracle_swiglu_bf16.argtypes = [P, P, I64, P]
        L.oracle_swiglu_bwd_bf16.argtypes = [P, P, P, I64, P, P]
        L.oracle_philox4x32_10.argtypes = [P, P, P]
        L.oracle_sr_byte.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.oracle_sr_byte.restype = ctypes.c_uint8
        L.oracle_e4m3_encode_sr.argtypes = [ctypes.c_double, ctypes.c_uint32]
        L.oracle_e4m3_encode_sr.restype = ctypes.c_uint8
        L.oracle_rht_signs.argtypes = [ctypes.c_uint64, P]
        L.oracle_rht32.argtypes = [P, P, P]
        L.oracle_quantize_block_at.argtypes = [P, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_uint, ctypes.c_uint64, P]
        L.oracle_quantize_block_at.restype = ctypes.c_uint8
        L.oracle_quantize_rows_opts.argtypes = [P, I64, I64, ctypes.c_uint, ctypes.c_uint64, P, P]
        L.oracle_quantize_cols_opts.argtypes = [P, I64, I64, ctypes.c_uint, ctypes.c_uint64, P, P]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16 inputs are passed as uint16 bit patterns"
    return x


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of the oracle's OpenMP GEMM loops (1 = single-threaded)."""
    lib().oracle_set_num_threads(int(n))


# ---------------------------------------------------------------- scalars
def bf16_to_f64(b: int) -> float:
    return lib().oracle_bf16_to_f64(int(b))


def e4m3_to_f64(q: int) -> float:
    return lib().oracle_e4m3_to_f64(int(q))


def e8m0_to_f64(s: int) -> float:
    return lib().oracle_e8m0_to_f64(int(s))


def e4m3_encode(y: float) -> int:
    return int(lib().oracle_e4m3_encode(float(y)))


def e8m0_from_amax(amax: float) -> int:
    return int(lib().oracle_e8m0_from_amax(float(amax)))


def e4m3_table() -> np.ndarray:
    """fp64 value of every E4M3 code 0..255 (NaN for the two NaN codes)."""
    return np.array([e4m3_to_f64(c) for c in range(256)], dtype=np.float64)


def dequant(q: np.ndarray, s_expanded: np.ndarray) -> np.ndarray:
    """deq(q, s) = E4M3(q) * 2^(s-127), elementwise (s already broadcast to q's shape)."""
    tab = e4m3_table()
    sv = np.ldexp(1.0, s_expanded.astype(np.int64) - 127)
    return tab[q] * sv


# ---------------------------------------------------------------- quantize
def quantize_vec(x_u16: np.ndarray):
    x = _u16(x_u16).reshape(-1)
    n = x.size
    assert n % 32 == 0
    q = np.empty(n, np.uint8)
    s = np.empty(n // 32, np.uint8)
    lib().oracle_quantize_vec(_p(x), n, 1, _p(q), _p(s))
    return q, s


def quantize_rows(x_u16: np.ndarray):
    """Blocks of 32 along the last dim of x[R, C] -> q[R, C], compact s[R, C/32]."""
    x = _u16(x_u16)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    lib().oracle_quantize_rows(_p(x), R, C, _p(q), _p(s))
    return q, s


def quantize_cols(x_u16: np.ndarray):
    """Blocks of 32 along the first dim of x[R, C] -> qT[C, R], compact sT[C, R/32]."""
    x = _u16(x_u16)
    R, C = x.shape
    assert R % 32 == 0
    qT = np.empty((C, R), np.uint8)
    sT = np.empty((C, R // 32), np.uint8)
    lib().oracle_quantize_cols(_p(x), R, C, _p(qT), _p(sT))
    return qT, sT


def quantize_32x32(x_u16: np.ndarray):
    x = _u16(x_u16)
    R, C = x.shape
    assert R % 32 == 0 and C % 32 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R // 32, C // 32), np.uint8)
    lib().oracle_quantize_32x32(_p(x), R, C, _p(q), _p(s))
    return q, s


# ---------------------------------------------------------------- layouts
def blocked_offset(r: int, kb: int, kb_tiles: int) -> int:
    return int(lib().oracle_blocked_offset(r, kb, kb_tiles))


def _ends(ends) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(ends, dtype=np.int64))


def blocked_rowgroups_bytes(ends, Kb: int) -> int:
    e = _ends(ends)
    sizes = np.diff(np.concatenate([[0], e]))
    return int(sum(-(-int(m) // 128) * 128 for m in sizes) * (-(-Kb // 4)) * 4)


def blocked_rowgroups(s: np.ndarray, ends) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, Kb = s.shape
    e = _ends(ends)
    out = np.empty(blocked_rowgroups_bytes(e, Kb), np.uint8)
    n = lib().oracle_blocked_rowgroups(_p(s), R, Kb, _p(e), e.size, _p(out))
    assert n == out.size
    return out


def blocked_colgroups_bytes(R: int, ends) -> int:
    e = _ends(ends)
    sizes = np.diff(np.concatenate([[0], e]))
    return int(-(-R // 128) * 128 * sum(-(-int(m) // 128) * 4 for m in sizes))


def blocked_colgroups(s: np.ndarray, ends) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, Mb = s.shape
    e = _ends(ends)
    out = np.empty(blocked_colgroups_bytes(R, e), np.uint8)
    n = lib().oracle_blocked_colgroups(_p(s), R, Mb, _p(e), e.size, _p(out))
    assert n == out.size
    return out


# ---------------------------------------------------------------- GEMMs
def dot(a, sa, b, sb) -> float:
    a = np.ascontiguousarray(a, np.uint8)
    b = np.ascontiguousarray(b, np.uint8)
    sa = np.ascontiguousarray(sa, np.uint8)
    sb = np.ascontiguousarray(sb, np.uint8)
    assert a.size == b.size and a.size % 32 == 0
    return float(lib().oracle_dot(_p(a), _p(sa), _p(b), _p(sb), a.size))


def grouped_mm_rows(aq, as_, bq, bs, ends) -> np.ndarray:
    """fwd / dgrad: out[m, n] = sum_k A[m,k] B_g[n,k] for m in group g (fp64 [M, Nb])."""
    aq = np.ascontiguousarray(aq, np.uint8)
    as_ = np.ascontiguousarray(as_, np.uint8)
    bq = np.ascontiguousarray(bq, np.uint8)
    bs = np.ascontiguousarray(bs, np.uint8)
    M, K = aq.shape
    G, Nb, K2 = bq.shape
    assert K == K2
    e = _ends(ends)
    assert e.size == G and e[-1] == M
    out = np.zeros((M, Nb), np.float64)
    lib().oracle_grouped_mm_rows(_p(aq), _p(as_), _p(bq), _p(bs), _p(e), G, M, Nb, K, _p(out))
    return out


def grouped_mm_wgrad(dq, ds, aq, as_, ends) -> np.ndarray:
    """wgrad: out[g][n, k] = sum_{m in g} dOut[m,n] A[m,k] (fp64 [G, N, K])."""
    dq = np.ascontiguousarray(dq, np.uint8)
    ds = np.ascontiguousarray(ds, np.uint8)
    aq = np.ascontiguousarray(aq, np.uint8)
    as_ = np.ascontiguousarray(as_, np.uint8)
    N, M = dq.shape
    K, M2 = aq.shape
    assert M == M2
    e = _ends(ends)
    G = e.size
    out = np.zeros((G, N, K), np.float64)
    lib().oracle_grouped_mm_wgrad(_p(dq), _p(ds), _p(aq), _p(as_), _p(e), G, M, N, K, _p(out))
    return out


def _deq_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Dequantized fp64 values of codes q[..., C] with compact scales s[..., C/32] (one per 32)."""
    return dequant(np.ascontiguousarray(q, np.uint8), np.repeat(np.ascontiguousarray(s, np.uint8), 32, axis=-1))


def grouped_mm_rows_blas(aq, as_, bq, bs, ends) -> np.ndarray:
    """grouped_mm_rows with each group's contraction done by numpy's fp64 matmul (a library GEMM)
    on the operands dequantized by the format definitions above: the same sum, another order, for
    sizes where the scalar loops take minutes.  Pinned to grouped_mm_rows by the tests."""
    aq = np.ascontiguousarray(aq, np.uint8)
    M, K = aq.shape
    G, Nb, K2 = bq.shape
    assert K == K2
    e = _ends(ends)
    assert e.size == G and e[-1] == M
    out = np.zeros((M, Nb), np.float64)
    lo = 0
    for g in range(G):
        hi = int(e[g])
        if hi > lo:
            out[lo:hi] = _deq_rows(aq[lo:hi], as_[lo:hi]) @ _deq_rows(bq[g], bs[g]).T
        lo = hi
    return out


def grouped_mm_wgrad_blas(dq, ds, aq, as_, ends) -> np.ndarray:
    """grouped_mm_wgrad with numpy's fp64 matmul per group over the dequantized token-wise operands
    (dOut^T codes dq[N, M], A^T codes aq[K, M], compact scales along M).  Pinned to grouped_mm_wgrad."""
    N, M = dq.shape
    K, M2 = aq.shape
    assert M == M2
    e = _ends(ends)
    dd = _deq_rows(dq, ds)
    ad = _deq_rows(aq, as_)
    out = np.zeros((e.size, N, K), np.float64)
    lo = 0
    for g in range(e.size):
        hi = int(e[g])
        if hi > lo:
            out[g] = dd[:, lo:hi] @ ad[:, lo:hi].T
        lo = hi
    return out


# ---------------------------------------------------------------- SwiGLU stage of a routed expert
def bf16_from_f64(x) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), round to nearest even, one rounding."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_bf16_from_f64_array(_p(x), x.size, _p(out))
    return out


def swiglu_bf16(h1, h3) -> np.ndarray:
    """h = bf16(bf16(silu(h1)) * h3) over bf16 bit patterns (uint16 in, uint16 out)."""
    h1 = _u16(h1)
    h3 = _u16(h3)
    assert h1.shape == h3.shape
    out = np.empty(h1.shape, np.uint16)
    lib().oracle_swiglu_bf16(_p(h1), _p(h3), h1.size, _p(out))
    return out


def swiglu_bwd_bf16(dh, h1, h3):
    """(dh1, dh3) of h = silu(h1) * h3 at the rounding points of the bf16 autograd ops (uint16 patterns)."""
    dh, h1, h3 = _u16(dh), _u16(h1), _u16(h3)
    assert dh.shape == h1.shape == h3.shape
    dh1 = np.empty(dh.shape, np.uint16)
    dh3 = np.empty(dh.shape, np.uint16)
    lib().oracle_swiglu_bwd_bf16(_p(dh), _p(h1), _p(h3), dh.size, _p(dh1), _p(dh3))
    return dh1, dh3


def swiglu_bwd_quantized(dh, h1, h3) -> dict:
    """The SwiGLU backward stage followed by the quantization of dh1 and dh3 along the row (the
    gate/up dgrads' contraction H) and along the tokens (their wgrads): compact scales."""
    dh1, dh3 = swiglu_bwd_bf16(dh, h1, h3)
    out = dict(dh1=dh1, dh3=dh3)
    for name, t in (("dh1", dh1), ("dh3", dh3)):
        out[name + "_q"], out[name + "_s"] = quantize_rows(t)
        if t.shape[0] % 32 == 0:
            out[name + "T_q"], out[name + "T_s"] = quantize_cols(t)
    return out


def swiglu_gate_up(x_u16, wg_u16, wu_u16, ends, blas: bool = False) -> dict:
    """The gate/up half of a SwiGLU routed expert, from bf16 inputs: x [M, D], Wg and Wu
    [G, H, D].  x and the weights are quantized along D, both GEMMs run in fp64, and
    h1, h3, h follow the bf16 rounding points of oracle_swiglu_bf16.  Returns the fp64
    GEMM results (h1_f64, h3_f64), the bf16 patterns (h1, h3, h), and h quantized along
    H (h_q, h_s compact [M, H/32]) and along the tokens (hT_q [H, M], hT_s compact).  blas: the
    GEMMs by grouped_mm_rows_blas (large shapes)."""
    xq, xs = quantize_rows(x_u16)
    G = wg_u16.shape[0]
    wg = [quantize_rows(wg_u16[g]) for g in range(G)]
    wu = [quantize_rows(wu_u16[g]) for g in range(G)]
    mm = grouped_mm_rows_blas if blas else grouped_mm_rows
    h1f = mm(xq, xs, np.stack([q for q, _ in wg]), np.stack([s_ for _, s_ in wg]), ends)
    h3f = mm(xq, xs, np.stack([q for q, _ in wu]), np.stack([s_ for _, s_ in wu]), ends)
    h1, h3 = bf16_from_f64(h1f), bf16_from_f64(h3f)
    h = swiglu_bf16(h1, h3)
    out = dict(h1_f64=h1f, h3_f64=h3f, h1=h1, h3=h3, h=h)
    out["h_q"], out["h_s"] = quantize_rows(h)
    if h.shape[0] % 32 == 0:
        out["hT_q"], out["hT_s"] = quantize_cols(h)
    return out


# ---------------------------------------------------------------- stability variants
OPT_SR, OPT_RHT = 1, 2


def philox4x32_10(ctr, key) -> list:
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return [int(v) for v in out]


def sr_byte(seed: int, r: int, c: int, C: int) -> int:
    """The random byte of element (r, c) of an input with C columns (both copies use it)."""
    return int(lib().oracle_sr_byte(seed, r, c, C))


def e4m3_encode_sr(y: float, u: int) -> int:
    """E4M3 code of y rounded stochastically with the random byte u."""
    return int(lib().oracle_e4m3_encode_sr(float(y), int(u)))


def rht_signs(seed: int) -> np.ndarray:
    d = np.zeros(32, np.int8)
    lib().oracle_rht_signs(seed, _p(d))
    return d


def rht32(x, d) -> np.ndarray:
    """c * H * (D x) of one block of 32 fp32 values, in fp32 (butterfly order h = 1..16)."""
    x = np.ascontiguousarray(x, np.float32)
    d = np.ascontiguousarray(d, np.int8)
    assert x.size == 32 and d.size == 32
    y = np.zeros(32, np.float32)
    lib().oracle_rht32(_p(x), _p(d), _p(y))
    return y


def quantize_rows_opts(x_u16, opts: int, seed: int):
    """Row-wise quantization with options (OPT_SR: stochastic rounding; OPT_RHT: Hadamard transform
    of every block of 32 first): q [R, C], compact s [R, C/32]."""
    x = _u16(x_u16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s_ = np.empty((R, C // 32), np.uint8)
    lib().oracle_quantize_rows_opts(_p(x), R, C, opts, seed, _p(q), _p(s_))
    return q, s_


def quantize_cols_opts(x_u16, opts: int, seed: int):
    """Column-wise quantization with options, transposed: qT [C, R], compact sT [C, R/32]."""
    x = _u16(x_u16)
    R, C = x.shape
    qT = np.empty((C, R), np.uint8)
    sT = np.empty((C, R // 32), np.uint8)
    lib().oracle_quantize_cols_opts(_p(x), R, C, opts, seed, _p(qT), _p(sT))
    return qT, sT


def quantize_block_at(x32_u16, r0: int, c0: int, along_rows: bool, C: int, opts: int, seed: int):
    """One block of 32 bf16 values of an input with C columns, quantized with options: a row
    block (element i at row r0, column c0 + i) or, with along_rows, a column block (element i at
    row r0 + i, column c0).  Returns (codes [32], scale byte)."""
    x = _u16(x32_u16).reshape(-1)
    assert x.size == 32
    q = np.empty(32, np.uint8)
    dr, dc = (1, 0) if along_rows else (0, 1)
    s_ = lib().oracle_quantize_block_at(_p(x), r0, c0, dr, dc, C, opts, seed, _p(q))
    return q, int(s_)
