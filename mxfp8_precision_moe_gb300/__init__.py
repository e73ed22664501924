"""GB300 (sm_103a) MXFP8 routed-expert hot path: dynamic MXFP8 quantization and
block-scaled grouped GEMMs, the computation behind
``_to_mxfp8_then_scaled_grouped_mm`` ("MXFP8 training for MoEs", the engine
paragraph: quantize activations and weights dynamically, run a scaled grouped
GEMM, return the original precision, differentiable).

This module is a thin binding over the C ABI in ``include/mxfp8moe.h``
(``libmxfp8moe.so``): it allocates outputs with torch, passes raw device
pointers and the current CUDA stream, and raises on any status other than
MXFP8_OK.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback.

Tensors: bf16 inputs; e4m3 codes are returned as ``torch.uint8`` (view them as
``torch.float8_e4m3fn`` if needed); E8M0 scales are ``torch.uint8``; group
offsets are int32 cumulative end rows on the device.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import (BLOCK32X32, COL, MAX_GROUPS, OPT_HADAMARD_COL, OPT_HADAMARD_ROW, OPT_STOCHASTIC, ROW,
                   SCALES_BLOCKED, SCALES_COMPACT, Mxfp8Error, check, load)

__all__ = [
    "ROW", "COL", "BLOCK32X32", "SCALES_COMPACT", "SCALES_BLOCKED", "MAX_GROUPS", "Mxfp8Error",
    "OPT_STOCHASTIC", "OPT_HADAMARD_ROW", "OPT_HADAMARD_COL",
    "mxfp8_quantize_2d", "mxfp8_quantize_3d_experts", "mxfp8_grouped_mm_fwd", "mxfp8_grouped_mm_dgrad",
    "mxfp8_grouped_mm_wgrad", "mxfp8_scale_bytes", "mxfp8_scale_bytes_colgroups", "mxfp8_check_offsets",
    "mxfp8_debug_wait_timeout", "new_status", "read_status", "to_mxfp8_then_scaled_grouped_mm", "load",
    "quantize_expert_weights", "Mxfp8WeightCache", "mxfp8_grouped_mm_swiglu_fwd", "mxfp8_swiglu_expert",
    "mxfp8_swiglu_bwd_quantize", "mxfp8_grouped_mm_dgrad2",
]


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("mxfp8: every tensor must live on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("mxfp8: tensors must be contiguous")


def _u8(shape, device):
    return torch.empty(shape, dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- argument checks (host side, before any call)
# The C ABI takes raw pointers and cannot see buffer extents: a short scale buffer or an offsets
# array with fewer than G entries would make a kernel read past its allocation.  Every wrapper
# below therefore checks dtypes, shapes, offsets lengths and scale-buffer byte counts first.
def _tensor(t, name: str, dtype, ndim: int | None = None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name}: expected a tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dimensions, got shape {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _bytes_at_least(t, name: str, nbytes: int):
    _tensor(t, name, torch.uint8)
    if t.numel() < nbytes:
        raise ValueError(f"{name}: a scale buffer of at least {nbytes} bytes is needed, got {t.numel()}")


def _offsets(offs, G: int | None = None):
    _tensor(offs, "offs", torch.int32, 1)
    if offs.numel() < 1 or offs.numel() > MAX_GROUPS:
        raise ValueError(f"offs: 1 .. {MAX_GROUPS} groups, got {offs.numel()}")
    if G is not None and offs.numel() != G:
        raise ValueError(f"offs: one end offset per group expected ({G}), got {offs.numel()}")


def _status_word(dev_status):
    if dev_status is not None:
        _tensor(dev_status, "dev_status", torch.int32)
        if dev_status.numel() < 1:
            raise ValueError("dev_status: one int32 word needed")


def _expert_blocked_bytes(rows: int, K: int) -> int:
    """Blocked scale bytes of one expert matrix [rows, K] quantized along K."""
    return ((rows + 127) // 128) * 128 * ((K + 127) // 128) * 4


def new_status(device=None) -> torch.Tensor:
    """A zeroed int32 device word for device-detected errors."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status: torch.Tensor, where: str = "device") -> None:
    """Synchronize on the status word and raise if a kernel reported an error."""
    check(int(status.item()), where)


# ---------------------------------------------------------------- sizes
def mxfp8_scale_bytes(rows: int, K: int, G: int, scale_layout: int) -> int:
    return int(load().mxfp8_scale_bytes(rows, K, G, scale_layout))


def mxfp8_scale_bytes_colgroups(R: int, M: int, G: int) -> int:
    return int(load().mxfp8_scale_bytes_colgroups(R, M, G))


# ---------------------------------------------------------------- quantization
def mxfp8_quantize_2d(x: torch.Tensor, dirs: int = ROW, scale_layout: int = SCALES_BLOCKED,
                      offs: torch.Tensor | None = None, dev_status: torch.Tensor | None = None, opts: int = 0,
                      seed: int = 0):
    """Quantize x[M, K] (bf16).  Returns (q_row, s_row, q_col, s_col), None for
    directions not requested.  q_row [M, K]; q_col [K, M].  Compact scales are
    2D ([M, K/32], [K, M/32], or [M/32, K/32] for 32x32 blocks); blocked scales
    are flat byte buffers (upper-bound size, zero padded).  opts (OPT_STOCHASTIC,
    OPT_HADAMARD_ROW, OPT_HADAMARD_COL) and seed select the stability variants
    of mxfp8_quantize_2d_opts."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("mxfp8_quantize_2d: x must be a 2D bf16 tensor")
    if offs is not None:
        _offsets(offs)
    _status_word(dev_status)
    _cuda(x, offs, dev_status)
    M, K = x.shape
    G = int(offs.numel()) if offs is not None else 1
    dev = x.device
    q_row = s_row = q_col = s_col = None
    if dirs & (ROW | BLOCK32X32):
        q_row = _u8((M, K), dev)
        if dirs & BLOCK32X32:
            s_row = _u8((M // 32, K // 32), dev)
        elif scale_layout == SCALES_COMPACT:
            s_row = _u8((M, K // 32), dev)
        else:
            s_row = _u8((mxfp8_scale_bytes(M, K, G, SCALES_BLOCKED),), dev)
    if dirs & COL:
        q_col = _u8((K, M), dev)
        if scale_layout == SCALES_COMPACT:
            s_col = _u8((K, M // 32), dev)
        else:
            s_col = _u8((mxfp8_scale_bytes_colgroups(K, M, G),), dev)
    if opts:
        st = load().mxfp8_quantize_2d_opts(_p(x), M, K, dirs, scale_layout, _p(offs), G if offs is not None else 0,
                                           opts, seed & (2 ** 64 - 1), _p(q_row), _p(s_row), _p(q_col), _p(s_col),
                                           _p(dev_status), _stream(dev))
        check(st, "mxfp8_quantize_2d_opts")
        return q_row, s_row, q_col, s_col
    st = load().mxfp8_quantize_2d(_p(x), M, K, dirs, scale_layout, _p(offs), G if offs is not None else 0,
                                  _p(q_row), _p(s_row), _p(q_col), _p(s_col), _p(dev_status), _stream(dev))
    check(st, "mxfp8_quantize_2d")
    return q_row, s_row, q_col, s_col


def mxfp8_quantize_3d_experts(w: torch.Tensor, dirs: int = ROW | COL, scale_layout: int = SCALES_BLOCKED,
                              dev_status: torch.Tensor | None = None):
    """Quantize expert weights w[G, N, K] (bf16).  Returns (q, s, qT, sT):
    q [G, N, K] along K ("plain"), qT [G, K, N] along N ("transposed");
    scales [G, ...] per expert (compact 3D, or blocked flat per expert)."""
    if w.dtype != torch.bfloat16 or w.dim() != 3:
        raise ValueError("mxfp8_quantize_3d_experts: w must be a 3D bf16 tensor")
    _status_word(dev_status)
    _cuda(w, dev_status)
    G, N, K = w.shape
    dev = w.device
    q = s = qT = sT = None
    if dirs & ROW:
        q = _u8((G, N, K), dev)
        s = _u8((G, N, K // 32), dev) if scale_layout == SCALES_COMPACT else \
            _u8((G, ((N + 127) // 128) * 128 * ((K + 127) // 128) * 4), dev)
    if dirs & COL:
        qT = _u8((G, K, N), dev)
        sT = _u8((G, K, N // 32), dev) if scale_layout == SCALES_COMPACT else \
            _u8((G, ((K + 127) // 128) * 128 * ((N + 127) // 128) * 4), dev)
    st = load().mxfp8_quantize_3d_experts(_p(w), G, N, K, dirs, scale_layout, _p(q), _p(s), _p(qT), _p(sT),
                                          _p(dev_status), _stream(dev))
    check(st, "mxfp8_quantize_3d_experts")
    return q, s, qT, sT


# ---------------------------------------------------------------- grouped GEMMs
def mxfp8_grouped_mm_fwd(a_q, a_s, w_q, w_s, offs, out=None, dev_status=None):
    """out[m, n] = sum_k A[m,k] W[g][n,k] for rows m of group g; bf16 [M, N]."""
    _tensor(a_q, "a_q", torch.uint8, 2)
    _tensor(w_q, "w_q", torch.uint8, 3)
    M, K = a_q.shape
    G, N, _ = w_q.shape
    _tensor(w_q, "w_q", torch.uint8, shape=(G, N, K))
    _offsets(offs, G)
    _bytes_at_least(a_s, "a_s", mxfp8_scale_bytes(M, K, G, SCALES_BLOCKED))
    _bytes_at_least(w_s, "w_s", G * _expert_blocked_bytes(N, K))
    if out is not None:
        _tensor(out, "out", torch.bfloat16, shape=(M, N))
    _status_word(dev_status)
    _cuda(a_q, a_s, w_q, w_s, offs, out, dev_status)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    st = load().mxfp8_grouped_mm_fwd(_p(a_q), _p(a_s), _p(w_q), _p(w_s), _p(offs), G, M, N, K, _p(out),
                                     _p(dev_status), _stream(a_q.device))
    check(st, "mxfp8_grouped_mm_fwd")
    return out


def mxfp8_grouped_mm_dgrad(dout_q, dout_s, wt_q, wt_s, offs, out=None, dev_status=None):
    """dA[m, k] = sum_n dOut[m,n] W[g][n,k]; dout_q [M, N], wt_q [G, K, N]; bf16 [M, K]."""
    _tensor(dout_q, "dout_q", torch.uint8, 2)
    _tensor(wt_q, "wt_q", torch.uint8, 3)
    M, N = dout_q.shape
    G, K, _ = wt_q.shape
    _tensor(wt_q, "wt_q", torch.uint8, shape=(G, K, N))
    _offsets(offs, G)
    _bytes_at_least(dout_s, "dout_s", mxfp8_scale_bytes(M, N, G, SCALES_BLOCKED))
    _bytes_at_least(wt_s, "wt_s", G * _expert_blocked_bytes(K, N))
    if out is not None:
        _tensor(out, "out", torch.bfloat16, shape=(M, K))
    _status_word(dev_status)
    _cuda(dout_q, dout_s, wt_q, wt_s, offs, out, dev_status)
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=dout_q.device)
    st = load().mxfp8_grouped_mm_dgrad(_p(dout_q), _p(dout_s), _p(wt_q), _p(wt_s), _p(offs), G, M, N, K, _p(out),
                                       _p(dev_status), _stream(dout_q.device))
    check(st, "mxfp8_grouped_mm_dgrad")
    return out


def mxfp8_grouped_mm_dgrad2(dout1_q, dout1_s, wt1_q, wt1_s, dout2_q, dout2_s, wt2_q, wt2_s, offs, out=None,
                            dev_status=None):
    """dA = dOut1 W1[g] + dOut2 W2[g] in one GEMM (one fp32 accumulator, one bf16 rounding);
    operands as for mxfp8_grouped_mm_dgrad."""
    _tensor(dout1_q, "dout1_q", torch.uint8, 2)
    _tensor(wt1_q, "wt1_q", torch.uint8, 3)
    M, N = dout1_q.shape
    G, K, _ = wt1_q.shape
    _tensor(dout2_q, "dout2_q", torch.uint8, 2)
    _tensor(wt2_q, "wt2_q", torch.uint8, 3)
    if tuple(dout2_q.shape) != (M, N) or tuple(wt2_q.shape) != (G, K, N) or tuple(wt1_q.shape) != (G, K, N):
        raise ValueError("mxfp8_grouped_mm_dgrad2: both operand pairs must have the same shapes")
    _offsets(offs, G)
    for name, t in (("dout1_s", dout1_s), ("dout2_s", dout2_s)):
        _bytes_at_least(t, name, mxfp8_scale_bytes(M, N, G, SCALES_BLOCKED))
    for name, t in (("wt1_s", wt1_s), ("wt2_s", wt2_s)):
        _bytes_at_least(t, name, G * _expert_blocked_bytes(K, N))
    if out is not None:
        _tensor(out, "out", torch.bfloat16, shape=(M, K))
    _status_word(dev_status)
    _cuda(dout1_q, dout1_s, wt1_q, wt1_s, dout2_q, dout2_s, wt2_q, wt2_s, offs, out, dev_status)
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=dout1_q.device)
    st = load().mxfp8_grouped_mm_dgrad2(_p(dout1_q), _p(dout1_s), _p(wt1_q), _p(wt1_s), _p(dout2_q), _p(dout2_s),
                                        _p(wt2_q), _p(wt2_s), _p(offs), G, M, N, K, _p(out), _p(dev_status),
                                        _stream(dout1_q.device))
    check(st, "mxfp8_grouped_mm_dgrad2")
    return out


def mxfp8_grouped_mm_wgrad(doutT_q, doutT_s, aT_q, aT_s, offs, out=None, dev_status=None):
    """dW[g][n, k] = sum_{m in g} dOut[m,n] A[m,k]; doutT_q [N, M], aT_q [K, M]; bf16 [G, N, K]."""
    _tensor(doutT_q, "doutT_q", torch.uint8, 2)
    _tensor(aT_q, "aT_q", torch.uint8, 2)
    N, M = doutT_q.shape
    K = aT_q.shape[0]
    _tensor(aT_q, "aT_q", torch.uint8, shape=(K, M))
    _offsets(offs)
    G = int(offs.numel())
    _bytes_at_least(doutT_s, "doutT_s", mxfp8_scale_bytes_colgroups(N, M, G))
    _bytes_at_least(aT_s, "aT_s", mxfp8_scale_bytes_colgroups(K, M, G))
    if out is not None:
        _tensor(out, "out", torch.bfloat16, shape=(G, N, K))
    _status_word(dev_status)
    _cuda(doutT_q, doutT_s, aT_q, aT_s, offs, out, dev_status)
    if out is None:
        out = torch.empty((G, N, K), dtype=torch.bfloat16, device=doutT_q.device)
    st = load().mxfp8_grouped_mm_wgrad(_p(doutT_q), _p(doutT_s), _p(aT_q), _p(aT_s), _p(offs), G, M, N, K,
                                       _p(out), _p(dev_status), _stream(doutT_q.device))
    check(st, "mxfp8_grouped_mm_wgrad")
    return out


def mxfp8_grouped_mm_swiglu_fwd(x_q, x_s, wg_q, wg_s, wu_q, wu_s, offs, token_wise: bool = True,
                                dev_status=None):
    """Gate and up GEMMs with the SwiGLU and its MXFP8 quantization in the epilogue.

    x_q [M, D] (+ blocked row-group scales), wg_q / wu_q [G, H, D] (+ blocked
    per-expert scales).  Returns (h1, h3, h_q, h_s, hT_q, hT_s): h1 = x Wg^T and
    h3 = x Wu^T in bf16 [M, H]; h = bf16(bf16(silu(h1)) * h3) quantized along H
    (h_q [M, H], blocked row groups) and, if token_wise, along the tokens
    (hT_q [H, M], blocked token groups; group sizes must be multiples of 32)."""
    _tensor(x_q, "x_q", torch.uint8, 2)
    _tensor(wg_q, "wg_q", torch.uint8, 3)
    M, D = x_q.shape
    G, H, _ = wg_q.shape
    _tensor(wu_q, "wu_q", torch.uint8, 3)
    if tuple(wu_q.shape) != (G, H, D) or tuple(wg_q.shape) != (G, H, D):
        raise ValueError("gate and up weights must both be [G, H, D] with D the activations' width")
    _offsets(offs, G)
    _bytes_at_least(x_s, "x_s", mxfp8_scale_bytes(M, D, G, SCALES_BLOCKED))
    for name, t in (("wg_s", wg_s), ("wu_s", wu_s)):
        _bytes_at_least(t, name, G * _expert_blocked_bytes(H, D))
    _status_word(dev_status)
    _cuda(x_q, x_s, wg_q, wg_s, wu_q, wu_s, offs, dev_status)
    dev = x_q.device
    h1 = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    h3 = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    h_q = _u8((M, H), dev)
    h_s = _u8((mxfp8_scale_bytes(M, H, G, SCALES_BLOCKED),), dev)
    hT_q = _u8((H, M), dev) if token_wise else None
    hT_s = _u8((mxfp8_scale_bytes_colgroups(H, M, G),), dev) if token_wise else None
    st = load().mxfp8_grouped_mm_swiglu_fwd(_p(x_q), _p(x_s), _p(wg_q), _p(wg_s), _p(wu_q), _p(wu_s), _p(offs), G, M,
                                            H, D, _p(h1), _p(h3), _p(h_q), _p(h_s), _p(hT_q), _p(hT_s),
                                            _p(dev_status), _stream(dev))
    check(st, "mxfp8_grouped_mm_swiglu_fwd")
    return h1, h3, h_q, h_s, hT_q, hT_s


def mxfp8_swiglu_bwd_quantize(dh, h1, h3, offs, dev_status=None):
    """SwiGLU backward with the quantization of both outputs fused in: from dh, h1, h3
    [M, H] bf16 returns ((dh1_q, dh1_s, dh1T_q, dh1T_s), (dh3_q, dh3_s, dh3T_q, dh3T_s)),
    each as mxfp8_quantize_2d(ROW | COL, SCALES_BLOCKED, offs) returns it."""
    for t in (dh, h1, h3):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.shape != dh.shape:
            raise ValueError("mxfp8_swiglu_bwd_quantize: dh, h1, h3 must be bf16 [M, H]")
    _offsets(offs)
    _status_word(dev_status)
    _cuda(dh, h1, h3, offs, dev_status)
    M, H = dh.shape
    G = int(offs.numel())
    dev = dh.device

    def outs():
        return (_u8((M, H), dev), _u8((mxfp8_scale_bytes(M, H, G, SCALES_BLOCKED),), dev), _u8((H, M), dev),
                _u8((mxfp8_scale_bytes_colgroups(H, M, G),), dev))

    o1, o3 = outs(), outs()
    st = load().mxfp8_swiglu_bwd_quantize(_p(dh), _p(h1), _p(h3), M, H, _p(offs), G, *[_p(t) for t in o1],
                                          *[_p(t) for t in o3], _p(dev_status), _stream(dev))
    check(st, "mxfp8_swiglu_bwd_quantize")
    return o1, o3


def mxfp8_check_offsets(offs: torch.Tensor, M: int, align: int, dev_status: torch.Tensor) -> None:
    """Enqueue a device check of offs (monotone, ending at M, group sizes % align == 0); a failure
    writes MXFP8_ERR_OFFSETS into dev_status (read it with read_status)."""
    _offsets(offs)
    if dev_status is None:
        raise ValueError("mxfp8_check_offsets: a dev_status word is required")
    _status_word(dev_status)
    _cuda(offs, dev_status)
    st = load().mxfp8_check_offsets(_p(offs), int(offs.numel()), M, align, _p(dev_status), _stream(offs.device))
    check(st, "mxfp8_check_offsets")


def mxfp8_debug_wait_timeout(dev_status: torch.Tensor, limit_ns: int) -> None:
    _cuda(dev_status)
    st = load().mxfp8_debug_wait_timeout(_p(dev_status), int(limit_ns), _stream(dev_status.device))
    check(st, "mxfp8_debug_wait_timeout")


# ---------------------------------------------------------------- composite differentiable op
class _ToMxfp8ThenScaledGroupedMM(torch.autograd.Function):
    """Forward: quantize A along K (and along the tokens for the wgrad), quantize
    W plain (forward) and transposed (dgrad), one grouped GEMM.  Backward:
    quantize dOut along N (dgrad) and along the tokens (wgrad), two grouped
    GEMMs.  Quantization is treated as the identity for gradients."""

    @staticmethod
    def forward(ctx, A, W, offs, w_mxfp8, w_block32x32, stability, check_offsets):
        need_dA = ctx.needs_input_grad[0]
        need_dW = ctx.needs_input_grad[1]
        sr, rht, seed = stability
        st = None
        if check_offsets:
            # the token-wise copies of the wgrad need group sizes that are multiples of 32
            st = new_status(A.device)
            mxfp8_check_offsets(offs, A.shape[0], 32 if need_dW else 1, st)
        a_dirs = ROW | (COL if need_dW else 0)
        a_opts = OPT_HADAMARD_COL if (rht and need_dW) else 0
        aq, as_, aTq, aTs = mxfp8_quantize_2d(A.contiguous(), a_dirs, SCALES_BLOCKED, offs, st, opts=a_opts,
                                              seed=seed)
        if w_mxfp8 is None:
            w_dirs = ROW | (COL if need_dA else 0) | (BLOCK32X32 if w_block32x32 else 0)
            wq, ws, wTq, wTs = mxfp8_quantize_3d_experts(W.contiguous(), w_dirs, SCALES_BLOCKED, st)
        else:
            wq, ws, wTq, wTs = _check_quad(w_mxfp8, W, need_dA)
        out = mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs, dev_status=st)
        if st is not None:
            read_status(st, "to_mxfp8_then_scaled_grouped_mm (group offsets)")
        ctx.save_for_backward(aTq, aTs, wTq, wTs, offs)
        ctx.shape = (A.shape[0], W.shape[0], W.shape[1], W.shape[2])
        ctx.stability = stability
        return out

    @staticmethod
    def backward(ctx, dOut):
        aTq, aTs, wTq, wTs, offs = ctx.saved_tensors
        need_dA, need_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dirs = (ROW if need_dA else 0) | (COL if need_dW else 0)
        if dirs == 0:
            return None, None, None, None, None, None, None
        sr, rht, seed = ctx.stability
        d_opts = (OPT_STOCHASTIC if sr else 0) | (OPT_HADAMARD_COL if (rht and need_dW) else 0)
        dq, ds, dTq, dTs = mxfp8_quantize_2d(dOut.contiguous().to(torch.bfloat16), dirs, SCALES_BLOCKED, offs,
                                             opts=d_opts, seed=seed)
        dA = mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs) if need_dA else None
        dW = mxfp8_grouped_mm_wgrad(dTq, dTs, aTq, aTs, offs) if need_dW else None
        return dA, dW, None, None, None, None, None


def _blocked_bytes(rows: int, cols: int) -> int:
    return ((rows + 127) // 128) * 128 * ((cols // 32 + 3) // 4) * 4


def _check_quad(quad, W: torch.Tensor, need_t: bool):
    """Validate a prequantized (weight_fp8, weight_scale, weight_t_fp8, weight_t_scale)
    quadruple against W[G, N, K]; the transposed pair may be None when no dgrad is needed."""
    if len(quad) != 4:
        raise ValueError("w_mxfp8 must be (weight_fp8, weight_scale, weight_t_fp8, weight_t_scale)")
    wq, ws, wTq, wTs = quad
    G, N, K = W.shape
    want = [(wq, (G, N, K)), (ws, (G, _blocked_bytes(N, K)))]
    if need_t or wTq is not None:
        want += [(wTq, (G, K, N)), (wTs, (G, _blocked_bytes(K, N)))]
    for t, shape in want:
        if t is None or t.dtype != torch.uint8 or tuple(t.shape) != shape or t.device != W.device \
                or not t.is_contiguous():
            raise ValueError(f"w_mxfp8: expected a contiguous uint8 tensor of shape {shape} on {W.device}")
    return wq, ws, wTq, wTs


def quantize_expert_weights(W: torch.Tensor, block32x32: bool = False):
    """One fused launch: W[G, N, K] -> (weight_fp8 [G, N, K], weight_scale, weight_t_fp8 [G, K, N],
    weight_t_scale), scales in the blocked layout, one flat buffer per expert.  With block32x32,
    one scale per 32x32 block: weight_t_fp8 is exactly weight_fp8 transposed (one quantization
    serves the forward and the dgrad)."""
    dirs = ROW | COL | (BLOCK32X32 if block32x32 else 0)
    return mxfp8_quantize_3d_experts(W.detach().contiguous(), dirs, SCALES_BLOCKED)


def to_mxfp8_then_scaled_grouped_mm(A: torch.Tensor, W: torch.Tensor, offs: torch.Tensor, *, w_mxfp8=None,
                                    weight_cache=None, weight_block32x32: bool = False,
                                    stochastic_rounding: bool = False, hadamard_wgrad: bool = False,
                                    seed: int | None = None, check_offsets: bool = True) -> torch.Tensor:
    """Differentiable MXFP8 grouped GEMM: out[m] = A[m] @ W[g]^T for rows m of
    group g (offs = int32 cumulative end rows).  A [M, K] bf16, W [G, N, K] bf16,
    out [M, N] bf16.  Group sizes must be multiples of 32 when gradients of W
    are needed (token-wise quantization for the wgrad).

    The expert weights are quantized on the fly unless they come prequantized:
    ``w_mxfp8`` = (weight_fp8, weight_scale, weight_t_fp8, weight_t_scale) as
    returned by ``quantize_expert_weights(W)``, or ``weight_cache`` = an
    ``Mxfp8WeightCache`` that keeps that quadruple across microbatches until W
    changes or the optimizer steps.  Gradients still flow to W.  weight_block32x32:
    quantize W on the fly with one scale per 32x32 block, so the forward and the
    dgrad use the same quantization of W (transposed for the dgrad).

    Stability variants ("MXFP8 (Micro-scaling FP8)", "Numerical stability"):
    stochastic_rounding rounds the output gradient's codes stochastically (both of
    its copies); hadamard_wgrad applies the same random Hadamard transform along the
    tokens to both wgrad operands (A's and the output gradient's column-wise copies),
    which leaves their product unchanged.  seed keys both (Philox4x32-10); None draws
    one from torch's default CPU generator per forward call.

    check_offsets (default True): the forward checks offs on the device (monotone, ending at
    M, group sizes multiples of 32 when W needs a gradient) and raises Mxfp8Error on bad
    offsets instead of returning outputs the kernels skipped.  The check reads a status word
    back, which synchronizes the stream once per forward; pass False when the offsets are
    known to be valid (e.g. produced by the router on the device) to keep the forward
    asynchronous."""
    if A.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("to_mxfp8_then_scaled_grouped_mm expects bf16 A and W")
    if offs.dtype != torch.int32:
        raise ValueError("offs must be int32")
    if A.dim() != 2 or W.dim() != 3 or A.shape[1] != W.shape[2]:
        raise ValueError("to_mxfp8_then_scaled_grouped_mm: A [M, K] and W [G, N, K] expected")
    _offsets(offs, W.shape[0])
    if w_mxfp8 is not None and weight_cache is not None:
        raise ValueError("pass w_mxfp8 or weight_cache, not both")
    if weight_cache is not None:
        w_mxfp8 = weight_cache.get(W)
    if weight_block32x32 and w_mxfp8 is not None:
        raise ValueError("weight_block32x32 applies to on-the-fly quantization; prequantize with "
                         "quantize_expert_weights(W, block32x32=True) instead")
    if (stochastic_rounding or hadamard_wgrad) and seed is None:
        seed = int(torch.randint(0, 2 ** 62, (1,)).item())
    stability = (bool(stochastic_rounding), bool(hadamard_wgrad), int(seed or 0))
    return _ToMxfp8ThenScaledGroupedMM.apply(A, W, offs, w_mxfp8, weight_block32x32, stability, bool(check_offsets))


from .weight_cache import Mxfp8WeightCache  # noqa: E402  (uses quantize_expert_weights above)
from .swiglu import mxfp8_swiglu_expert  # noqa: E402
