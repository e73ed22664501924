"""Comparison helpers for quantized outputs whose inputs may differ from the oracle's by a bf16
rounding (test code, no quantization arithmetic): blocked-scale decoding through the oracle's own
layout function, and the one-E4M3-step comparison."""
import numpy as np

import oracle


def decode_blocked(kind, R, Kb, ends):
    """Blocked-layout position of every compact scale (r, kb), found by passing probe arrays
    through the oracle's own layout function; also the mask of bytes that hold a scale."""
    if kind == "rows":
        place = lambda a: oracle.blocked_rowgroups(a, ends)
    else:
        place = lambda a: oracle.blocked_colgroups(a, ends)
    r = np.arange(R)[:, None] + np.zeros((1, Kb), np.int64)
    k = np.zeros((R, 1), np.int64) + np.arange(Kb)[None, :]
    probes = [place(((v >> sh) & 0xFF).astype(np.uint8)) for v in (r, k) for sh in (0, 8, 16)]
    valid = place(np.ones((R, Kb), np.uint8)).astype(bool)
    pr = probes[0].astype(np.int64) | (probes[1].astype(np.int64) << 8) | (probes[2].astype(np.int64) << 16)
    pk = probes[3].astype(np.int64) | (probes[4].astype(np.int64) << 8) | (probes[5].astype(np.int64) << 16)
    pos = np.zeros((R, Kb), np.int64)
    idx = np.nonzero(valid)[0]
    pos[pr[idx], pk[idx]] = idx
    return pos, valid


def e4m3_step(v, s):
    """One E4M3 quantum at magnitude |v| in a block with scale byte s (subnormal step 2^-9)."""
    e = s.astype(np.int64) - 127
    y = np.abs(v) * np.ldexp(1.0, -e)
    ex = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    return np.ldexp(1.0, (ex - 3 + e).astype(np.int64))


def compare_quantized(q_gpu, s_gpu_blk, q_o, s_o, kind, ends, exact, exclude=None, what="", min_code_eq=0.99,
                      min_scale_eq=0.999):
    R, C = q_o.shape
    pos, valid = decode_blocked(kind, R, C // 32, ends)
    s_blk = s_gpu_blk[:valid.size]
    assert np.all(s_blk[~valid] == 0), f"{what}: padding bytes not zero"
    s_g = s_blk[pos]
    if exact:
        keep = np.ones(q_o.shape, bool) if exclude is None else ~exclude
        blk_keep = keep.reshape(R, C // 32, 32).all(axis=2)
        assert np.array_equal(s_g[blk_keep], s_o[blk_keep]), f"{what}: scales differ"
        sel = keep & np.repeat(blk_keep, 32, axis=1)
        assert np.array_equal(q_gpu[sel], q_o[sel]), f"{what}: {int((q_gpu != q_o)[sel].sum())} codes differ"
        return
    tab = oracle.e4m3_table()
    sg_e, so_e = np.repeat(s_g, 32, axis=1), np.repeat(s_o, 32, axis=1)
    dg = tab[q_gpu] * np.ldexp(1.0, sg_e.astype(np.int64) - 127)
    do = tab[q_o] * np.ldexp(1.0, so_e.astype(np.int64) - 127)
    step = e4m3_step(np.maximum(np.abs(dg), np.abs(do)), np.maximum(sg_e, so_e))
    assert np.all(np.abs(s_g.astype(int) - s_o.astype(int)) <= 1), f"{what}: a scale differs by more than one"
    assert np.all(np.abs(dg - do) <= step), f"{what}: {int((np.abs(dg - do) > step).sum())} elements beyond one step"
    assert (q_gpu == q_o).mean() >= min_code_eq, f"{what}: code agreement {(q_gpu == q_o).mean():.5f}"
    assert (s_g == s_o).mean() >= min_scale_eq, f"{what}: scale agreement {(s_g == s_o).mean():.5f}"
