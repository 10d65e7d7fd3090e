"""CPU oracle of the decode-step MoE layer tail (ctypes binding of moe_tail_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product library and its binding never do.
It shares no code with the CUDA path.

Every function takes and returns numpy arrays; bf16 values travel as their uint16 bits.
Parity of each function is pinned by the CPU tests (tests/test_oracle_pins.py) against
closed forms, brute force and special cases that the method's definition fixes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_e2m1.argtypes = [I]
        lib.oracle_e2m1.restype = D
        lib.oracle_e8m0.argtypes = [I]
        lib.oracle_e8m0.restype = D
        lib.oracle_bf16_round.argtypes = [D]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D
        lib.oracle_silu.argtypes = [D]
        lib.oracle_silu.restype = D
        lib.oracle_mxfp4_dequant_row.argtypes = [P, P, ctypes.c_int64, P]
        lib.oracle_mxfp4_dequant_row.restype = None
        lib.oracle_add_rmsnorm.argtypes = [I, I, P, P, P, D, P, P, P]
        lib.oracle_add_rmsnorm.restype = None
        lib.oracle_router.argtypes = [I, I, I, P, P, P]
        lib.oracle_router.restype = None
        lib.oracle_topk.argtypes = [I, I, I, P, P, P]
        lib.oracle_topk.restype = None
        lib.oracle_expert.argtypes = [I, I, I, P, P, P, P, P, P, P]
        lib.oracle_expert.restype = None
        lib.oracle_shared.argtypes = [I, I, P, P, P, P, P]
        lib.oracle_shared.restype = None
        lib.oracle_moe_tail.argtypes = [I, I, I, I, I, I, D] + [P] * 15 + [I]
        lib.oracle_moe_tail.restype = I
        lib.oracle_shared_gate.argtypes = [I, I, P, P, P]
        lib.oracle_shared_gate.restype = None
        lib.oracle_out_proj.argtypes = [I, I, I, P, P, P]
        lib.oracle_out_proj.restype = None
        lib.oracle_moe_tail_gated.argtypes = [I, I, I, I, I, I, D] + [P] * 16 + [I]
        lib.oracle_moe_tail_gated.restype = I
        lib.oracle_attnres_mix.argtypes = [I, I, I, I, D] + [P] * 9
        lib.oracle_attnres_mix.restype = I
        _lib = lib
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1(code: int) -> float:
    return _load().oracle_e2m1(int(code))


def e8m0(s: int) -> float:
    return _load().oracle_e8m0(int(s))


def bf16_round(v: float) -> int:
    return int(_load().oracle_bf16_round(float(v)))


def bf16_to_double(b: int) -> float:
    return _load().oracle_bf16_to_double(int(b))


def silu(z: float) -> float:
    return _load().oracle_silu(float(z))


def mxfp4_dequant_row(codes, scales, K: int):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    assert codes.size * 2 >= K and scales.size * 32 >= K
    out = np.empty(K, dtype=np.float64)
    _load().oracle_mxfp4_dequant_row(_p(codes), _p(scales), K, _p(out))
    return out


def add_rmsnorm(x, residual, gamma, eps):
    x = _c(x, np.uint16)
    residual = _c(residual, np.uint16)
    gamma = _c(gamma, np.uint16)
    R, H = x.shape
    r_new = np.empty((R, H), np.uint16)
    n = np.empty((R, H), np.uint16)
    rstd = np.empty(R, np.float64)
    _load().oracle_add_rmsnorm(R, H, _p(x), _p(residual), _p(gamma), float(eps), _p(r_new),
                               _p(n), _p(rstd))
    return r_new, n, rstd


def router(n, w_r):
    n = _c(n, np.uint16)
    w_r = _c(w_r, np.uint16)
    R, H = n.shape
    E = w_r.shape[0]
    assert w_r.shape[1] == H
    logits = np.empty((R, E), np.float64)
    _load().oracle_router(R, H, E, _p(n), _p(w_r), _p(logits))
    return logits


def topk(logits, k: int):
    logits = _c(logits, np.float64)
    R, E = logits.shape
    ids = np.empty((R, k), np.int32)
    wts = np.empty((R, k), np.float64)
    _load().oracle_topk(R, E, int(k), _p(logits), _p(ids), _p(wts))
    return ids, wts


def expert(n_row, e: int, w13_codes, w13_scales, w2_codes, w2_scales):
    """One activation row through routed expert e; returns (y [H] float64, mid [I] bf16 bits)."""
    n_row = _c(n_row, np.uint16)
    H = n_row.shape[0]
    I = w2_codes.shape[2] * 2
    w13_codes = _c(w13_codes, np.uint8)
    w13_scales = _c(w13_scales, np.uint8)
    w2_codes = _c(w2_codes, np.uint8)
    w2_scales = _c(w2_scales, np.uint8)
    assert w13_codes.shape[1:] == (2 * I, H // 2) and w2_codes.shape[1:] == (H, I // 2)
    assert 0 <= e < w13_codes.shape[0]
    y = np.empty(H, np.float64)
    mid = np.empty(I, np.uint16)
    _load().oracle_expert(H, I, int(e), _p(n_row), _p(w13_codes), _p(w13_scales), _p(w2_codes),
                          _p(w2_scales), _p(y), _p(mid))
    return y, mid


def shared(n_row, ws13, ws2):
    """One activation row through the bf16 shared expert; returns (ys [H], ms [Is] bits)."""
    n_row = _c(n_row, np.uint16)
    ws13 = _c(ws13, np.uint16)
    ws2 = _c(ws2, np.uint16)
    H = n_row.shape[0]
    Is = ws2.shape[1]
    assert ws13.shape == (2 * Is, H) and ws2.shape == (H, Is)
    ys = np.empty(H, np.float64)
    ms = np.empty(Is, np.uint16)
    _load().oracle_shared(H, Is, _p(n_row), _p(ws13), _p(ws2), _p(ys), _p(ms))
    return ys, ms


def out_proj(attn, w_o):
    """Attention output projection: attn [R,Ha] bf16 bits, w_o [H,Ha] bf16 bits -> x [R,H]
    bf16 bits."""
    attn = _c(attn, np.uint16)
    w_o = _c(w_o, np.uint16)
    R, Ha = attn.shape
    H = w_o.shape[0]
    assert w_o.shape == (H, Ha)
    x = np.empty((R, H), np.uint16)
    _load().oracle_out_proj(R, Ha, H, _p(attn), _p(w_o), _p(x))
    return x


def shared_gate(n, g):
    """Per-row sigmoid gate of the shared expert: n [R,H] bf16 bits, g [H] bf16 bits ->
    [R] float64."""
    n = _c(n, np.uint16)
    g = _c(g, np.uint16)
    R, H = n.shape
    assert g.shape == (H,)
    gate = np.empty(R, np.float64)
    _load().oracle_shared_gate(R, H, _p(n), _p(g), _p(gate))
    return gate


def moe_tail(inputs: dict, k: int, eps: float, nthreads: int = 1):
    """The whole tail.  `inputs` holds the arrays made by moe_layer_tail_gb300.inputs; an
    optional "ws_gate" [H] (bf16 bits) gates the shared expert's output per row; with
    "w_o" [H,Ha] and "attn" [R,Ha] the input x is the projection out_proj(attn, w_o).

    Returns dict(out [R,H] bf16 bits, out_exact [R,H] float64 (before the bf16 rounding),
    residual [R,H] bf16 bits (r_new), ids [R,k], wts [R,k] float64, logits [R,E] float64).
    The caller's arrays are not modified.
    """
    if inputs.get("w_o") is not None:
        x = out_proj(inputs["attn"], inputs["w_o"])
    else:
        x = _c(inputs["x"], np.uint16)
    res = np.array(inputs["residual"], dtype=np.uint16, copy=True, order="C")
    gamma = _c(inputs["gamma"], np.uint16)
    w_r = _c(inputs["w_r"], np.uint16)
    w13c = _c(inputs["w13_codes"], np.uint8)
    w13s = _c(inputs["w13_scales"], np.uint8)
    w2c = _c(inputs["w2_codes"], np.uint8)
    w2s = _c(inputs["w2_scales"], np.uint8)
    ws13 = _c(inputs["ws13"], np.uint16)
    ws2 = _c(inputs["ws2"], np.uint16)
    wsg = _c(inputs["ws_gate"], np.uint16) if inputs.get("ws_gate") is not None else None
    R, H = x.shape
    E = w_r.shape[0]
    I = w2c.shape[2] * 2
    Is = ws2.shape[1]
    out = np.empty((R, H), np.uint16)
    ids = np.empty((R, k), np.int32)
    wts = np.empty((R, k), np.float64)
    logits = np.empty((R, E), np.float64)
    exact = np.empty((R, H), np.float64)
    rc = _load().oracle_moe_tail_gated(R, H, E, int(k), I, Is, float(eps), _p(x), _p(res),
                                       _p(gamma), _p(w_r), _p(w13c), _p(w13s), _p(w2c),
                                       _p(w2s), _p(ws13), _p(ws2), _p(wsg), _p(out), _p(ids),
                                       _p(wts), _p(logits), _p(exact), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_moe_tail rejected the shapes (rc=%d)" % rc)
    return dict(out=out, out_exact=exact, residual=res, ids=ids, wts=wts, logits=logits)


def attnres_mix(sub, prefix, blocks, n_blocks: int, commit: bool, q, gamma, eps: float):
    """One call of the AttnRes residual mix + RMSNorm for R rows.

    sub, prefix [R,H] bf16 bits; blocks [B,R,H] bf16 bits with B > n_blocks when commit
    (blocks 0 .. n_blocks-1 are the committed sources); q, gamma [H] bf16 bits.
    Returns dict(prefix [R,H] (zero after a commit), blocks (block n_blocks holds the
    committed prefix after a commit), mix [R,H], y [R,H], alpha [R,S], score [R,S]) with
    S = n_blocks + 1; the caller's arrays are not modified.
    """
    sub = _c(sub, np.uint16)
    pre = np.array(prefix, dtype=np.uint16, copy=True, order="C")
    blk = np.array(blocks, dtype=np.uint16, copy=True, order="C")
    q = _c(q, np.uint16)
    gamma = _c(gamma, np.uint16)
    R, H = sub.shape
    assert pre.shape == (R, H) and q.shape == (H,) and gamma.shape == (H,)
    assert blk.ndim == 3 and blk.shape[1:] == (R, H)
    assert blk.shape[0] >= n_blocks + (1 if commit else 0)
    S = n_blocks + 1
    mix = np.empty((R, H), np.uint16)
    y = np.empty((R, H), np.uint16)
    alpha = np.empty((R, S), np.float64)
    score = np.empty((R, S), np.float64)
    rc = _load().oracle_attnres_mix(R, H, int(n_blocks), int(bool(commit)), float(eps),
                                    _p(sub), _p(pre), _p(blk), _p(q), _p(gamma), _p(mix),
                                    _p(y), _p(alpha), _p(score))
    if rc != 0:
        raise ValueError("oracle_attnres_mix rejected the shapes (rc=%d)" % rc)
    return dict(prefix=pre, blocks=blk, mix=mix, y=y, alpha=alpha, score=score)


def bf16_bits_to_f64(a):
    """uint16 bf16 bits -> float64 (exact), vectorised."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1
