"""CUDA AttnRes mix vs the oracle, element by element, through the C ABI (attnres_mix.h).

Covers one-CTA, two-CTA and eight-CTA rows (the thread-block cluster per row), one source
and the maximum of 32, commits, the largest hidden size and row count, both input families
(unit and large-magnitude rows), the full 187-call decoder sequence at 1, 8 and 16 rows,
determinism, CUDA-graph replay with and without programmatic dependent launches, and the
refusal codes on a real device.

Tolerances (derived from the arithmetic: fp32 partial sums and scores on the GPU, fp64 in
the oracle):
  prefix, committed blocks  bit-exact (one rounding of an exact bf16 + bf16 sum);
  mixture                   within one bf16 step of the oracle's value, plus 2^-16 of
                            sum_i alpha_i |v_i| for the fp32 accumulation and the fp32
                            weights (elements whose exact value sits at a rounding boundary
                            or cancels to near zero);
  y                         within one bf16 step (plus 2^-16 relative) of the fp64 RMSNorm of
                            the GPU's own mixture; against the oracle's y, within a bf16 step
                            on each side plus the difference of the two mixtures carried
                            through the norm (|dmix| rstd |gamma|), cosine >= 0.99999 per row.
"""
import numpy as np
import pytest

import oracle
from moe_layer_tail_gb300 import (ATTNRES_MIX_DEBUG_STALL, ATTNRES_MIX_PDL, ERR_INVALID_ARG,
                                  ERR_UNSUPPORTED, STATUS_TIMEOUT, MoeTailError, acts_to_device,
                                  attnres_mix, attnres_mix_ctas_per_row, attnres_mix_status,
                                  bf16_tensor_to_bits)
from moe_layer_tail_gb300 import inputs as gen
from parity import bf16_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def _step(v):
    """The spacing of bf16 values at the magnitude of each float64 value."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(int) - 7)


def _inputs(R, H, n_blocks, seed, family="unit", commit=False):
    rng = np.random.default_rng([seed, 91])
    sub = rng.standard_normal(size=(R, H)).astype(np.float32)
    pre = rng.standard_normal(size=(R, H)).astype(np.float32)
    blk = rng.standard_normal(size=(n_blocks, R, H)).astype(np.float32)
    if family == "scaled":
        sub *= np.exp2(rng.integers(0, 12, size=(R, 1))).astype(np.float32)
        pre *= np.exp2(rng.integers(0, 12, size=(R, 1))).astype(np.float32)
        blk *= np.exp2(rng.integers(0, 12, size=(n_blocks, R, 1))).astype(np.float32)
    blocks = np.zeros((n_blocks + (1 if commit else 0), R, H), np.uint16)
    blocks[:n_blocks] = gen.to_bf16_bits(blk)
    q = gen.to_bf16_bits(rng.standard_normal(size=H).astype(np.float32) / np.sqrt(H))
    gamma = gen.to_bf16_bits(1.0 + 0.1 * rng.standard_normal(size=H).astype(np.float32))
    return dict(sub=gen.to_bf16_bits(sub), prefix=gen.to_bf16_bits(pre), blocks=blocks, q=q,
                gamma=gamma)


def _to_dev(d):
    return {k: acts_to_device(v) for k, v in d.items()}


def _run(dd, n_blocks, commit, eps=1e-6, flags=0):
    R, H = dd["sub"].shape
    mix = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(mix)
    attnres_mix(dd["sub"], dd["prefix"], dd["blocks"] if dd["blocks"].numel() else None,
                n_blocks, commit, dd["q"], dd["gamma"], mix, y, eps=eps, flags=flags)
    torch.cuda.synchronize()
    return bf16_tensor_to_bits(mix), bf16_tensor_to_bits(y)


def check_mix(gpu_mix, gpu_y, orc, srcs, alpha, gamma, eps):
    """srcs [S,R,H] float64 (the oracle's sources), alpha [R,S] (the oracle's weights)."""
    om = _f64(orc["mix"])
    gm = _f64(gpu_mix)
    absmix = np.einsum("rs,srh->rh", alpha, np.abs(srcs))
    tol = bf16_step(orc["mix"]) + 2.0 ** -16 * absmix
    bad = np.abs(gm - om) > tol
    assert not bad.any(), "mixture off at %d elements, worst %g" % (
        bad.sum(), np.max(np.abs(gm - om) - tol))
    # y against the fp64 RMSNorm of the GPU's own mixture
    rstd = 1.0 / np.sqrt((gm ** 2).mean(axis=1, keepdims=True) + eps)
    yx = gm * rstd * _f64(gamma)[None]
    gy = _f64(gpu_y)
    tol_y = _step(yx) + 2.0 ** -16 * np.abs(yx)
    assert np.all(np.abs(gy - yx) <= tol_y)
    # and against the oracle's y: one rounding step on each side, plus what a differing
    # mixture element carries through the norm
    oy = _f64(orc["y"])
    rstd_o = 1.0 / np.sqrt((om ** 2).mean(axis=1, keepdims=True) + eps)
    tol_o = (_step(oy) + _step(yx) + 1.01 * np.abs(gm - om) * rstd_o * np.abs(_f64(gamma))[None]
             + 2.0 ** -16 * np.abs(oy))
    assert np.all(np.abs(gy - oy) <= tol_o)
    for r in range(oy.shape[0]):
        cos = gy[r] @ oy[r] / (np.linalg.norm(gy[r]) * np.linalg.norm(oy[r]))
        assert cos >= 0.99999, cos


@pytest.mark.parametrize("R,H,n_blocks,commit,family", [
    (1, 7168, 0, False, "unit"),      # one source: the plain add + RMSNorm, 8 CTAs
    (8, 7168, 8, False, "unit"),
    (16, 7168, 8, True, "scaled"),    # large-magnitude rows, commit
    (16, 7168, 31, True, "unit"),     # the maximum source count
    (3, 256, 4, True, "unit"),        # two CTAs per row
    (4, 512, 6, False, "unit"),       # four CTAs per row
    (3, 5408, 12, True, "scaled"),    # four CTAs of 169 vectors (register kernel)
    (2, 7168, 21, False, "unit"),     # 22 sources (register kernel, up to 32)
    (2, 17408, 6, True, "unit"),      # 272-vector chunks: staged kernel, just above 48 KB
    (2, 1000, 3, False, "scaled"),    # one CTA per row, hidden not a multiple of 64
    (5, 8192, 5, False, "unit"),
    (2, 65536, 8, True, "unit"),      # the largest hidden size (staged kernel)
    (4096, 64, 2, True, "unit"),      # the largest row count
])
def test_mix_matches_oracle(R, H, n_blocks, commit, family):
    seed = 1000 + R + H + n_blocks
    d = _inputs(R, H, n_blocks, seed, family, commit)
    eps = 1e-6
    orc = oracle.attnres_mix(d["sub"], d["prefix"], d["blocks"], n_blocks, commit, d["q"],
                             d["gamma"], eps)
    dd = _to_dev(d)
    gm, gy = _run(dd, n_blocks, commit, eps)
    assert np.array_equal(bf16_tensor_to_bits(dd["prefix"]), orc["prefix"])
    assert np.array_equal(bf16_tensor_to_bits(dd["blocks"]), orc["blocks"])
    pre_new = orc["blocks"][n_blocks] if commit else orc["prefix"]
    srcs = np.concatenate([_f64(d["blocks"][:n_blocks]), _f64(pre_new)[None]], axis=0)
    check_mix(gm, gy, orc, srcs, orc["alpha"], d["gamma"], eps)
    if n_blocks == 0:
        assert np.array_equal(gm, pre_new)  # one source: alpha = 1, the mixture is prefix'
    exp_ctas = {7168: 8, 256: 2, 512: 4, 5408: 4, 17408: 8, 1000: 1, 8192: 8, 65536: 8, 64: 1}[H]
    assert attnres_mix_ctas_per_row(H, n_blocks) == exp_ctas


def test_mix_is_deterministic_and_row_independent():
    R, H, nb = 16, 7168, 6
    d = _inputs(R, H, nb, 5)
    runs = []
    for _ in range(3):
        dd = _to_dev(d)
        runs.append(_run(dd, nb, False) + (bf16_tensor_to_bits(dd["prefix"]),))
    for a, b in zip(runs[0], runs[1]):
        assert np.array_equal(a, b)
    for a, b in zip(runs[0], runs[2]):
        assert np.array_equal(a, b)
    # rows 3..5 alone give the same bits as inside the 16-row call
    sl = {k: (v[:, 3:6] if k == "blocks" else v[3:6] if v.ndim == 2 else v) for k, v in d.items()}
    dd = _to_dev(sl)
    gm, gy = _run(dd, nb, False)
    assert np.array_equal(gm, runs[0][0][3:6]) and np.array_equal(gy, runs[0][1][3:6])


def _sequence_on_gpu(seq, dd, flags=0, stream=None):
    L = seq.L
    mix = torch.empty((L, seq.R, seq.H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(mix)
    for l in range(L):
        attnres_mix(dd["sub"][l], dd["prefix"], dd["blocks"], seq.n_blocks(l), seq.commit(l),
                    dd["q"][l], dd["gamma"][l], mix[l], y[l], eps=seq.eps, flags=flags,
                    stream=stream)
    return mix, y


@pytest.mark.parametrize("R,family", [(1, "unit"), (8, "unit"), (16, "scaled")])
def test_decoder_sequence_matches_oracle(R, family):
    seq = gen.MixSequence(R=R)
    d = gen.make_mix_sequence(seq, 2026 + R, family)
    dd = _to_dev(d)
    mix, y = _sequence_on_gpu(seq, dd, flags=ATTNRES_MIX_PDL)
    torch.cuda.synchronize()
    gmix, gy = bf16_tensor_to_bits(mix), bf16_tensor_to_bits(y)
    pre, blk = d["prefix"], d["blocks"]
    for l in range(seq.L):
        nb, com = seq.n_blocks(l), seq.commit(l)
        orc = oracle.attnres_mix(d["sub"][l], pre, blk, nb, com, d["q"][l], d["gamma"][l],
                                 seq.eps)
        pre_new = orc["blocks"][nb] if com else orc["prefix"]
        srcs = np.concatenate([_f64(blk[:nb]), _f64(pre_new)[None]], axis=0)
        check_mix(gmix[l], gy[l], orc, srcs, orc["alpha"], d["gamma"][l], seq.eps)
        pre, blk = orc["prefix"], orc["blocks"]
    assert np.array_equal(bf16_tensor_to_bits(dd["prefix"]), pre)
    assert np.array_equal(bf16_tensor_to_bits(dd["blocks"]), blk)
    assert attnres_mix_status() == 0


@pytest.mark.parametrize("flags", [0, ATTNRES_MIX_PDL])
def test_decoder_sequence_graph_replays_match_eager(flags):
    seq = gen.MixSequence(R=8)
    d = gen.make_mix_sequence(seq, 77)
    dd = _to_dev(d)
    pre0, blk0 = dd["prefix"].clone(), dd["blocks"].clone()
    mix_e, y_e = _sequence_on_gpu(seq, dd, flags)
    torch.cuda.synchronize()
    ref = [bf16_tensor_to_bits(t) for t in (mix_e, y_e, dd["prefix"], dd["blocks"])]
    dd["prefix"].copy_(pre0)
    dd["blocks"].copy_(blk0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mix_g, y_g = _sequence_on_gpu(seq, dd, flags)
    # 2,000 replays of the 187-call sequence, compared with the eager run every 500
    for i in range(2000):
        dd["prefix"].copy_(pre0)
        dd["blocks"].copy_(blk0)
        g.replay()
        if i % 500 == 499:
            torch.cuda.synchronize()
            got = [bf16_tensor_to_bits(t) for t in (mix_g, y_g, dd["prefix"], dd["blocks"])]
            for a, b in zip(ref, got):
                assert np.array_equal(a, b)


def test_mix_refusals_on_device():
    d = _to_dev(_inputs(2, 7168, 2, 9))
    mix = torch.empty((2, 7168), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(mix)
    with pytest.raises(MoeTailError) as e:
        attnres_mix(d["sub"], d["prefix"], d["blocks"], 32, False, d["q"], d["gamma"], mix, y)
    assert e.value.code == ERR_UNSUPPORTED
    with pytest.raises(MoeTailError) as e:
        attnres_mix(d["sub"], d["prefix"], d["blocks"], 2, False, d["q"], d["gamma"], mix, y,
                    eps=0.0)
    assert e.value.code == ERR_INVALID_ARG
    # a misaligned view (one element in) is refused, nothing launched
    flat = torch.empty(2 * 7168 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeTailError) as e:
        attnres_mix(flat[1:1 + 2 * 7168].view(2, 7168), d["prefix"], d["blocks"], 2, False,
                    d["q"], d["gamma"], mix, y)
    assert e.value.code == ERR_INVALID_ARG
    # the inputs were not touched
    assert np.array_equal(bf16_tensor_to_bits(d["prefix"]), _inputs(2, 7168, 2, 9)["prefix"])


def test_stalled_exchange_is_reported_and_the_device_stays_usable():
    # one CTA waits for a partial sum that never comes: its bounded wait gives up, the
    # status word says so, the call still completes with the right results (every real
    # value had arrived), and the next call runs normally
    R, H, nb = 4, 7168, 5
    d = _inputs(R, H, nb, 21)
    ref_m, ref_y = _run(_to_dev(d), nb, False)
    assert attnres_mix_status(clear=True) == 0
    gm, gy = _run(_to_dev(d), nb, False, flags=ATTNRES_MIX_DEBUG_STALL)
    assert attnres_mix_status(clear=True) & STATUS_TIMEOUT
    assert np.array_equal(gm, ref_m) and np.array_equal(gy, ref_y)
    gm2, gy2 = _run(_to_dev(d), nb, False)
    assert attnres_mix_status() == 0
    assert np.array_equal(gm2, ref_m) and np.array_equal(gy2, ref_y)
