"""Pins of the CPU oracle against what the number formats and the mathematics fix.

Each test checks the oracle against something other than itself: the OCP bit-field
definitions, exact closed forms, brute force with numpy/scipy on tiny shapes, and special
cases (k = E is the plain softmax, identical experts make the output independent of the
routing, zero routed weights leave the shared expert alone, scaling w2 by two doubles the
routed part).  A plausible slip in the oracle (a dropped term, a swapped nibble, a wrong
sign or index, gate and up swapped, a missing renormalisation) fails at least one of them.
"""
import math
import struct

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from helpers import (bf16_decode, e2m1_value_from_bits, is_nearest_bf16, np_mxfp4_dequant,
                     quantize_to_nearest_bf16_bits, silu)
from moe_layer_tail_gb300 import inputs as gen

# ------------------------------------------------------------------ formats ----


def test_e2m1_all_codes_match_bit_fields_and_ocp_table():
    ocp_magnitudes = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for code in range(16):
        v = oracle.e2m1(code)
        assert v == e2m1_value_from_bits(code)
        assert abs(v) == ocp_magnitudes[code & 7]
        assert math.copysign(1.0, v) == (-1.0 if code & 8 else 1.0)


def _e8m0_by_float_bits(s: int) -> float:
    if s == 0:
        return struct.unpack("<f", struct.pack("<I", 0x00400000))[0]  # 2^-127, subnormal
    return struct.unpack("<f", struct.pack("<I", s << 23))[0]


@pytest.mark.parametrize("s", [0, 1, 126, 127, 128, 254])
def test_e8m0_times_e2m1_exhaustive(s):
    assert oracle.e8m0(s) == _e8m0_by_float_bits(s)
    # one 32-element block holding every code twice, decoded through the packed-row routine
    codes = np.array([(c & 15) | (((c + 1) & 15) << 4) for c in range(0, 32, 2)], np.uint8)
    row = oracle.mxfp4_dequant_row(codes, np.array([s], np.uint8), 32)
    expect = [e2m1_value_from_bits(k & 15) * math.ldexp(1.0, s - 127) for k in range(32)]
    assert row.tolist() == expect


@pytest.mark.parametrize("idx", [0, 1, 2, 7, 30, 31, 32, 33, 62, 63])
def test_nibble_order_single_nonzero(idx):
    K = 64
    codes = np.zeros(K // 2, np.uint8)
    codes[idx // 2] = (0x3 << 4) if idx % 2 else 0x3  # code 3 = 1.5
    scales = np.array([127, 128], np.uint8)           # block 0 x1, block 1 x2
    row = oracle.mxfp4_dequant_row(codes, scales, K)
    expect = np.zeros(K)
    expect[idx] = 1.5 * (2.0 if idx >= 32 else 1.0)
    assert np.array_equal(row, expect)


def test_mxfp4_pack_roundtrip_and_numpy_decoder_agree():
    rng = np.random.default_rng(11)
    K = 256
    codes_unpacked = rng.integers(0, 16, K)
    scales = rng.integers(100, 150, K // 32).astype(np.uint8)
    exact = np.array([e2m1_value_from_bits(int(c)) for c in codes_unpacked]) * \
        np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32)
    packed = (codes_unpacked[0::2] | (codes_unpacked[1::2] << 4)).astype(np.uint8)
    assert np.array_equal(oracle.mxfp4_dequant_row(packed, scales, K), exact)
    assert np.array_equal(np_mxfp4_dequant(packed, scales), exact)


def test_bf16_round_hand_cases():
    u = 2.0 ** -8
    cases = [
        (1.0, 0x3F80), (1.0 + u, 0x3F80),               # tie -> even (down)
        (1.0 + 3 * u, 0x3F82),                          # tie -> even (up)
        (1.0 + u + 2.0 ** -30, 0x3F81),                 # just above the tie
        (-1.0 - u - 2.0 ** -30, 0xBF81),
        (0.0, 0x0000), (-0.0, 0x8000),
        (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),   # smallest subnormal; tie to zero
        (3 * 2.0 ** -134, 0x0002),                      # 1.5 quanta -> 2 (even)
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),         # largest finite
        (2.0 ** 128, 0x7F80), (-2.0 ** 130, 0xFF80),    # overflow -> inf
        (float("inf"), 0x7F80),
    ]
    for v, bits in cases:
        assert oracle.bf16_round(v) == bits, (v, hex(oracle.bf16_round(v)), hex(bits))
    assert (oracle.bf16_round(float("nan")) & 0x7FC0) == 0x7FC0


def test_bf16_round_matches_torch_on_float32_inputs():
    # float32 -> bf16 is a single rounding in torch; the oracle rounds the same value once.
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 10,
                        rng.standard_normal(1000).astype(np.float32) * 1e-38,
                        (rng.standard_normal(1000) * 1e30).astype(np.float32)])
    t = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(x)) for x in v], np.uint16)
    assert np.array_equal(got, t)


def test_bf16_round_is_nearest_on_float64_inputs():
    rng = np.random.default_rng(6)
    v = rng.standard_normal(2000) * np.exp(rng.uniform(-30, 30, 2000))
    got = np.array([oracle.bf16_round(float(x)) for x in v], np.uint16)
    assert is_nearest_bf16(got, v, slack=0).all()
    assert np.array_equal(got, quantize_to_nearest_bf16_bits(v))


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(50.0) == pytest.approx(50.0, rel=1e-15)
    assert abs(oracle.silu(-50.0)) < 1e-19
    for z in (-3.0, -0.5, 0.7, 2.0):
        assert oracle.silu(z) == pytest.approx(z * scipy.special.expit(z), rel=1e-15)


# --------------------------------------------------------- residual add + RMSNorm ----


def test_rmsnorm_constant_row_closed_form():
    H, eps = 64, 1e-6
    rng = np.random.default_rng(3)
    gamma = gen.to_bf16_bits(1 + 0.1 * rng.standard_normal(H))
    for c in (0.75, -2.5, 1e-3, 96.0):
        x = np.full((1, H), gen.to_bf16_bits(np.array([c]))[0], np.uint16)
        res = np.zeros((1, H), np.uint16)
        r_new, n, rstd = oracle.add_rmsnorm(x, res, gamma, eps)
        cb = float(bf16_decode(x[0, 0]))
        assert np.array_equal(r_new, x)
        assert rstd[0] == pytest.approx(1.0 / math.sqrt(cb * cb + eps), rel=1e-15)
        exact = np.sign(cb) * bf16_decode(gamma) * abs(cb) / math.sqrt(cb * cb + eps)
        assert is_nearest_bf16(n[0], exact, slack=1e-12).all()


def test_residual_add_rounds_once_and_rows_are_independent():
    rng = np.random.default_rng(4)
    R, H = 3, 96
    x = gen.to_bf16_bits(rng.standard_normal((R, H)))
    res = gen.to_bf16_bits(rng.standard_normal((R, H)) * 300)
    gamma = gen.to_bf16_bits(np.ones(H))
    r_new, n, rstd = oracle.add_rmsnorm(x, res, gamma, 1e-6)
    exact = bf16_decode(x) + bf16_decode(res)
    assert is_nearest_bf16(r_new, exact, slack=0).all()
    # each row alone gives the same result
    for r in range(R):
        r1, n1, _ = oracle.add_rmsnorm(x[r:r + 1], res[r:r + 1], gamma, 1e-6)
        assert np.array_equal(r1[0], r_new[r]) and np.array_equal(n1[0], n[r])
    # the norm uses the rounded sum: rms of gamma=1 output is ~1
    nv = bf16_decode(n)
    assert np.allclose(np.sqrt((nv ** 2).mean(axis=1)), 1.0, rtol=2e-3)
    rv = bf16_decode(r_new)
    want = rv / np.sqrt((rv ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert is_nearest_bf16(n, want, slack=1e-12).all()


# --------------------------------------------------------------- router + top-k ----


def test_router_matches_numpy_dot():
    rng = np.random.default_rng(7)
    R, H, E = 3, 64, 6
    n = gen.to_bf16_bits(rng.standard_normal((R, H)))
    w = gen.to_bf16_bits(rng.standard_normal((E, H)) / 8)
    got = oracle.router(n, w)
    want = bf16_decode(n) @ bf16_decode(w).T
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    assert not np.allclose(got, bf16_decode(n) @ bf16_decode(w)[::-1].T)


def _brute_topk(l, k):
    order = sorted(range(len(l)), key=lambda e: (-np.float32(l[e]), e))
    return order[:k]


def test_topk_bruteforce_order_and_weights():
    rng = np.random.default_rng(8)
    R, E, k = 6, 12, 4
    logits = rng.standard_normal((R, E))
    ids, wts = oracle.topk(logits, k)
    for r in range(R):
        assert ids[r].tolist() == _brute_topk(logits[r], k)
        p = scipy.special.softmax(logits[r])
        want = p[ids[r]] / p[ids[r]].sum()
        assert np.allclose(wts[r], want, rtol=1e-13)
        assert np.allclose(wts[r], scipy.special.softmax(logits[r][ids[r]]), rtol=1e-13)
        assert abs(wts[r].sum() - 1.0) < 1e-12
        assert np.all(np.diff(wts[r]) <= 0)  # pick order = descending weight


def test_topk_k_equals_E_is_plain_softmax():
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((2, 9)) * 3
    ids, wts = oracle.topk(logits, 9)
    for r in range(2):
        assert sorted(ids[r].tolist()) == list(range(9))
        assert np.allclose(wts[r], scipy.special.softmax(logits[r])[ids[r]], rtol=1e-13)


def test_topk_exact_ties_pick_lowest_id_in_order():
    logits = np.array([[0.5, 2.0, 1.0, 2.0, 1.0, -1.0, 1.0]])
    ids, wts = oracle.topk(logits, 4)
    assert ids[0].tolist() == [1, 3, 2, 4]
    assert wts[0][0] == wts[0][1] and wts[0][2] == wts[0][3]
    # the rank key is the fp32 logit: values equal in fp32 tie even if they differ in fp64
    a = 1.0
    b = 1.0 + 2.0 ** -40
    ids, _ = oracle.topk(np.array([[a, 0.0, b]]), 1)
    assert ids[0, 0] == 0


def test_router_identical_rows_tie_to_lowest_id():
    rng = np.random.default_rng(10)
    H, E = 64, 8
    n = gen.to_bf16_bits(rng.standard_normal((1, H)))
    w = gen.to_bf16_bits(rng.standard_normal((E, H)) / 8)
    l0 = oracle.router(n, w)[0]
    top = int(np.argmax(l0))
    w[5] = w[top] if top != 5 else w[2]
    twin = top if top != 5 else 2
    ids, _ = oracle.topk(oracle.router(n, w), 2)
    assert ids[0].tolist() == [min(twin, 5), max(twin, 5)]


# ------------------------------------------------------------------- experts ----


def _tiny_weights(seed, H=64, I=32, E=3, Is=32):
    return gen.make_weights(gen.TailShape(1, H, E, 2, I, Is), seed)


def test_routed_expert_bruteforce():
    w = _tiny_weights(12)
    H = w["w13_codes"].shape[2] * 2
    I = w["w2_codes"].shape[2] * 2
    rng = np.random.default_rng(12)
    n = gen.to_bf16_bits(rng.standard_normal(H))
    for e in range(3):
        y, mid = oracle.expert(n, e, w["w13_codes"], w["w13_scales"], w["w2_codes"],
                               w["w2_scales"])
        W13 = np_mxfp4_dequant(w["w13_codes"][e], w["w13_scales"][e])
        W2 = np_mxfp4_dequant(w["w2_codes"][e], w["w2_scales"][e])
        nv = bf16_decode(n)
        g, u = W13[:I] @ nv, W13[I:] @ nv
        assert is_nearest_bf16(mid, silu(g) * u, slack=1e-12).all()
        # gate and up are not interchangeable: swapping them changes mid
        assert not np.array_equal(quantize_to_nearest_bf16_bits(silu(u) * g), mid)
        assert np.allclose(y, W2 @ bf16_decode(mid), rtol=1e-12, atol=1e-12)


def test_shared_expert_bruteforce():
    w = _tiny_weights(13)
    H, Is = w["ws2"].shape
    rng = np.random.default_rng(13)
    n = gen.to_bf16_bits(rng.standard_normal(H))
    ys, ms = oracle.shared(n, w["ws13"], w["ws2"])
    W13 = bf16_decode(w["ws13"])
    nv = bf16_decode(n)
    g, u = W13[:Is] @ nv, W13[Is:] @ nv
    assert is_nearest_bf16(ms, silu(g) * u, slack=1e-12).all()
    assert np.allclose(ys, bf16_decode(w["ws2"]) @ bf16_decode(ms), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------- the whole tail ----


def _tail_inputs(seed, R=3, H=64, E=6, k=2, I=32, Is=32):
    shape = gen.TailShape(R, H, E, k, I, Is)
    d = gen.make_weights(shape, seed)
    d.update(gen.make_activations(shape, seed))
    return shape, d


def _numpy_tail(d, k, eps):
    """Whole tail by brute force with numpy, independent of the oracle's code."""
    x, res = bf16_decode(d["x"]), bf16_decode(d["residual"])
    r_new = quantize_to_nearest_bf16_bits(x + res).reshape(x.shape)
    rv = bf16_decode(r_new)
    rstd = 1.0 / np.sqrt((rv ** 2).mean(axis=1, keepdims=True) + eps)
    n = bf16_decode(quantize_to_nearest_bf16_bits(rv * rstd * bf16_decode(d["gamma"])))
    n = n.reshape(x.shape)
    logits = n @ bf16_decode(d["w_r"]).T
    E = logits.shape[1]
    I = d["w2_codes"].shape[2] * 2
    Is = d["ws2"].shape[1]
    out = np.zeros_like(x)
    W13s, W2s = bf16_decode(d["ws13"]), bf16_decode(d["ws2"])
    for r in range(x.shape[0]):
        ids = _brute_topk(logits[r], k)
        p = scipy.special.softmax(logits[r])
        wts = p[ids] / p[ids].sum()
        acc = np.zeros(x.shape[1])
        for i, e in enumerate(ids):
            W13 = np_mxfp4_dequant(d["w13_codes"][e], d["w13_scales"][e])
            W2 = np_mxfp4_dequant(d["w2_codes"][e], d["w2_scales"][e])
            g, u = W13[:I] @ n[r], W13[I:] @ n[r]
            mid = bf16_decode(quantize_to_nearest_bf16_bits(silu(g) * u))
            acc += wts[i] * (W2 @ mid)
        g, u = W13s[:Is] @ n[r], W13s[Is:] @ n[r]
        ms = bf16_decode(quantize_to_nearest_bf16_bits(silu(g) * u))
        gate = 1.0
        if d.get("ws_gate") is not None:
            gate = scipy.special.expit(n[r] @ bf16_decode(d["ws_gate"]))
        acc += gate * (W2s @ ms)
        out[r] = acc
    return r_new, out


def test_whole_tail_matches_numpy_bruteforce():
    shape, d = _tail_inputs(21)
    got = oracle.moe_tail(d, shape.k, shape.eps)
    r_new, out_exact = _numpy_tail(d, shape.k, shape.eps)
    assert np.array_equal(got["residual"], r_new)
    assert is_nearest_bf16(got["out"], out_exact, slack=1e-9).all()
    # the exact (pre-rounding) output agrees with the brute force, and rounds to `out`
    assert np.allclose(got["out_exact"], out_exact, rtol=1e-10, atol=1e-12)
    assert np.array_equal(got["out"], quantize_to_nearest_bf16_bits(got["out_exact"]).reshape(got["out"].shape))
    assert abs(got["wts"].sum(axis=1) - 1).max() < 1e-12


def test_identical_experts_make_output_routing_independent():
    shape, d = _tail_inputs(22, R=4, E=5, k=3)
    for key in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        d[key] = np.repeat(d[key][:1], shape.E, axis=0)
    got = oracle.moe_tail(d, shape.k, shape.eps)
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    for r in range(shape.R):
        y, _ = oracle.expert(n[r], 0, d["w13_codes"], d["w13_scales"], d["w2_codes"],
                             d["w2_scales"])
        ys, _ = oracle.shared(n[r], d["ws13"], d["ws2"])
        assert is_nearest_bf16(got["out"][r], y + ys, slack=1e-12).all()


def test_zero_routed_weights_leave_shared_expert():
    shape, d = _tail_inputs(23)
    d["w13_codes"][:] = 0
    d["w2_codes"][:] = 0
    got = oracle.moe_tail(d, shape.k, shape.eps)
    r_new, out_exact = _numpy_tail(d, shape.k, shape.eps)
    assert is_nearest_bf16(got["out"], out_exact, slack=1e-9).all()
    assert np.count_nonzero(got["out"]) > 0


def test_doubling_w2_scales_doubles_routed_part_exactly():
    shape, d = _tail_inputs(24)
    d["ws2"][:] = 0  # remove the shared expert's contribution
    base = oracle.moe_tail(d, shape.k, shape.eps)
    d2 = dict(d)
    d2["w2_scales"] = (d["w2_scales"].astype(np.int32) + 1).astype(np.uint8)
    twice = oracle.moe_tail(d2, shape.k, shape.eps)
    assert np.array_equal(bf16_decode(twice["out"]), 2 * bf16_decode(base["out"]))
    assert np.array_equal(twice["ids"], base["ids"])


# ------------------------------------------------------- shared-expert gate ----


def _gate_vector(seed, H):
    rng = np.random.default_rng(seed)
    return gen.to_bf16_bits(rng.standard_normal(H) / np.sqrt(H))


def test_shared_gate_matches_scipy_expit():
    shape, d = _tail_inputs(26, R=5)
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    g = _gate_vector(26, shape.H)
    got = oracle.shared_gate(n, g)
    want = scipy.special.expit(bf16_decode(n).reshape(shape.R, shape.H) @ bf16_decode(g))
    assert np.allclose(got, want, rtol=1e-14, atol=0)
    assert (got > 0).all() and (got < 1).all()


def test_gated_tail_matches_numpy_bruteforce():
    shape, d = _tail_inputs(27)
    d["ws_gate"] = _gate_vector(27, shape.H)
    got = oracle.moe_tail(d, shape.k, shape.eps)
    _, out_exact = _numpy_tail(d, shape.k, shape.eps)
    assert np.allclose(got["out_exact"], out_exact, rtol=1e-10, atol=1e-12)
    ungated = oracle.moe_tail({k: v for k, v in d.items() if k != "ws_gate"}, shape.k, shape.eps)
    assert not np.array_equal(got["out"], ungated["out"])
    assert np.array_equal(got["ids"], ungated["ids"])  # the gate does not touch the routing


def test_zero_gate_halves_the_shared_part_exactly():
    # sigmoid(0) = 1/2, applied to the shared expert's output only: the same as halving every
    # shared down weight (an exact exponent decrement for these normal bf16 values)
    shape, d = _tail_inputs(28)
    gated = dict(d)
    gated["ws_gate"] = np.zeros(shape.H, np.uint16)
    a = oracle.moe_tail(gated, shape.k, shape.eps)
    half = dict(d)
    ws2 = d["ws2"].astype(np.uint32)
    exp = (ws2 >> 7) & 0xFF
    assert ((exp > 1) | (ws2 & 0x7FFF == 0)).all()
    half["ws2"] = np.where(ws2 & 0x7FFF, ws2 - 0x80, ws2).astype(np.uint16)
    b = oracle.moe_tail(half, shape.k, shape.eps)
    assert np.array_equal(a["out_exact"], b["out_exact"])
    assert np.array_equal(a["out"], b["out"])


def test_closed_gate_removes_the_shared_expert():
    # a gate vector anti-parallel to the row's activations drives the logit far below -745,
    # where e^-z overflows and the gate is exactly 0: the output is the routed part alone
    shape, d = _tail_inputs(29, R=1)
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    gated = dict(d)
    gated["ws_gate"] = gen.to_bf16_bits(-64.0 * bf16_decode(n[0]))
    assert oracle.shared_gate(n, gated["ws_gate"])[0] == 0.0
    a = oracle.moe_tail(gated, shape.k, shape.eps)
    no_shared = dict(d)
    no_shared["ws2"] = np.zeros_like(d["ws2"])
    b = oracle.moe_tail(no_shared, shape.k, shape.eps)
    assert np.array_equal(a["out_exact"], b["out_exact"])


# --------------------------------------------------- attention out_proj ----


def test_out_proj_matches_numpy_dot():
    rng = np.random.default_rng(30)
    R, Ha, H = 3, 96, 64
    attn = gen.to_bf16_bits(rng.standard_normal((R, Ha)))
    w_o = gen.to_bf16_bits(rng.standard_normal((H, Ha)) / np.sqrt(Ha))
    x = oracle.out_proj(attn, w_o)
    want = bf16_decode(attn).reshape(R, Ha) @ bf16_decode(w_o).reshape(H, Ha).T
    assert is_nearest_bf16(x, want, slack=1e-12).all()


def test_out_proj_with_a_selection_matrix_copies_its_input():
    # w_o = [identity | 0]: x is the first H columns of attn, bit for bit
    rng = np.random.default_rng(31)
    R, Ha, H = 4, 96, 64
    attn = gen.to_bf16_bits(rng.standard_normal((R, Ha)))
    w_o = np.zeros((H, Ha), np.uint16)
    w_o[np.arange(H), np.arange(H)] = 0x3F80  # bf16 1.0
    assert np.array_equal(oracle.out_proj(attn, w_o), attn[:, :H])


def test_tail_from_attention_output_projects_first():
    shape, d = _tail_inputs(32)
    rng = np.random.default_rng(32)
    Ha = 96
    d2 = {k: v for k, v in d.items() if k != "x"}
    d2["attn"] = gen.to_bf16_bits(rng.standard_normal((shape.R, Ha)))
    d2["w_o"] = gen.to_bf16_bits(rng.standard_normal((shape.H, Ha)) / np.sqrt(Ha))
    got = oracle.moe_tail(d2, shape.k, shape.eps)
    d3 = dict(d)
    d3["x"] = quantize_to_nearest_bf16_bits(
        bf16_decode(d2["attn"]).reshape(shape.R, Ha) @ bf16_decode(d2["w_o"]).reshape(shape.H, Ha).T
    ).reshape(shape.R, shape.H)
    _, out_exact = _numpy_tail(d3, shape.k, shape.eps)
    assert np.allclose(got["out_exact"], out_exact, rtol=1e-10, atol=1e-12)


def test_oracle_is_deterministic_and_thread_count_invariant():
    shape, d = _tail_inputs(25, R=4, E=8, k=3)
    a = oracle.moe_tail(d, shape.k, shape.eps, nthreads=1)
    b = oracle.moe_tail(d, shape.k, shape.eps, nthreads=1)
    c = oracle.moe_tail(d, shape.k, shape.eps, nthreads=5)
    for key in ("out", "residual", "ids", "wts", "logits"):
        assert np.array_equal(a[key], b[key]) and np.array_equal(a[key], c[key])


def test_tiny_workload_runs_and_inputs_are_reproducible():
    d1 = gen.make_inputs("tiny")
    d2 = gen.make_inputs("tiny")
    for key in d1:
        assert np.array_equal(d1[key], d2[key])
    wl = gen.WORKLOADS["tiny"]
    got = oracle.moe_tail(d1, wl.shape.k, wl.shape.eps)
    assert got["out"].shape == (1, 256)
    assert np.isfinite(bf16_decode(got["out"])).all()


# ------------------------------------------------ AttnRes residual mix (second workload) ----

def _mix_inputs(R, H, n_blocks, seed, B=None):
    rng = np.random.default_rng([seed, 77])

    def bits(shape, std=1.0):
        return gen.to_bf16_bits(rng.standard_normal(size=shape).astype(np.float32) * std)

    B = n_blocks + 1 if B is None else B
    blocks = np.zeros((B, R, H), np.uint16)
    blocks[:n_blocks] = bits((n_blocks, R, H))
    return dict(sub=bits((R, H)), prefix=bits((R, H)), blocks=blocks,
                q=bits((H,), 1.0 / math.sqrt(H)),
                gamma=gen.to_bf16_bits(1.0 + 0.1 * rng.standard_normal(size=H).astype(np.float32)))


def _mix(d, n_blocks, commit=False, eps=1e-6):
    return oracle.attnres_mix(d["sub"], d["prefix"], d["blocks"], n_blocks, commit, d["q"],
                              d["gamma"], eps)


def test_mix_with_no_committed_block_is_the_plain_add_rmsnorm():
    d = _mix_inputs(3, 256, 0, 1)
    m = _mix(d, 0)
    r_new, n, _ = oracle.add_rmsnorm(d["sub"], d["prefix"], d["gamma"], 1e-6)
    assert np.all(m["alpha"] == 1.0)
    assert np.array_equal(m["prefix"], r_new)
    assert np.array_equal(m["mix"], r_new)
    assert np.array_equal(m["y"], n)


def test_mix_residual_add_is_the_float32_sum_rounded_once():
    d = _mix_inputs(4, 512, 2, 2)
    m = _mix(d, 2)
    t = (torch.from_numpy(bf16_decode(d["prefix"]).astype(np.float32))
         + torch.from_numpy(bf16_decode(d["sub"]).astype(np.float32))).to(torch.bfloat16)
    assert np.array_equal(m["prefix"], t.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(m["blocks"], d["blocks"])  # no commit: the blocks stay


def test_mix_zero_query_gives_the_plain_mean():
    R, H, nb = 2, 128, 3
    d = _mix_inputs(R, H, nb, 3)
    d["q"] = np.zeros(H, np.uint16)
    m = _mix(d, nb)
    assert np.all(m["alpha"] == 0.25)
    pnew = bf16_decode(m["prefix"])
    srcs = np.concatenate([bf16_decode(d["blocks"][:nb]), pnew[None]], axis=0)
    mean = srcs.sum(axis=0) / 4.0  # exact: four bf16 values of N(0, 1) data
    assert np.array_equal(m["mix"], quantize_to_nearest_bf16_bits(mean.ravel()).reshape(R, H))


def test_mix_scores_and_weights_match_closed_forms():
    # source i = c_i * (a pattern of +-1 with a_i plus signs), q = 1/8 everywhere:
    # q . v_i = c_i (2 a_i - H) / 8 and mean(v_i^2) = c_i^2, so
    # score_i = c_i (2 a_i - H) / 8 / sqrt(c_i^2 + eps) and alpha = softmax(score)
    H, eps = 64, 1e-3
    c = [1.0, 0.25, 2.0 ** -5, 4.0]
    a = [40, 20, 64, 31]
    nb = len(c) - 1
    blocks = np.zeros((nb + 1, 1, H), np.uint16)
    pats = []
    for i in range(len(c)):
        pat = -np.ones(H)
        pat[:a[i]] = 1.0
        np.random.default_rng(i).shuffle(pat)
        pats.append(c[i] * pat)
    for i in range(nb):
        blocks[i, 0] = gen.to_bf16_bits(pats[i])
    d = dict(sub=np.zeros((1, H), np.uint16), prefix=gen.to_bf16_bits(pats[nb])[None],
             blocks=blocks, q=gen.to_bf16_bits(np.full(H, 0.125)),
             gamma=gen.to_bf16_bits(np.ones(H)))
    m = _mix(d, nb, eps=eps)
    score = np.array([c[i] * (2 * a[i] - H) / 8.0 / math.sqrt(c[i] ** 2 + eps)
                      for i in range(len(c))])
    np.testing.assert_allclose(m["score"][0], score, rtol=1e-13, atol=0)
    np.testing.assert_allclose(m["alpha"][0], scipy.special.softmax(score), rtol=1e-13, atol=0)


def test_mix_scores_ignore_a_source_scale():
    d = _mix_inputs(2, 256, 3, 4)
    m = _mix(d, 3, eps=1e-30)  # eps far below ulp(mean(v^2)): the scores are exact ratios
    d8 = dict(d)
    d8["blocks"] = d["blocks"].copy()
    d8["blocks"][1] = gen.to_bf16_bits(bf16_decode(d["blocks"][1]) * 8.0)  # exact
    m8 = _mix(d8, 3, eps=1e-30)
    np.testing.assert_allclose(m8["score"], m["score"], rtol=1e-15, atol=0)


def test_mix_is_the_nearest_bf16_of_the_weighted_sum_and_y_its_rmsnorm():
    R, H, nb = 3, 192, 4
    d = _mix_inputs(R, H, nb, 5)
    m = _mix(d, nb)
    assert np.allclose(m["alpha"].sum(axis=1), 1.0, rtol=0, atol=1e-15)
    srcs = np.concatenate([bf16_decode(d["blocks"][:nb]), bf16_decode(m["prefix"])[None]])
    exact = np.einsum("rs,srh->rh", m["alpha"], srcs)
    assert is_nearest_bf16(m["mix"].ravel(), exact.ravel(), slack=1e-13).all()
    lo, hi = srcs.min(axis=0), srcs.max(axis=0)
    mv = bf16_decode(m["mix"])
    assert np.all(mv >= lo) and np.all(mv <= hi)  # a convex combination
    rstd = 1.0 / np.sqrt((mv ** 2).mean(axis=1, keepdims=True) + 1e-6)
    yx = mv * rstd * bf16_decode(d["gamma"])[None]
    assert is_nearest_bf16(m["y"].ravel(), yx.ravel(), slack=1e-13).all()


def test_mix_commit_stores_the_prefix_and_starts_a_new_block():
    R, H, nb = 2, 128, 2
    d = _mix_inputs(R, H, nb, 6, B=nb + 1)
    plain = _mix(d, nb, commit=False)
    com = _mix(d, nb, commit=True)
    assert np.array_equal(com["blocks"][nb], plain["prefix"])
    assert np.array_equal(com["blocks"][:nb], d["blocks"][:nb])
    assert not com["prefix"].any()
    for k in ("mix", "y", "alpha"):
        assert np.array_equal(com[k], plain[k])


def test_mix_sequence_blocks_are_running_bf16_sums_of_the_sublayer_outputs():
    seq = gen.MixSequence(R=2, H=64, L=11, block_calls=4)
    d = gen.make_mix_sequence(seq, 7)
    pre, blk = d["prefix"], d["blocks"]
    run = torch.zeros(seq.R, seq.H, dtype=torch.bfloat16)
    committed = 1
    for l in range(seq.L):
        m = oracle.attnres_mix(d["sub"][l], pre, blk, seq.n_blocks(l), seq.commit(l), d["q"][l],
                               d["gamma"][l], seq.eps)
        pre, blk = m["prefix"], m["blocks"]
        o = torch.from_numpy(bf16_decode(d["sub"][l]).astype(np.float32))
        run = (run.float() + o).to(torch.bfloat16)
        if seq.commit(l):
            assert np.array_equal(blk[committed], run.view(torch.int16).numpy().view(np.uint16))
            committed += 1
            run.zero_()
        assert np.array_equal(pre, run.view(torch.int16).numpy().view(np.uint16))
    assert committed == seq.max_blocks


def test_mix_permuting_the_committed_blocks_permutes_the_weights():
    R, H, nb = 2, 256, 4
    d = _mix_inputs(R, H, nb, 8)
    m = _mix(d, nb)
    perm = [2, 0, 3, 1]
    dp = dict(d)
    dp["blocks"] = d["blocks"].copy()
    dp["blocks"][:nb] = d["blocks"][perm]
    mp = _mix(dp, nb)
    assert np.array_equal(mp["score"][:, :nb], m["score"][:, perm])
    np.testing.assert_allclose(mp["alpha"][:, :nb], m["alpha"][:, perm], rtol=1e-14, atol=0)
    assert np.abs(mp["mix"].astype(np.int32) - m["mix"].astype(np.int32)).max() <= 1
