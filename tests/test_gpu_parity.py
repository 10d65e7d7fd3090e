"""CUDA path vs the oracle, element by element, through the C ABI.

Covers every workload at full size (all outputs compared), small shapes that span several
tiles with ragged tails, and the edge cases of the method: one row, the maximum row
count, k = 1, k = E, a single expert, identical experts, exact router ties (lowest id
wins), repeated experts across rows, batch invariance, determinism, CUDA-graph replay,
host-buffer runs and the refusal/error codes.
"""
import os

import numpy as np
import pytest

import oracle
from moe_layer_tail_gb300 import (ERR_INVALID_ARG, ERR_UNSUPPORTED, STATUS_BAD_ROUTING, MoeTail,
                                  MoeTailError, acts_to_device, bf16_tensor_to_bits,
                                  weights_to_device)
from moe_layer_tail_gb300 import inputs as gen
from moe_layer_tail_gb300 import MODE_PERSISTENT as MODE_PERSISTENT_ID
from parity import bf16_step, check_parity, inject_near_ties

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NTHREADS = max(1, min(32, os.cpu_count() or 1))


def run_gpu(tail, d, rows=None):
    x = acts_to_device(d["x"])
    res = acts_to_device(d["residual"])
    R = x.shape[0] if rows is None else rows
    out = torch.empty_like(x)
    tail.run(x, res, out, rows=R)
    torch.cuda.synchronize()
    ids, wts, nd = tail.routing(R)
    tail.check_scratch()  # no kernel wrote past the end of a scratch buffer
    return bf16_tensor_to_bits(out[:R]), bf16_tensor_to_bits(res[:R]), ids, wts, nd


_CACHE = {}


def workload_inputs(name):
    if name not in _CACHE:
        _CACHE.clear()
        wl = gen.WORKLOADS[name]
        d = gen.make_inputs(wl)
        if wl.kind == "neartie":
            d["x"], margins = inject_near_ties(d["x"], d["residual"], d["gamma"], d["w_r"],
                                               wl.shape.eps, wl.shape.k)
            assert np.all(np.abs(margins - 1e-2) <= 1.01e-4), margins
        dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
        orc = oracle.moe_tail(d, wl.shape.k, wl.shape.eps, nthreads=NTHREADS)
        _CACHE[name] = (wl, d, dev, orc)
    return _CACHE[name]


@pytest.mark.parametrize("name", list(gen.WORKLOADS))
def test_workload_parity_full_size(name):
    wl, d, dev, orc = workload_inputs(name)
    tail = MoeTail(wl.shape, dev, max_rows=wl.shape.R)
    assert tail.launches_per_run(wl.shape.R) == 5
    out, res, ids, wts, nd = run_gpu(tail, d)
    figs = check_parity(out, res, ids, orc, wl.shape.k)
    assert nd == len(np.unique(orc["ids"]))
    # weights: renormalised softmax of the picked logits.  The GPU's fp32 rstd can round a
    # few elements of n to the other bf16 neighbour than the oracle's fp64 rstd, which moves
    # a logit by ~1e-4 and a weight by up to ~1e-4: allow 5e-4.
    for r in range(wl.shape.R):
        if set(ids[r]) == set(orc["ids"][r]):
            o = {e: w for e, w in zip(orc["ids"][r], orc["wts"][r])}
            g = {e: w for e, w in zip(ids[r], wts[r])}
            assert max(abs(o[e] - g[e]) for e in o) < 5e-4
        assert abs(float(wts[r].sum()) - 1.0) < 1e-5
    assert tail.status() == 0
    if wl.kind == "similar" and wl.shape.R == 8:
        assert 0.3 <= 1 - nd / ids.size <= 0.5  # ~40% of the picks repeat
    print(name, figs)


def _small(seed, R=3, H=512, E=12, k=3, I=256, Is=192, kind="plain"):
    shape = gen.TailShape(R, H, E, k, I, Is)
    d = gen.make_weights(shape, seed)
    d.update(gen.make_activations(shape, seed, kind, c=0.8))
    return shape, d


SIMPLE = 1  # debug flag: warp-per-row CUDA-core expert kernels instead of the streaming ones
NO_PDL = 2  # debug flag: plain stream-ordered launches (no programmatic dependent launch)
STALL = 4   # debug flag: one producer leaves a stage unpublished (failure injection)
FUSED_FRONT = 8  # debug flag: the single-launch front
STATUS_TIMEOUT = 4  # device status bit: a bounded wait expired


def _check_small(shape, d, max_rows=None, rows=None, flags=0):
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    orc = oracle.moe_tail(d, shape.k, shape.eps, nthreads=NTHREADS)
    tail = MoeTail(shape, dev, max_rows=max_rows or shape.R, debug_flags=flags)
    out, res, ids, wts, nd = run_gpu(tail, d, rows)
    check_parity(out, res, ids, orc, shape.k)
    assert tail.status() == 0
    return tail, dev, orc, (out, res, ids, wts, nd)


@pytest.mark.parametrize("flags", [0, SIMPLE, NO_PDL, FUSED_FRONT])
@pytest.mark.parametrize("R,H,E,k,I,Is", [
    (1, 256, 1, 1, 128, 64),       # a single expert, smallest shapes
    (2, 512, 12, 3, 256, 192),     # several tiles, ragged tails
    (5, 768, 33, 7, 384, 320),     # odd expert count, k not a power of two
    (3, 2560, 6, 2, 2560, 192),    # several E8M0 windows per row (CUDA-core form), the last ragged
    (16, 3072, 2, 2, 128, 64),     # 16 users of each expert (two N-tiles), long K
    (16, 256, 16, 16, 128, 128),   # k = E: every expert, maximum rows
    (16, 512, 64, 1, 256, 64),     # k = 1, maximum rows
    (4, 1024, 40, 32, 128, 256),   # k at its maximum
    (4, 256, 1024, 8, 128, 64),    # the maximum expert count
])
def test_small_shapes(R, H, E, k, I, Is, flags):
    shape, d = _small(100 + R + E, R, H, E, k, I, Is)
    _check_small(shape, d, flags=flags)


@pytest.mark.parametrize("flags", [0, SIMPLE])
def test_repeated_experts_and_dedup_count(flags):
    shape, d = _small(7, R=8, H=512, E=16, k=4, I=256, Is=128, kind="similar")
    _, _, orc, (_, _, ids, _, nd) = _check_small(shape, d, flags=flags)
    assert nd == len(np.unique(orc["ids"])) < shape.R * shape.k


@pytest.mark.parametrize("shift", [12, -16])
def test_mid_outside_f16_range_takes_block_scales(shift):
    """SiLU*up values far above (gate/up E8M0 scales x 2^12) or below (x 2^-16) the f16 range
    make the gate/up epilogue store mid with per-block powers of two, and the down launch
    apply them; the result still matches the oracle."""
    shape, d = _small(15, R=4, H=512, E=10, k=3, I=256, Is=128)
    d["w13_scales"] = (d["w13_scales"].astype(np.int32) + shift).astype(np.uint8)
    _check_small(shape, d)


@pytest.mark.parametrize("mode", [0, MODE_PERSISTENT_ID])
def test_refresh_scales_follows_in_place_scale_changes(mode):
    """The tensor-core forms read the routed experts' E8M0 scales from a copy the handle makes
    at create (scale-factor atoms).  After the caller rewrites w13_scales and w2_scales in
    place, moe_tail_refresh_scales makes the next run follow the new scales: checked against
    the oracle on the changed weights, with I = 384 (a half stage at the end of every down
    item), in the multi-kernel form and the persistent launch."""
    shape, d = _small(23, R=5, H=768, E=9, k=3, I=384, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    orc = oracle.moe_tail(d, shape.k, shape.eps, nthreads=NTHREADS)
    tail = MoeTail(shape, dev, mode=mode)
    out, res, ids, _, _ = run_gpu(tail, d)
    check_parity(out, res, ids, orc, shape.k)
    rng = np.random.default_rng(231)
    d2 = dict(d)
    for key in ("w13_scales", "w2_scales"):
        step = rng.integers(-1, 2, size=d[key].shape)
        d2[key] = (d[key].astype(np.int32) + step).astype(np.uint8)
        dev[key].copy_(torch.from_numpy(d2[key]))  # same device buffer, new values
    tail.refresh_scales()
    orc2 = oracle.moe_tail(d2, shape.k, shape.eps, nthreads=NTHREADS)
    out, res, ids, _, _ = run_gpu(tail, d2)
    check_parity(out, res, ids, orc2, shape.k)
    assert tail.status() == 0
    tail.close()


def test_identical_experts_output_independent_of_routing():
    shape, d = _small(8, R=4, E=6, k=2)
    for key in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        d[key] = np.repeat(d[key][:1], shape.E, axis=0)
    _check_small(shape, d)


def test_exact_router_tie_picks_lowest_id():
    shape, d = _small(9, R=2, H=256, E=10, k=3, I=128, Is=64)
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    l = oracle.router(n, d["w_r"])[0]
    order = sorted(range(shape.E), key=lambda e: (-np.float32(l[e]), e))
    a, b = order[shape.k - 1], order[shape.k]  # rank k-1 (picked) and rank k (not picked)
    lo, hi = min(a, b), max(a, b)
    d["w_r"][hi] = d["w_r"][lo]  # bitwise-identical rows straddling the cut
    tail, dev, orc, (out, res, ids, wts, nd) = _check_small(shape, d)
    assert lo in ids[0] and hi not in ids[0]
    assert lo in orc["ids"][0] and hi not in orc["ids"][0]


def test_nan_router_logits_flag_routing():
    # experts 2..9 get NaN router rows: each row picks the two finite experts by value, then
    # the lowest NaN id, and the status word records the bad routing
    shape, d = _small(16, R=2, H=256, E=10, k=3, I=128, Is=64)
    d["w_r"][2:] = 0x7FC0  # bf16 quiet NaN
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    l = oracle.router(n, d["w_r"])
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=shape.R)
    _, _, ids, _, nd = run_gpu(tail, d)
    for r in range(shape.R):
        assert sorted(ids[r][:2]) == [0, 1] and ids[r][2] == 2, (r, ids[r])
        if abs(l[r, 0] - l[r, 1]) > 1e-3:
            assert ids[r][0] == (0 if l[r, 0] > l[r, 1] else 1), (r, ids[r], l[r, :2])
    assert nd == 3
    assert tail.status() & STATUS_BAD_ROUTING
    tail.clear_status()
    assert tail.status() == 0


@pytest.mark.parametrize("flags", [0, SIMPLE, NO_PDL])
@pytest.mark.parametrize("R,H,E,k,I,Is", [
    (3, 512, 12, 3, 256, 192),     # several tiles
    (8, 2560, 20, 4, 512, 256),    # long K, repeated experts
    (16, 256, 16, 16, 128, 128),   # maximum rows, every expert
])
def test_shared_expert_gate(R, H, E, k, I, Is, flags):
    shape, d = _small(200 + R + E, R, H, E, k, I, Is)
    d["ws_gate"] = gen.make_weight(shape, 200 + R + E, "ws_gate")
    tail, dev, orc, (out, res, ids, wts, nd) = _check_small(shape, d, flags=flags)
    # the gate moves the output: the ungated oracle does not match it
    plain = oracle.moe_tail({kk: v for kk, v in d.items() if kk != "ws_gate"}, shape.k, shape.eps,
                            nthreads=NTHREADS)
    assert not np.array_equal(orc["out"], plain["out"])


def test_shared_expert_gate_refused_with_fused_front():
    shape, d = _small(210)
    d["ws_gate"] = gen.make_weight(shape, 210, "ws_gate")
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    with pytest.raises(MoeTailError) as ei:
        MoeTail(shape, dev, max_rows=shape.R, debug_flags=FUSED_FRONT)
    assert ei.value.code == ERR_UNSUPPORTED


@pytest.mark.parametrize("flags", [0, SIMPLE, NO_PDL, FUSED_FRONT])
@pytest.mark.parametrize("R,H,E,k,I,Is,Ha", [
    (3, 512, 12, 3, 256, 192, 768),      # several K stages and output boxes
    (8, 2560, 20, 4, 512, 256, 4096),    # long K, repeated experts
    (16, 256, 16, 16, 128, 128, 64),     # one stage, maximum rows
    (4, 1024, 16, 4, 256, 128, 512),     # eight K parts per box
    (2, 768, 8, 2, 128, 128, 128),       # two K parts per box
])
def test_attention_out_proj(R, H, E, k, I, Is, Ha, flags):
    shape = gen.TailShape(R, H, E, k, I, Is, Ha=Ha)
    seed = 300 + R + E
    d = gen.make_weights(shape, seed, keys=gen._LAYER_WEIGHTS + ("w_o",))
    d.update(gen.make_activations(shape, seed))
    d["attn"] = gen.make_attention_output(shape, seed)
    orc = oracle.moe_tail(d, shape.k, shape.eps, nthreads=NTHREADS)
    dev = weights_to_device({kk: v for kk, v in d.items() if kk not in ("x", "residual", "attn")})
    tail = MoeTail(shape, dev, max_rows=R, debug_flags=flags)
    attn = acts_to_device(d["attn"])
    res = acts_to_device(d["residual"])
    out = torch.empty_like(res)
    tail.run_attn(attn, res, out)
    torch.cuda.synchronize()
    ids, wts, nd = tail.routing(R)
    # x = bf16(attn . W_o^T) sums in fp32 here and in fp64 in the oracle: an element may round
    # to the neighbouring bf16 value, and r_new = bf16(x + residual) with it
    x_orc = oracle.out_proj(d["attn"], d["w_o"])
    tol = bf16_step(x_orc) + bf16_step(orc["residual"])
    figs = check_parity(bf16_tensor_to_bits(out), bf16_tensor_to_bits(res), ids, orc, shape.k,
                        residual_tol=tol)
    assert tail.status() == 0
    # the same handle still runs the plain call (x given directly)
    plain = oracle.moe_tail({kk: v for kk, v in d.items() if kk not in ("attn", "w_o")}, shape.k,
                            shape.eps, nthreads=NTHREADS)
    got = run_gpu(tail, d)
    check_parity(got[0], got[1], got[2], plain, shape.k)


def test_run_attn_needs_attn_dim():
    shape, d = _small(310)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=shape.R)
    x = acts_to_device(d["x"])
    with pytest.raises(MoeTailError) as ei:
        tail.run_attn(x, x.clone(), torch.empty_like(x))
    assert ei.value.code == ERR_UNSUPPORTED


def test_rows_below_max_and_batch_invariance():
    shape, d = _small(10, R=6, H=512, E=20, k=4, I=256, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=16)
    full = run_gpu(tail, d)
    for r in range(shape.R):
        one = run_gpu(tail, {"x": d["x"][r:r + 1], "residual": d["residual"][r:r + 1]})
        assert np.array_equal(one[0][0], full[0][r]), "row %d differs alone vs batched" % r
        assert np.array_equal(one[1][0], full[1][r])
    sub = run_gpu(tail, {"x": d["x"][2:5], "residual": d["residual"][2:5]})
    assert np.array_equal(sub[0], full[0][2:5])


def test_batch_invariance_above_eight_rows():
    """Twelve rows in one call equal each row alone and a 9-row subset, bit for bit: the
    router's split over its warps, the expert stages' columns and the combine are the same
    whatever the call's row count."""
    shape, d = _small(18, R=12, H=512, E=20, k=4, I=256, Is=128, kind="similar")
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=16)
    full = run_gpu(tail, d)
    for r in (0, 5, 11):
        one = run_gpu(tail, {"x": d["x"][r:r + 1], "residual": d["residual"][r:r + 1]})
        assert np.array_equal(one[0][0], full[0][r]), "row %d differs alone vs batched" % r
        assert np.array_equal(one[1][0], full[1][r])
    sub = run_gpu(tail, {"x": d["x"][1:10], "residual": d["residual"][1:10]})
    assert np.array_equal(sub[0], full[0][1:10])
    assert np.array_equal(sub[1], full[1][1:10])


def test_determinism_and_graph_replay():
    shape, d = _small(11, R=4, H=512, E=24, k=4, I=256, Is=192)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev)
    x = acts_to_device(d["x"])
    res0 = acts_to_device(d["residual"])
    eager_outs = []
    for _ in range(2):
        res = res0.clone()
        out = torch.empty_like(x)
        tail.run(x, res, out)
        torch.cuda.synchronize()
        eager_outs.append((bf16_tensor_to_bits(out), bf16_tensor_to_bits(res)))
    assert all(np.array_equal(a, b) for a, b in zip(eager_outs[0], eager_outs[1]))
    # capture one call; each replay recomputes from a fresh copy of the residual
    res = res0.clone()
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tail.run(x, res, out, stream=s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res.copy_(res0)
        tail.run(x, res, out)
    for i in range(1000):
        g.replay()
        if i % 250 == 249:
            torch.cuda.synchronize()
            assert np.array_equal(bf16_tensor_to_bits(out), eager_outs[0][0])
            assert np.array_equal(bf16_tensor_to_bits(res), eager_outs[0][1])
    assert tail.status() == 0


def test_run_host_matches_device_run():
    shape, d = _small(12, R=3)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev)
    out_d, res_d, *_ = run_gpu(tail, d)
    x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    res = torch.from_numpy(d["residual"].view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    out = torch.empty_like(x).pin_memory()
    tail.run_host(x, res, out)
    assert np.array_equal(bf16_tensor_to_bits(out), out_d)
    assert np.array_equal(bf16_tensor_to_bits(res), res_d)
    # pageable buffers: in place where the device uses the host's page tables, else copied
    x2 = torch.from_numpy(d["x"].view(np.int16).copy()).view(torch.bfloat16)
    res2 = torch.from_numpy(d["residual"].view(np.int16).copy()).view(torch.bfloat16)
    out2 = torch.empty_like(x2)
    assert not x2.is_pinned()
    tail.run_host(x2, res2, out2)
    assert np.array_equal(bf16_tensor_to_bits(out2), out_d)
    assert np.array_equal(bf16_tensor_to_bits(res2), res_d)


def test_run_host_page_locked_buffers_match_device_runs():
    """Page-locked host buffers, read and written in place by the call's kernels, on a
    non-default stream, over calls of two row counts (a block [x; residual; out] per call):
    every call matches the device-buffer run bit for bit."""
    shape, d = _small(14, R=4, H=512, E=12, k=3, I=256, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=4)
    stream = torch.cuda.Stream()
    H = shape.H
    for rows, seed in ((4, 1), (4, 2), (2, 3), (4, 4), (2, 5)):
        a = gen.make_activations(shape, 500 + seed, "plain", rows=rows)
        dd = dict(d)
        dd["x"], dd["residual"] = a["x"], a["residual"]
        out_d, res_d, *_ = run_gpu(tail, dd, rows)
        blk = torch.empty((3, rows, H), dtype=torch.bfloat16).pin_memory()
        blk[0].copy_(torch.from_numpy(a["x"].view(np.int16)).view(torch.bfloat16))
        blk[1].copy_(torch.from_numpy(a["residual"].view(np.int16)).view(torch.bfloat16))
        tail.run_host(blk[0], blk[1], blk[2], rows=rows, stream=stream)
        assert np.array_equal(bf16_tensor_to_bits(blk[2]), out_d), (rows, seed)
        assert np.array_equal(bf16_tensor_to_bits(blk[1]), res_d), (rows, seed)
    ids, _, _ = tail.routing(2)
    assert ids.shape == (2, shape.k)
    assert tail.status() == 0


@pytest.mark.parametrize("mode", [0, MODE_PERSISTENT_ID])
def test_run_host_returns_complete_results_back_to_back(mode):
    """Twenty host-buffer calls in a row on one page-locked block each (the call returns when
    the completion word its last kernel sets says so): every call's out and residual, read
    right after it returns, match the device-buffer run of the same inputs bit for bit."""
    shape, d = _small(19, R=3, H=512, E=12, k=3, I=256, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, mode=mode)
    stream = torch.cuda.Stream()
    H = shape.H
    for seed in range(20):
        a = gen.make_activations(shape, 900 + seed, "plain")
        dd = dict(d)
        dd["x"], dd["residual"] = a["x"], a["residual"]
        out_d, res_d, *_ = run_gpu(tail, dd)
        blk = torch.empty((3, shape.R, H), dtype=torch.bfloat16).pin_memory()
        blk[0].copy_(torch.from_numpy(a["x"].view(np.int16)).view(torch.bfloat16))
        blk[1].copy_(torch.from_numpy(a["residual"].view(np.int16)).view(torch.bfloat16))
        blk[2].fill_(0)
        tail.run_host(blk[0], blk[1], blk[2], stream=stream)
        assert np.array_equal(bf16_tensor_to_bits(blk[2]), out_d), seed
        assert np.array_equal(bf16_tensor_to_bits(blk[1]), res_d), seed
    assert tail.status() == 0


def test_run_rejects_bad_arguments():
    shape, d = _small(13, R=2)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=2)
    x = acts_to_device(d["x"])
    res = acts_to_device(d["residual"])
    out = torch.empty_like(x)
    for rows in (0, 3, -1):
        with pytest.raises(MoeTailError) as ei:
            tail.run(x, res, out, rows=rows)
        assert ei.value.code == ERR_INVALID_ARG
    big = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")
    mis = big[1:1 + x.numel()].view(x.shape)  # 2-byte offset: misaligned
    with pytest.raises(MoeTailError) as ei:
        tail.run(mis, res, out)
    assert ei.value.code == ERR_INVALID_ARG
    # unsupported shapes are refused at creation
    for bad in (gen.TailShape(2, 200, 12, 3, 256, 192), gen.TailShape(2, 512, 12, 13, 256, 192),
                gen.TailShape(2, 512, 12, 3, 100, 192), gen.TailShape(2, 2304, 12, 3, 256, 192)):
        with pytest.raises(MoeTailError) as ei:
            MoeTail(bad, dev)
        assert ei.value.code == ERR_UNSUPPORTED
    assert tail.status() == 0


def test_device_wait_timeout_is_reported_and_context_survives():
    """Failure detection without a fault: a stage that is never published makes the
    consumers' bounded wait (5 ms here) expire; the kernel records the timeout in the
    status word and returns, and the next call on a healthy handle is correct."""
    shape, d = _small(14, R=2, H=512, E=8, k=2, I=256, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    bad = MoeTail(shape, dev, wait_budget_us=5000, debug_flags=STALL)
    x = acts_to_device(d["x"])
    res = acts_to_device(d["residual"])
    out = torch.empty_like(x)
    bad.run(x, res, out)
    torch.cuda.synchronize()
    st = bad.status()
    assert st & STATUS_TIMEOUT, st
    bad.clear_status()
    assert bad.status() == 0
    bad.close()
    _check_small(shape, d)  # the context is healthy: a normal handle matches the oracle


# ------------------------------------------------------------ single persistent launch ----

from moe_layer_tail_gb300 import MODE_PERSISTENT  # noqa: E402


@pytest.mark.parametrize("name", list(gen.WORKLOADS))
def test_persistent_mode_parity_full_size(name):
    wl, d, dev, orc = workload_inputs(name)
    tail = MoeTail(wl.shape, dev, max_rows=wl.shape.R, mode=MODE_PERSISTENT)
    assert tail.launches_per_run(wl.shape.R) == 1
    got = run_gpu(tail, d)
    check_parity(got[0], got[1], got[2], orc, wl.shape.k)
    assert tail.status() == 0


@pytest.mark.parametrize("R,H,E,k,I,Is,gated", [
    (1, 256, 8, 2, 128, 128, False),
    (5, 768, 20, 4, 384, 192, True),    # ragged rows, shared-expert gate
    (16, 512, 12, 3, 256, 64, False),   # maximum rows, repeated experts
    (3, 512, 4, 4, 256, 192, True),     # k = E
    (32, 1024, 40, 6, 384, 128, True),  # 32 rows (128 plane columns), half last down stage
])
def test_persistent_mode_small_shapes(R, H, E, k, I, Is, gated):
    shape = gen.TailShape(R, H, E, k, I, Is)
    seed = 500 + R + E
    keys = gen._LAYER_WEIGHTS + (("ws_gate",) if gated else ())
    d = gen.make_weights(shape, seed, keys=keys)
    d.update(gen.make_activations(shape, seed))
    orc = oracle.moe_tail(d, k, shape.eps, nthreads=NTHREADS)
    dev = weights_to_device({kk: v for kk, v in d.items() if kk not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=R, mode=MODE_PERSISTENT)
    got = run_gpu(tail, d)
    check_parity(got[0], got[1], got[2], orc, k)
    # fewer rows on the same handle
    if R > 1:
        d2 = dict(d)
        d2["x"], d2["residual"] = d["x"][:R - 1], d["residual"][:R - 1]
        orc2 = oracle.moe_tail(d2, k, shape.eps, nthreads=NTHREADS)
        got2 = run_gpu(tail, d2)
        check_parity(got2[0], got2[1], got2[2], orc2, k)
    assert tail.status() == 0


def test_persistent_mode_determinism_and_graph_replay():
    shape, d = _small(13, R=4, H=512, E=24, k=4, I=256, Is=192)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, mode=MODE_PERSISTENT)
    x = acts_to_device(d["x"])
    res0 = acts_to_device(d["residual"])
    eager = []
    for _ in range(3):
        res = res0.clone()
        out = torch.empty_like(x)
        tail.run(x, res, out)
        torch.cuda.synchronize()
        eager.append((bf16_tensor_to_bits(out), bf16_tensor_to_bits(res)))
    assert all(np.array_equal(a, b) for a, b in zip(eager[0], eager[1]))
    assert all(np.array_equal(a, b) for a, b in zip(eager[0], eager[2]))
    res = res0.clone()
    out = torch.empty_like(x)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res.copy_(res0)
        tail.run(x, res, out)
    for i in range(100):
        g.replay()
        if i % 25 == 24:
            torch.cuda.synchronize()
            assert np.array_equal(bf16_tensor_to_bits(out), eager[0][0])
            assert np.array_equal(bf16_tensor_to_bits(res), eager[0][1])
    assert tail.status() == 0


def test_persistent_mode_refuses_out_proj():
    shape = gen.TailShape(2, 256, 8, 2, 128, 128, Ha=128)
    d = gen.make_weights(shape, 7, keys=gen._LAYER_WEIGHTS + ("w_o",))
    dev = weights_to_device(d)
    with pytest.raises(MoeTailError) as e:
        MoeTail(shape, dev, max_rows=2, mode=MODE_PERSISTENT)
    assert e.value.code == ERR_UNSUPPORTED


def test_persistent_mode_barrier_timeout_is_reported_and_reset():
    """A CTA that never arrives at the grid barrier makes the others' bounded waits (5 ms)
    expire: the status reports the timeout, the call completes, clear_status resets the
    barrier, the same stalled handle times out again the same way (no hang), and a healthy
    persistent handle is correct afterwards."""
    shape, d = _small(15, R=2, H=512, E=8, k=2, I=256, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    bad = MoeTail(shape, dev, mode=MODE_PERSISTENT, wait_budget_us=5000, debug_flags=STALL)
    x = acts_to_device(d["x"])
    for _ in range(2):
        res = acts_to_device(d["residual"])
        out = torch.empty_like(x)
        bad.run(x, res, out)
        torch.cuda.synchronize()
        assert bad.status() & STATUS_TIMEOUT
        bad.clear_status()
        assert bad.status() == 0
    bad.close()
    good = MoeTail(shape, dev, mode=MODE_PERSISTENT)
    orc = oracle.moe_tail(d, shape.k, shape.eps, nthreads=NTHREADS)
    got = run_gpu(good, d)
    check_parity(got[0], got[1], got[2], orc, shape.k)
    assert good.status() == 0


def test_graph_of_mixed_widths_replays_bitwise():
    """Six calls of widths 8, 1, 3, 8, 2, 5 captured in one CUDA graph (each on its own
    buffers) replay bitwise equal to the same calls run eagerly."""
    shape, d = _small(16, R=8, H=512, E=24, k=4, I=256, Is=192)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=8)
    widths = [8, 1, 3, 8, 2, 5]
    xs = [acts_to_device(gen.make_activations(shape, 700 + i, rows=w)["x"])
          for i, w in enumerate(widths)]
    r0 = [acts_to_device(gen.make_activations(shape, 700 + i, rows=w)["residual"])
          for i, w in enumerate(widths)]
    eager = []
    for x, r in zip(xs, r0):
        res, out = r.clone(), torch.empty_like(x)
        tail.run(x, res, out)
        torch.cuda.synchronize()
        eager.append((bf16_tensor_to_bits(out), bf16_tensor_to_bits(res)))
    res = [r.clone() for r in r0]
    outs = [torch.empty_like(x) for x in xs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for x, rr, r, o in zip(xs, r0, res, outs):
            r.copy_(rr)
            tail.run(x, r, o)
    for i in range(200):
        g.replay()
        if i % 100 == 99:
            torch.cuda.synchronize()
            for (eo, er), o, r in zip(eager, outs, res):
                assert np.array_equal(bf16_tensor_to_bits(o), eo)
                assert np.array_equal(bf16_tensor_to_bits(r), er)
    assert tail.status() == 0


def test_back_to_back_mixed_widths_match_one_at_a_time():
    """Calls of widths 8, 1, 5, 8, 2, 8, 3 issued back to back on one stream (each launch
    may start while the previous one still runs) equal the same calls run one at a time."""
    shape, d = _small(17, R=8, H=512, E=24, k=4, I=256, Is=192, kind="similar")
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=8)
    widths = [8, 1, 5, 8, 2, 8, 3]
    acts = [gen.make_activations(shape, 800 + i, rows=w) for i, w in enumerate(widths)]
    xs = [acts_to_device(a["x"]) for a in acts]
    r0 = [acts_to_device(a["residual"]) for a in acts]
    single = []
    for x, r in zip(xs, r0):
        res, out = r.clone(), torch.empty_like(x)
        tail.run(x, res, out)
        torch.cuda.synchronize()
        single.append((bf16_tensor_to_bits(out), bf16_tensor_to_bits(res)))
    for _ in range(3):
        res = [r.clone() for r in r0]
        outs = [torch.empty_like(x) for x in xs]
        torch.cuda.synchronize()
        for x, r, o in zip(xs, res, outs):
            tail.run(x, r, o)
        torch.cuda.synchronize()
        for (so, sr), o, r in zip(single, outs, res):
            assert np.array_equal(bf16_tensor_to_bits(o), so)
            assert np.array_equal(bf16_tensor_to_bits(r), sr)
    assert tail.status() == 0
