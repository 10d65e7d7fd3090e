"""The two streaming forms of the expert stages side by side: the default tensor-core form
(tcgen05 block-scaled E2M1 x E2M1 MMAs for the routed MXFP4 experts, bf16 MMAs for the shared
expert) and the CUDA-core form (MOE_TAIL_DEBUG_MMA_SYNC: E2M1 -> f16 conversion into
mma.sync), each against the oracle element by element through the C ABI under the same
parity rule: every workload at full size, small shapes with ragged tails and the edge cases,
graph replay, the launch modes and the bounded-wait failure path."""
import numpy as np
import pytest

import oracle
from moe_layer_tail_gb300 import MoeTail, acts_to_device, bf16_tensor_to_bits, weights_to_device
from moe_layer_tail_gb300 import inputs as gen
from parity import check_parity
from test_gpu_parity import NTHREADS, _small, run_gpu, workload_inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TC = 0       # the default (tcgen05) expert stages
MMA_SYNC = 16  # debug flag: the CUDA-core mma.sync streaming kernels
NO_PDL = 2   # plain stream-ordered launches
STALL = 4    # failure injection: one producer leaves a stage unpublished
STATUS_TIMEOUT = 4


def _check(shape, d, flags=TC, rows=None, max_rows=None):
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    orc = oracle.moe_tail(d, shape.k, shape.eps, nthreads=NTHREADS)
    tail = MoeTail(shape, dev, max_rows=max_rows or shape.R, debug_flags=flags)
    out, res, ids, wts, nd = run_gpu(tail, d, rows)
    figs = check_parity(out, res, ids, orc, shape.k, rows=rows)
    assert tail.status() == 0
    return tail, dev, orc, figs, (out, res, ids, wts, nd)


def test_tiny_first():
    # the smallest case first: one row, two experts, K of 128 in the down contraction
    wl = gen.WORKLOADS["tiny"]
    d = gen.make_inputs(wl)
    _check(wl.shape, d)


@pytest.mark.parametrize("flags", [TC, MMA_SYNC])
@pytest.mark.parametrize("name", list(gen.WORKLOADS))
def test_workload_parity_full_size(name, flags):
    if flags == MMA_SYNC and gen.WORKLOADS[name].shape.R > 16:
        pytest.skip("the CUDA-core form takes 16 rows at most (refused at create)")
    wl, d, dev, orc = workload_inputs(name)
    tail = MoeTail(wl.shape, dev, max_rows=wl.shape.R, debug_flags=flags)
    out, res, ids, wts, nd = run_gpu(tail, d)
    figs = check_parity(out, res, ids, orc, wl.shape.k)
    assert nd == len(np.unique(orc["ids"]))
    assert tail.status() == 0
    print(name, figs)


@pytest.mark.parametrize("flags", [TC, TC | NO_PDL, MMA_SYNC])
@pytest.mark.parametrize("R,H,E,k,I,Is", [
    (1, 256, 1, 1, 128, 64),       # a single expert, smallest shapes
    (2, 512, 12, 3, 256, 192),     # several tiles, ragged tails
    (5, 768, 33, 7, 384, 320),     # odd expert count; the down K ends half-way in a stage
    (3, 2560, 6, 2, 2560, 192),    # several E8M0 windows per row, the last one ragged
    (16, 3072, 2, 2, 128, 64),     # 16 users of each expert (64 plane columns), long K
    (16, 256, 16, 16, 128, 128),   # k = E: every expert, maximum rows
    (16, 512, 64, 1, 256, 64),     # k = 1, maximum rows
    (4, 1024, 40, 32, 128, 256),   # k at its maximum
    (4, 256, 1024, 8, 128, 64),    # the maximum expert count
    (8, 512, 16, 4, 256, 128),     # eight rows: 32 plane columns
])
def test_small_shapes(R, H, E, k, I, Is, flags):
    shape, d = _small(100 + R + E, R, H, E, k, I, Is)
    _check(shape, d, flags=flags)


@pytest.mark.parametrize("R,H,E,k,I,Is", [
    (17, 512, 24, 4, 256, 192),    # just past 16 rows: 128 plane columns, one accumulator slot
    (24, 768, 40, 6, 384, 320),    # ragged down K, several users per expert
    (32, 256, 32, 32, 128, 128),   # every row picks every expert: 32 users (128 plane rows)
    (32, 2560, 8, 3, 2560, 128),   # several E8M0 windows per row, the last one ragged
    (32, 1024, 1024, 8, 128, 64),  # the maximum expert count
])
def test_more_than_16_rows(R, H, E, k, I, Is):
    shape, d = _small(300 + R + E, R, H, E, k, I, Is, kind="similar")
    tail, _, orc, figs, (_, _, ids, _, nd) = _check(shape, d)
    assert nd == len(np.unique(orc["ids"]))
    # fewer rows than the handle's
    r = R - 5
    _check(shape, {**d, "x": d["x"][:r], "residual": d["residual"][:r]}, rows=r, max_rows=R)


@pytest.mark.parametrize("flags", [TC, MMA_SYNC])
@pytest.mark.parametrize("shift", [12, -16])
def test_mid_far_from_unit_scale(shift, flags):
    """Gate/up weights scaled by 2^12 or 2^-16: the planes' own E8M0 scales follow mid."""
    shape, d = _small(15, R=4, H=512, E=10, k=3, I=256, Is=128)
    d["w13_scales"] = (d["w13_scales"].astype(np.int32) + shift).astype(np.uint8)
    _check(shape, d, flags=flags)


def test_fewer_rows_than_the_handle():
    shape, d = _small(21, R=6, H=1024, E=24, k=4, I=256, Is=128)
    _check(shape, d, max_rows=16, rows=6)


def test_the_two_forms_agree_closely():
    """Both forms pass the rule against the oracle; here also against each other."""
    shape, d = _small(22, R=8, H=2048, E=32, k=4, I=512, Is=256, kind="similar")
    _, _, _, _, (out_tc, res_tc, ids_tc, _, _) = _check(shape, d)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    ref = MoeTail(shape, dev, max_rows=shape.R, debug_flags=MMA_SYNC)
    out, res, ids, _, _ = run_gpu(ref, d)
    assert np.array_equal(res, res_tc) and np.array_equal(ids, ids_tc)
    a = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = (out_tc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(shape.R):
        cos = a[r] @ b[r] / (np.linalg.norm(a[r]) * np.linalg.norm(b[r]))
        assert cos > 0.99995, (r, cos)


def test_graph_replay_bitwise_equal_to_eager():
    shape, d = _small(23, R=8, H=1024, E=24, k=4, I=256, Is=128, kind="similar")
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    tail = MoeTail(shape, dev, max_rows=shape.R, debug_flags=TC)
    x = acts_to_device(d["x"])
    res0 = acts_to_device(d["residual"])
    res = res0.clone()
    out = torch.empty_like(x)
    tail.run(x, res, out)
    torch.cuda.synchronize()
    eager_out, eager_res = out.clone(), res.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    res.copy_(res0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tail.run(x, res, out, stream=s)
    for _ in range(200):
        res.copy_(res0)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager_out) and torch.equal(res, eager_res)
    assert tail.status() == 0


@pytest.mark.parametrize("flags", [TC, MMA_SYNC])
def test_device_wait_timeout_is_reported_and_context_survives(flags):
    shape, d = _small(24, R=2, H=512, E=8, k=2, I=256, Is=128)
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    bad = MoeTail(shape, dev, max_rows=shape.R, debug_flags=flags | STALL, wait_budget_us=20000)
    x = acts_to_device(d["x"])
    res = acts_to_device(d["residual"])
    out = torch.empty_like(x)
    bad.run(x, res, out)
    torch.cuda.synchronize()
    assert bad.status() & STATUS_TIMEOUT
    bad.close()
    # a healthy handle on the same device still matches the oracle
    _check(shape, d, flags=flags)


def test_timeline_milestones_in_order():
    """The tracing option: every milestone of a default-form call recorded, in causal order."""
    from moe_layer_tail_gb300 import DEBUG_TIMELINE
    shape, d = _small(25, R=8, H=1024, E=32, k=4, I=512, Is=256, kind="similar")
    tail, _, _, _, _ = _check(shape, d, flags=DEBUG_TIMELINE)
    t = tail.timeline()
    assert all(v is not None for v in t.values()), t
    assert t["norm_start"] == 0.0
    for a, b in [("norm_start", "norm_end"), ("router_start", "router_all_started"),
                 ("router_all_started", "topk_start"),
                 ("topk_start", "routed"), ("gate_up_start", "gate_up_first_copy"),
                 ("gate_up_first_copy", "gate_up_all_copying"),
                 ("gate_up_all_copying", "gate_up_end"),
                 ("routed", "gate_up_routed"), ("gate_up_routed", "gate_up_end"),
                 ("down_start", "down_first_copy"), ("down_first_copy", "down_end"),
                 ("combine_start", "combine_end"), ("down_end", "combine_end")]:
        assert t[a] <= t[b], (a, b, t)
    assert t["combine_end"] < 1e4  # microseconds: one call


def test_timeline_milestones_in_order_persistent():
    """The same milestones recorded by the single persistent launch, in causal order (its
    combine starts once a CTA has left its down roles)."""
    from moe_layer_tail_gb300 import DEBUG_TIMELINE, MODE_PERSISTENT
    shape, d = _small(26, R=8, H=1024, E=32, k=4, I=512, Is=256, kind="similar")
    dev = weights_to_device({k: v for k, v in d.items() if k not in ("x", "residual")})
    orc = oracle.moe_tail(d, shape.k, shape.eps, nthreads=NTHREADS)
    tail = MoeTail(shape, dev, mode=MODE_PERSISTENT, debug_flags=DEBUG_TIMELINE)
    x = acts_to_device(d["x"])
    res = acts_to_device(d["residual"])
    out = torch.empty_like(x)
    tail.run(x, res, out)
    torch.cuda.synchronize()
    ids, _, _ = tail.routing(shape.R)
    check_parity(bf16_tensor_to_bits(out), bf16_tensor_to_bits(res), ids, orc, shape.k)
    t = tail.timeline()
    assert all(v is not None for v in t.values()), t
    for a, b in [("norm_start", "norm_end"), ("norm_end", "router_start"),
                 ("router_start", "router_all_started"), ("router_all_started", "topk_start"),
                 ("topk_start", "routed"),
                 ("gate_up_start", "gate_up_first_copy"), ("routed", "gate_up_routed"),
                 ("gate_up_first_copy", "gate_up_all_copying"),
                 ("down_start", "down_first_copy"), ("down_first_copy", "down_end"),
                 ("combine_start", "combine_end"), ("down_end", "combine_end")]:
        assert t[a] <= t[b], (a, b, t)
    assert tail.status() == 0
