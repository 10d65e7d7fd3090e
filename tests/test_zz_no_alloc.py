"""moe_tail_route_noalloc: routing for callers that cannot allocate device memory (a host
framework that owns every allocation and passes a plugin only its tensors, or a decode
step run from a memory pool frozen after warm-up).  Its scratch is a fixed array
inside the library, so this file runs last: if it fails, every other test has already run.

The entry point is checked against the CPU oracle with the parity rule of the other tests
(identical selection wherever the oracle's fp32 k-th/(k+1)-th margin exceeds 1e-3, routing
weights within 5e-4, the distinct count of the oracle's picks), and against the routing of
the allocating entry point (moe_tail_run) under the same rule, on two calls in a row."""
import ctypes

import numpy as np
import pytest

import moe_layer_tail_gb300 as mt
import oracle
from moe_layer_tail_gb300 import inputs as gen
from parity import MARGIN, fp32_margins

P = ctypes.c_void_p
I32 = ctypes.c_int32
WTS_TOL = 5e-4


def _lib():
    lib = mt.load_library()
    f = lib.moe_tail_route_noalloc
    f.argtypes = [P, P, P, P, I32, I32, I32, I32, ctypes.c_float, P, P, P, P, P]
    f.restype = ctypes.c_int
    return lib


def test_sizes_beyond_the_fixed_scratch_are_refused():
    lib = _lib()
    fake = P(256)  # never dereferenced: the size check comes first
    for rows, e, k in ((17, 8, 2), (4, 1025, 2), (4, 64, 33), (0, 8, 2)):
        rc = lib.moe_tail_route_noalloc(fake, fake, fake, fake, rows, 256, e, k, 1e-6, fake,
                                        fake, None, None, None)
        assert rc == mt.ERR_UNSUPPORTED, (rows, e, k, rc)


def _same_rule(ids_a, ids_b, margins):
    """Selections agree wherever the margin exceeds the near-tie threshold."""
    for r in range(ids_a.shape[0]):
        if margins[r] > MARGIN:
            assert set(ids_a[r].tolist()) == set(ids_b[r].tolist()), (r, ids_a[r], ids_b[r])


def _route(lib, torch, x, res, dev, R, H, E, k, eps):
    """One call of the entry point on caller-owned buffers; returns ids, wts, nd, status."""
    ids = torch.full((R, k), -1, dtype=torch.int32, device="cuda")
    wts = torch.zeros((R, k), dtype=torch.float32, device="cuda")
    nd = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.moe_tail_route_noalloc(
        P(x.data_ptr()), P(res.data_ptr()), P(dev["gamma"].data_ptr()), P(dev["w_r"].data_ptr()),
        R, H, E, k, float(eps), P(ids.data_ptr()), P(wts.data_ptr()), P(nd.data_ptr()),
        P(st.data_ptr()), P(stream))
    assert rc == mt.OK, rc
    torch.cuda.synchronize()
    return ids.cpu().numpy(), wts.cpu().numpy(), int(nd.item()), int(st.item())


@pytest.mark.gpu
@pytest.mark.parametrize("seed,R,H,E,k", [
    (31, 5, 512, 24, 4),      # E <= 256: the sorted-candidate top-k
    (32, 16, 768, 40, 6),     # maximum rows
    (33, 4, 1024, 512, 10),   # 256 < E <= 512
    (34, 3, 512, 1024, 32),   # the largest E and k the array holds
])
def test_route_noalloc_matches_oracle_and_run_on_two_calls(seed, R, H, E, k):
    torch = pytest.importorskip("torch")
    lib = _lib()
    shape = gen.TailShape(R, H, E, k, 256, 128)
    d = gen.make_weights(shape, seed)
    d.update(gen.make_activations(shape, seed, "similar", c=0.7))
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    logits = oracle.router(n, d["w_r"])
    ids_o, wts_o = oracle.topk(logits, k)
    margins = fp32_margins(logits, k)
    assert np.mean(margins > MARGIN) > 0.5  # the rule compares most rows
    dev = mt.weights_to_device(d)
    x = mt.acts_to_device(d["x"])
    res = mt.acts_to_device(d["residual"])
    # the existing entry point (allocating handle) and its routing
    tail = mt.MoeTail(shape, {k2: v for k2, v in dev.items() if k2 not in ("x", "residual")})
    out = torch.empty_like(x)
    tail.run(x, res.clone(), out)
    torch.cuda.synchronize()
    ids_run, wts_run, nd_run = tail.routing(R)
    tail.close()
    for call in range(2):  # two calls in a row share (and must clear) the fixed array
        ids, wts, nd, st = _route(lib, torch, x, res, dev, R, H, E, k, shape.eps)
        assert st == 0, (call, st)
        _same_rule(ids, ids_o, margins)
        _same_rule(ids, ids_run, margins)
        for r in range(R):
            if margins[r] > MARGIN:
                # weights in pick order: compare by expert id
                got = dict(zip(ids[r].tolist(), wts[r].tolist()))
                ref = dict(zip(ids_o[r].tolist(), wts_o[r].tolist()))
                run = dict(zip(ids_run[r].tolist(), wts_run[r].tolist()))
                assert max(abs(got[e] - ref[e]) for e in ref) < WTS_TOL, (call, r)
                assert max(abs(got[e] - run[e]) for e in run) < WTS_TOL, (call, r)
                assert abs(sum(got.values()) - 1.0) < 1e-5
        if (margins > MARGIN).all():
            assert nd == len(np.unique(ids_o)) == nd_run, (call, nd, nd_run)


@pytest.mark.gpu
def test_route_noalloc_reports_nan_routing_and_clears_it_next_call():
    torch = pytest.importorskip("torch")
    lib = _lib()
    R, H, E, k = 2, 256, 10, 3
    shape = gen.TailShape(R, H, E, k, 128, 64)
    d = gen.make_weights(shape, 41)
    d.update(gen.make_activations(shape, 41))
    clean = mt.weights_to_device(d)
    bad_w = dict(d)
    bad_w["w_r"] = d["w_r"].copy()
    bad_w["w_r"][2:] = 0x7FC0  # bf16 quiet NaN: only experts 0 and 1 have numeric logits
    bad = mt.weights_to_device(bad_w)
    x = mt.acts_to_device(d["x"])
    res = mt.acts_to_device(d["residual"])
    ids, wts, nd, st = _route(lib, torch, x, res, bad, R, H, E, k, shape.eps)
    assert st & mt.STATUS_BAD_ROUTING, st
    for r in range(R):
        # the two numeric experts by value, then the lowest untaken id
        assert sorted(ids[r][:2].tolist()) == [0, 1] and ids[r][2] == 2, (r, ids[r])
    assert nd == 3
    # the next call with numeric weights reports a clean status (the word is per call)
    ids, wts, nd, st = _route(lib, torch, x, res, clean, R, H, E, k, shape.eps)
    assert st == 0, st
    _, n, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["gamma"], shape.eps)
    logits = oracle.router(n, d["w_r"])
    ids_o, _ = oracle.topk(logits, k)
    _same_rule(ids, ids_o, fp32_margins(logits, k))
