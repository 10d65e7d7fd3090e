"""moe_tail_route_noalloc: routing for callers that cannot allocate device memory (a host
framework that owns every allocation and passes a plugin only its tensors, or a decode
step replayed from a frozen memory pool).  Its scratch is a fixed array inside the library,
so this file runs last: if it fails, every other test has already run."""
import ctypes

import numpy as np
import pytest

import moe_layer_tail_gb300 as mt
from moe_layer_tail_gb300 import inputs as gen

P = ctypes.c_void_p
I32 = ctypes.c_int32


def _lib():
    lib = mt.load_library()
    f = lib.moe_tail_route_noalloc
    f.argtypes = [P, P, P, P, I32, I32, I32, I32, ctypes.c_float, P, P, P, P]
    f.restype = ctypes.c_int
    return lib


def test_sizes_beyond_the_fixed_scratch_are_refused():
    lib = _lib()
    fake = P(256)  # never dereferenced: the size check comes first
    for rows, e, k in ((17, 8, 2), (4, 1025, 2), (4, 64, 33), (0, 8, 2)):
        rc = lib.moe_tail_route_noalloc(fake, fake, fake, fake, rows, 256, e, k, 1e-6, fake,
                                        fake, None, None)
        assert rc == mt.ERR_UNSUPPORTED, (rows, e, k, rc)


@pytest.mark.gpu
def test_route_noalloc_matches_run_routing_on_two_calls():
    torch = pytest.importorskip("torch")
    lib = _lib()
    for seed, (R, H, E, k) in ((31, (5, 512, 24, 4)), (32, (16, 768, 40, 6))):
        shape = gen.TailShape(R, H, E, k, 256, 128)
        d = gen.make_weights(shape, seed)
        d.update(gen.make_activations(shape, seed, "similar", c=0.7))
        dev = mt.weights_to_device(d)
        x = mt.acts_to_device(d["x"])
        res = mt.acts_to_device(d["residual"])
        # the existing entry point (allocating handle) and its routing
        tail = mt.MoeTail(shape, {k2: v for k2, v in dev.items() if k2 not in ("x", "residual")})
        out = torch.empty_like(x)
        tail.run(x, res.clone(), out)
        torch.cuda.synchronize()
        ids_ref, wts_ref, nd_ref = tail.routing(R)
        # the allocation-free entry point, on buffers the caller owns
        ids = torch.full((R, k), -1, dtype=torch.int32, device="cuda")
        wts = torch.zeros((R, k), dtype=torch.float32, device="cuda")
        nd = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.moe_tail_route_noalloc(
            P(x.data_ptr()), P(res.data_ptr()), P(dev["gamma"].data_ptr()),
            P(dev["w_r"].data_ptr()), R, H, E, k, float(shape.eps), P(ids.data_ptr()),
            P(wts.data_ptr()), P(nd.data_ptr()), P(stream))
        assert rc == mt.OK, rc
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        # the routing-weight tolerance of the parity tests
        assert np.max(np.abs(wts.cpu().numpy() - wts_ref)) < 5e-4
        assert int(nd.item()) == nd_ref
        tail.close()
