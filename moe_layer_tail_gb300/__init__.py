"""moe_layer_tail_gb300 -- Python binding of libmoe_tail.so (the decode-step MoE layer tail
on one GB300, sm_103a).

The binding marshals arguments only: every step of the tail runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  If the compiled library is missing
the binding raises: there is no CPU or PyTorch fallback.

    from moe_layer_tail_gb300 import MoeTail
    tail = MoeTail(shape, weights, max_rows=8)      # weights: dict of CUDA tensors
    tail.run(x, residual, out)                      # bf16 CUDA tensors [rows, H]
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_tail.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_TIMEOUT = -4
ERR_NOT_CORESIDENT = -5
ERR_DEVICE = -6

# bits of the device status word (moe_tail_get_status)
STATUS_BAD_ROUTING = 1
STATUS_BAD_DISTINCT = 2
STATUS_TIMEOUT = 4
STATUS_BAD_TILE = 8

MODE_MULTI_KERNEL = 0
MODE_PERSISTENT = 1

# debug_flags bits (moe_tail.h)
DEBUG_SIMPLE_KERNELS = 1
DEBUG_NO_PDL = 2
DEBUG_STALL_FIRST_STAGE = 4
DEBUG_FUSED_FRONT = 8
DEBUG_MMA_SYNC = 16
DEBUG_TIMELINE = 32

# timeline slots (moe_tail_debug_timeline)
TL_NAMES = ("norm_start", "norm_end", "router_start", "topk_start", "routed", "gate_up_start",
            "gate_up_first_copy", "gate_up_routed", "gate_up_end", "down_start",
            "down_first_copy", "down_end", "combine_start", "combine_end",
            "router_all_started", "gate_up_all_copying")

# moe_attnres_mix launch flags (attnres_mix.h)
ATTNRES_MIX_PDL = 1
ATTNRES_MIX_DEBUG_STALL = 2


class Config(ctypes.Structure):
    _fields_ = [("max_rows", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("expert_inter", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("norm_topk_prob", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("wait_budget_us", ctypes.c_uint32),
                ("debug_flags", ctypes.c_uint32), ("attn_dim", ctypes.c_int32)]


class WeightPtrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("gamma", "router_w", "w13_codes", "w13_scales", "w2_codes", "w2_scales",
                 "shared_w13", "shared_w2", "shared_gate", "out_proj")]


class MoeTailError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        lib = _lib_or_none()
        msg = lib.moe_tail_strerror(code).decode() if lib else str(code)
        if code == ERR_CUDA and lib:
            msg += " (" + lib.moe_tail_last_cuda_error().decode() + ")"
        super().__init__("%s: %s [%d]" % (what, msg, code))


_lib = None


def _lib_or_none():
    return _lib


def load_library(path: str = None):
    """Load libmoe_tail.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libmoe_tail.so is not built (%s); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.moe_tail_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(WeightPtrs),
                                    ctypes.POINTER(P)]
    lib.moe_tail_create.restype = ctypes.c_int
    lib.moe_tail_run.argtypes = [P, P, P, P, i32, P]
    lib.moe_tail_run.restype = ctypes.c_int
    lib.moe_tail_run_host.argtypes = [P, P, P, P, i32, P]
    lib.moe_tail_run_host.restype = ctypes.c_int
    lib.moe_tail_run_attn.argtypes = [P, P, P, P, i32, P]
    lib.moe_tail_run_attn.restype = ctypes.c_int
    lib.moe_tail_get_status.argtypes = [P, ctypes.POINTER(i32)]
    lib.moe_tail_get_status.restype = ctypes.c_int
    lib.moe_tail_check_scratch.argtypes = [P]
    lib.moe_tail_check_scratch.restype = ctypes.c_int
    lib.moe_tail_clear_status.argtypes = [P]
    lib.moe_tail_clear_status.restype = ctypes.c_int
    lib.moe_tail_debug_routing.argtypes = [P, P, P, ctypes.POINTER(i32), P]
    lib.moe_tail_debug_routing.restype = ctypes.c_int
    lib.moe_tail_set_stage_events.argtypes = [P, P, i32]
    lib.moe_tail_set_stage_events.restype = ctypes.c_int
    lib.moe_tail_launches_per_run.argtypes = [P, i32]
    lib.moe_tail_launches_per_run.restype = ctypes.c_int
    lib.moe_tail_debug_timeline.argtypes = [P, P, i32]
    lib.moe_tail_debug_timeline.restype = ctypes.c_int
    lib.moe_tail_refresh_scales.argtypes = [P, P]
    lib.moe_tail_refresh_scales.restype = ctypes.c_int
    lib.moe_tail_destroy.argtypes = [P]
    lib.moe_tail_destroy.restype = None
    lib.moe_tail_strerror.argtypes = [ctypes.c_int]
    lib.moe_tail_strerror.restype = ctypes.c_char_p
    lib.moe_tail_last_cuda_error.argtypes = []
    lib.moe_tail_last_cuda_error.restype = ctypes.c_char_p
    lib.moe_attnres_mix.argtypes = [i32, i32, i32, i32, ctypes.c_float] + [P] * 7 + \
        [ctypes.c_uint, P]
    lib.moe_attnres_mix.restype = ctypes.c_int
    lib.moe_attnres_mix_get_status.argtypes = [ctypes.POINTER(i32), i32]
    lib.moe_attnres_mix_get_status.restype = ctypes.c_int
    lib.moe_attnres_mix_ctas_per_row.argtypes = [i32, i32]
    lib.moe_attnres_mix_ctas_per_row.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(shape, max_rows=None, mode=MODE_MULTI_KERNEL, wait_budget_us=0,
                debug_flags=0) -> Config:
    return Config(max_rows=int(max_rows if max_rows is not None else shape.R),
                  hidden=shape.H, n_experts=shape.E, top_k=shape.k, expert_inter=shape.I,
                  shared_inter=shape.Is, rms_eps=float(shape.eps), norm_topk_prob=1,
                  mode=int(mode), wait_budget_us=int(wait_budget_us),
                  debug_flags=int(debug_flags), attn_dim=int(getattr(shape, "Ha", 0)))


_WEIGHT_KEYS = {"gamma": "gamma", "router_w": "w_r", "w13_codes": "w13_codes",
                "w13_scales": "w13_scales", "w2_codes": "w2_codes", "w2_scales": "w2_scales",
                "shared_w13": "ws13", "shared_w2": "ws2", "shared_gate": "ws_gate",
                "out_proj": "w_o"}
_OPTIONAL_WEIGHTS = ("ws_gate", "w_o")  # absent: a null pointer


class MoeTail:
    """One layer's tail: borrowed device weights plus the library handle and its scratch."""

    def __init__(self, shape, weights: dict, max_rows: int = None, mode=MODE_MULTI_KERNEL,
                 wait_budget_us=0, debug_flags=0):
        lib = load_library()
        self.shape = shape
        self._weights = weights  # keep the borrowed tensors alive
        self.cfg = make_config(shape, max_rows, mode, wait_budget_us, debug_flags)
        wp = WeightPtrs(**{f: (weights[k].data_ptr() if weights.get(k) is not None else None)
                           for f, k in _WEIGHT_KEYS.items()
                           if k in weights or k not in _OPTIONAL_WEIGHTS})
        h = ctypes.c_void_p()
        rc = lib.moe_tail_create(ctypes.byref(self.cfg), ctypes.byref(wp), ctypes.byref(h))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_create")
        self._h = h
        self._lib = lib

    @property
    def handle(self):
        return self._h

    def run(self, x, residual, out, rows: int = None, stream=None) -> None:
        """x, residual, out: bf16 CUDA tensors [>= rows, H]; residual is updated in place."""
        rows = int(x.shape[0] if rows is None else rows)
        rc = self._lib.moe_tail_run(self._h, _ptr(x), _ptr(residual), _ptr(out), rows,
                                    _stream_handle(stream))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_run")

    def run_attn(self, attn, residual, out, rows: int = None, stream=None) -> None:
        """The call with the attention output projection in front: attn bf16 [>= rows, Ha]
        (the handle's shape has Ha > 0 and its weights a "w_o" [H, Ha])."""
        rows = int(attn.shape[0] if rows is None else rows)
        rc = self._lib.moe_tail_run_attn(self._h, _ptr(attn), _ptr(residual), _ptr(out), rows,
                                         _stream_handle(stream))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_run_attn")

    def run_host(self, x, residual, out, rows: int = None, stream=None) -> None:
        """Same call on host (CPU) tensors: copies in, runs, copies back, synchronises."""
        rows = int(x.shape[0] if rows is None else rows)
        rc = self._lib.moe_tail_run_host(self._h, _ptr(x), _ptr(residual), _ptr(out), rows,
                                         _stream_handle(stream))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_run_host")

    def status(self) -> int:
        v = ctypes.c_int32(0)
        rc = self._lib.moe_tail_get_status(self._h, ctypes.byref(v))
        if rc not in (OK, ERR_DEVICE, ERR_TIMEOUT):
            raise MoeTailError(rc, "moe_tail_get_status")
        return int(v.value)

    def check_scratch(self) -> None:
        """Raise if a kernel wrote past the end of a scratch buffer (guard words)."""
        rc = self._lib.moe_tail_check_scratch(self._h)
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_check_scratch")

    def clear_status(self) -> None:
        rc = self._lib.moe_tail_clear_status(self._h)
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_clear_status")

    def routing(self, rows: int, stream=None):
        """(ids int32 [rows, k], wts float32 [rows, k], distinct experts) of the last run."""
        import numpy as np
        ids = np.zeros((rows, self.shape.k), np.int32)
        wts = np.zeros((rows, self.shape.k), np.float32)
        nd = ctypes.c_int32(0)
        rc = self._lib.moe_tail_debug_routing(self._h, ids.ctypes.data_as(ctypes.c_void_p),
                                              wts.ctypes.data_as(ctypes.c_void_p),
                                              ctypes.byref(nd), _stream_handle(stream))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_debug_routing")
        return ids, wts, int(nd.value)

    def set_stage_events(self, handles) -> None:
        """Record caller-owned CUDA events around each launch of later runs (list of
        cudaEvent_t handles, two per launch), or stop recording (None)."""
        if handles is None:
            rc = self._lib.moe_tail_set_stage_events(self._h, None, 0)
        else:
            arr = (ctypes.c_void_p * len(handles))(*handles)
            self._stage_events = arr
            rc = self._lib.moe_tail_set_stage_events(self._h, arr, len(handles))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_set_stage_events")

    def timeline(self) -> dict:
        """The last run's milestone stamps (handles with DEBUG_TIMELINE): microseconds after
        the norm launch passed its wait, None for a milestone not reached."""
        import numpy as np
        buf = np.zeros(len(TL_NAMES), np.uint64)
        rc = self._lib.moe_tail_debug_timeline(self._h, buf.ctypes.data_as(ctypes.c_void_p),
                                               len(TL_NAMES))
        if rc < 0:
            raise MoeTailError(rc, "moe_tail_debug_timeline")
        t0 = int(buf[0])
        return {n: (None if int(v) == 0 else (int(v) - t0) / 1000.0)
                for n, v in zip(TL_NAMES, buf)}

    def refresh_scales(self, stream=None) -> None:
        """Re-read w13s and w2s into the handle's copy in scale-factor atoms (after the
        caller changed them in place); enqueued on `stream`."""
        rc = self._lib.moe_tail_refresh_scales(self._h, _stream_handle(stream))
        if rc != OK:
            raise MoeTailError(rc, "moe_tail_refresh_scales")

    def launches_per_run(self, rows: int) -> int:
        return int(self._lib.moe_tail_launches_per_run(self._h, int(rows)))

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.moe_tail_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def attnres_mix(sub, prefix, blocks, n_blocks: int, commit: bool, q, gamma, mix, y,
                eps: float = 1e-6, rows: int = None, flags: int = 0, stream=None) -> None:
    """One call of the AttnRes residual mix + RMSNorm (attnres_mix.h): bf16 CUDA tensors
    sub, prefix, mix, y [rows, H], blocks [>= n_blocks (+1 on a commit), rows, H] (may be
    None when n_blocks == 0 and there is no commit), q, gamma [H].  prefix is updated in
    place; on a commit block n_blocks receives the new prefix and the prefix is zeroed."""
    lib = load_library()
    rows = int(sub.shape[0] if rows is None else rows)
    H = int(sub.shape[-1])
    rc = lib.moe_attnres_mix(rows, H, int(n_blocks), int(bool(commit)), float(eps), _ptr(sub),
                             _ptr(prefix), _ptr(blocks), _ptr(q), _ptr(gamma), _ptr(mix),
                             _ptr(y), int(flags), _stream_handle(stream))
    if rc != OK:
        raise MoeTailError(rc, "moe_attnres_mix")


def attnres_mix_status(clear: bool = False) -> int:
    """The mix's device status word (STATUS_* bits; synchronous); clear: zero it after."""
    v = ctypes.c_int32(0)
    rc = load_library().moe_attnres_mix_get_status(ctypes.byref(v), int(bool(clear)))
    if rc not in (OK, ERR_DEVICE):
        raise MoeTailError(rc, "moe_attnres_mix_get_status")
    return int(v.value)


def attnres_mix_ctas_per_row(hidden: int, n_blocks: int) -> int:
    """CTAs (one cluster) per row that attnres_mix launches for this shape (host only)."""
    rc = load_library().moe_attnres_mix_ctas_per_row(int(hidden), int(n_blocks))
    if rc < 0:
        raise MoeTailError(rc, "moe_attnres_mix_ctas_per_row")
    return rc


def weights_to_device(weights: dict, device="cuda"):
    """numpy weight arrays (from moe_layer_tail_gb300.inputs) -> CUDA tensors, same bits."""
    import numpy as np
    import torch
    out = {}
    for k, v in weights.items():
        if v.dtype == np.uint16:
            t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(v)
        out[k] = t.to(device)
    return out


def acts_to_device(a, device="cuda"):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_bits(t):
    import numpy as np
    import torch
    return t.detach().to("cpu").view(torch.int16).numpy().view(np.uint16).copy()
