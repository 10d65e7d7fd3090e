"""Seeded synthetic inputs of the MoE layer tail, shared by the tests and the benchmark.

This module draws random numbers and packs them into the library's storage formats; it
holds none of the tail's arithmetic (no norm, routing, dequantisation or expert math), so
both the CUDA path and the CPU oracle can take their inputs from it.

Workloads (shapes and value distributions of the five configurations the method is
measured on; R rows, hidden H, E experts top-k, expert inter I, shared inter Is):

  tiny                       R 1,  H 256,  E 8,   k 2,  I 128,  Is 128
  r1_h7168_e256k8            R 1,  H 7168, E 256, k 8,  I 2048, Is 2048
  r8_h7168_e256k8_similar    R 8,  same shapes; rows correlated so ~40% of picks repeat
  r4_h8192_e512k10           R 4,  H 8192, E 512, k 10, I 1024, Is 4096
  r16_h8192_e512k10_neartie  R 16, same shapes; the parity tests inject k-th/(k+1)-th
                             router-logit margins of 1e-2 into these rows
  r32_h7168_e256k8_similar   R 32, the shapes of the 8-row workload: more than 16 rows per
                             call (MTP verify / short prefill widths; the default expert form)

Recipe (numpy PCG64 seeded by the workload's seed; bf16 values are float32 draws rounded
to bf16 by torch):
  x, residual       N(0, 1).  For the "similar" workload row r is
                    c * z0 + sqrt(1 - c^2) * z_r for both x and residual (z0 shared by all
                    rows); c is read from tests/golden/similar_c.json, which a committed
                    script fits with the oracle so that ~40% of the picks repeat.
  gamma             1 + N(0, 0.1)
  router W_r [E,H]  N(0, 1/sqrt(H))
  MXFP4 codes       uniform bytes (each nibble uniform over the 16 E2M1 codes)
  E8M0 scales       round(log2(1/sqrt(K))) + 127 + d, d uniform in {-1, 0, +1}, K the
                    matrix's reduction length (H for w13, I for w2); the jitter makes each
                    block's own scale matter.
  shared Ws13, Ws2  N(0, 1/sqrt(K)) in bf16, K = H and Is.
"""
import json
import math
import os
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class TailShape:
    R: int
    H: int
    E: int
    k: int
    I: int
    Is: int
    eps: float = 1e-6
    Ha: int = 0  # attention output width in front of the tail (0: none)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: TailShape
    seed: int
    kind: str  # "plain" | "similar" | "neartie"


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", TailShape(1, 256, 8, 2, 128, 128), 0, "plain"),
        Workload("r1_h7168_e256k8", TailShape(1, 7168, 256, 8, 2048, 2048), 1, "plain"),
        Workload("r8_h7168_e256k8_similar", TailShape(8, 7168, 256, 8, 2048, 2048), 2, "similar"),
        Workload("r4_h8192_e512k10", TailShape(4, 8192, 512, 10, 1024, 4096), 3, "plain"),
        Workload("r16_h8192_e512k10_neartie", TailShape(16, 8192, 512, 10, 1024, 4096), 4,
                 "neartie"),
        Workload("r32_h7168_e256k8_similar", TailShape(32, 7168, 256, 8, 2048, 2048), 5,
                 "similar"),
    ]
}

# The workload the benchmark times (8 rows, 256 experts top-8, ~40% repeated picks).
BENCH_WORKLOAD = "r8_h7168_e256k8_similar"

_GOLDEN = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests",
                       "golden")


def similar_c(default: float = None) -> float:
    """Row-correlation c of the 'similar' workload, as fitted by tests/golden/fit_similar_c.py."""
    path = os.path.join(_GOLDEN, "similar_c.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["c"])
    if default is None:
        raise FileNotFoundError(path)
    return default


def to_bf16_bits(a) -> np.ndarray:
    """float array -> uint16 bf16 bits (round to nearest even, via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _normal_bf16(rng, shape, std, mean=0.0):
    return to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
                        + np.float32(mean))


def _e8m0_scales(rng, shape, K):
    base = int(round(math.log2(1.0 / math.sqrt(K)))) + 127
    jitter = rng.integers(-1, 2, size=shape, dtype=np.int16)
    return (base + jitter).astype(np.uint8)


def _codes(rng, shape):
    """Uniform random bytes: the raw 64-bit outputs of the seeded PCG64 stream, little-endian."""
    n = int(np.prod(shape))
    raw = rng.bit_generator.random_raw((n + 7) // 8)
    return raw.astype("<u8", copy=False).view(np.uint8)[:n].reshape(shape)


_WEIGHT_STREAMS = ("gamma", "w_r", "w13_codes", "w13_scales", "w2_codes", "w2_scales", "ws13",
                   "ws2", "ws_gate", "w_o")
_LAYER_WEIGHTS = _WEIGHT_STREAMS[:-2]  # the shared-expert gate and out_proj are optional


def make_weight(shape: TailShape, seed: int, key: str) -> np.ndarray:
    """One weight array; each array has its own seeded stream, so any subset can be drawn."""
    H, E, I, Is = shape.H, shape.E, shape.I, shape.Is
    rng = np.random.default_rng([seed, 1, _WEIGHT_STREAMS.index(key)])
    if key == "gamma":
        return _normal_bf16(rng, (H,), 0.1, 1.0)
    if key == "w_r":
        return _normal_bf16(rng, (E, H), 1.0 / math.sqrt(H))
    if key == "w13_codes":
        return _codes(rng, (E, 2 * I, H // 2))
    if key == "w13_scales":
        return _e8m0_scales(rng, (E, 2 * I, H // 32), H)
    if key == "w2_codes":
        return _codes(rng, (E, H, I // 2))
    if key == "w2_scales":
        return _e8m0_scales(rng, (E, H, I // 32), I)
    if key == "ws13":
        return _normal_bf16(rng, (2 * Is, H), 1.0 / math.sqrt(H))
    if key == "ws2":
        return _normal_bf16(rng, (H, Is), 1.0 / math.sqrt(Is))
    if key == "ws_gate":  # logit n . g ~ N(0, 1) for normalised rows
        return _normal_bf16(rng, (H,), 1.0 / math.sqrt(H))
    if key == "w_o":  # attention output projection [H, Ha]
        return _normal_bf16(rng, (H, shape.Ha), 1.0 / math.sqrt(shape.Ha))
    raise KeyError(key)


def make_weights(shape: TailShape, seed: int, keys=_LAYER_WEIGHTS) -> dict:
    """Weights of one layer: gamma, router, routed MXFP4 experts, shared bf16 expert (add
    "ws_gate" to `keys` for the shared expert's sigmoid gate)."""
    return {key: make_weight(shape, seed, key) for key in keys}


def make_activations(shape: TailShape, seed: int, kind: str = "plain", c: float = None,
                     rows: int = None) -> dict:
    """x and residual [rows, H] bf16 bits.  kind 'similar' correlates the rows with weight c."""
    R = shape.R if rows is None else rows
    H = shape.H
    rng = np.random.default_rng([seed, 2])
    if kind == "similar":
        if c is None:
            c = similar_c()
        z0 = rng.standard_normal(size=(1, H), dtype=np.float32)
        zx = rng.standard_normal(size=(R, H), dtype=np.float32)
        w0 = rng.standard_normal(size=(1, H), dtype=np.float32)
        wr = rng.standard_normal(size=(R, H), dtype=np.float32)
        s = np.float32(math.sqrt(max(0.0, 1.0 - c * c)))
        x = np.float32(c) * z0 + s * zx
        res = np.float32(c) * w0 + s * wr
    else:
        x = rng.standard_normal(size=(R, H), dtype=np.float32)
        res = rng.standard_normal(size=(R, H), dtype=np.float32)
    return {"x": to_bf16_bits(x), "residual": to_bf16_bits(res)}


def make_attention_output(shape: TailShape, seed: int, rows: int = None) -> np.ndarray:
    """attn [rows, Ha] bf16 bits, N(0, 1): the input of the attention output projection."""
    R = shape.R if rows is None else rows
    rng = np.random.default_rng([seed, 3])
    return to_bf16_bits(rng.standard_normal(size=(R, shape.Ha), dtype=np.float32))


def make_inputs(name_or_wl, c: float = None) -> dict:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    d = make_weights(wl.shape, wl.seed)
    d.update(make_activations(wl.shape, wl.seed, wl.kind, c))
    return d


# ------------------------------------------ second workload: the AttnRes residual mix ----
#
# A decoder runs the mix once per sublayer: L calls on the same R rows, each adding its
# sublayer's output into the running sum of the current block (the prefix) and mixing the
# committed blocks with that prefix.  Block 0 (the embedding) is committed before the first
# call and the prefix starts at zero; every `block_calls` calls the last call of a block
# commits its prefix as the next block.  Recipe per family:
#   "unit"    sublayer outputs and the embedding N(0, 1)
#   "scaled"  the same, each (call, row) scaled by 2^u, u uniform in {0, ..., 11}, so rows
#             reach magnitudes of a few thousand
#   both      query q_l [H] N(0, 1/sqrt(H)) (source scores ~ N(0, 1)), gamma_l 1 + N(0, 0.1)


@dataclass(frozen=True)
class MixSequence:
    R: int
    H: int = 7168
    L: int = 187
    block_calls: int = 24
    eps: float = 1e-6

    def n_blocks(self, call: int) -> int:
        """Committed blocks before call `call` (0-based)."""
        return 1 + call // self.block_calls

    def commit(self, call: int) -> bool:
        return (call + 1) % self.block_calls == 0

    @property
    def max_blocks(self) -> int:
        """Blocks the buffer must hold: the committed ones plus the last call's commit."""
        last = self.L - 1
        return self.n_blocks(last) + (1 if self.commit(last) else 0)


def make_mix_sequence(seq: MixSequence, seed: int, family: str = "unit") -> dict:
    """sub [L,R,H], q [L,H], gamma [L,H], blocks [max_blocks,R,H] (block 0 the embedding,
    the rest zero) and prefix [R,H] (zero), all bf16 bits."""
    L, R, H = seq.L, seq.R, seq.H
    rng = np.random.default_rng([seed, 4])
    sub = rng.standard_normal(size=(L, R, H), dtype=np.float32)
    emb = rng.standard_normal(size=(R, H), dtype=np.float32)
    if family == "scaled":
        u = rng.integers(0, 12, size=(L, R, 1))
        sub = sub * np.exp2(u).astype(np.float32)
    elif family != "unit":
        raise ValueError(family)
    q = rng.standard_normal(size=(L, H), dtype=np.float32) * np.float32(1.0 / math.sqrt(H))
    gamma = np.float32(1.0) + rng.standard_normal(size=(L, H), dtype=np.float32) * np.float32(0.1)
    blocks = np.zeros((seq.max_blocks, R, H), np.uint16)
    blocks[0] = to_bf16_bits(emb)
    return {"sub": to_bf16_bits(sub), "q": to_bf16_bits(q), "gamma": to_bf16_bits(gamma),
            "blocks": blocks, "prefix": np.zeros((R, H), np.uint16)}


def mix_call_bytes(R: int, H: int, n_blocks: int, commit: bool) -> int:
    """Bytes one mix call must move: the committed sources, the prefix and the sublayer
    output read, q and gamma read, the prefix (and on a commit the new block) written, the
    mixture and the normalised output written."""
    return 2 * (n_blocks * R * H + 2 * R * H + 2 * H + (2 if commit else 1) * R * H + 2 * R * H)


def algorithmic_bytes(shape: TailShape, distinct: int, rows: int = None,
                      gated: bool = False, out_proj: bool = False) -> int:
    """Bytes one call must move: each distinct expert's MXFP4 codes and scales once, the bf16
    router, shared expert (and its gate vector), gamma once, and x, residual (read and
    write) and out; with out_proj, its [H, Ha] weights and the attention output instead of
    x."""
    R = shape.R if rows is None else rows
    H, E, I, Is = shape.H, shape.E, shape.I, shape.Is
    per_expert = 3 * I * H // 2 + 3 * I * H // 32
    b = (distinct * per_expert + E * H * 2 + 3 * Is * H * 2 + H * 2 + R * H * 2 * 4
         + (H * 2 if gated else 0))
    if out_proj:
        b += H * shape.Ha * 2 + R * shape.Ha * 2 - R * H * 2
    return b
