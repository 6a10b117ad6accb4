"""Seeded synthetic inputs for the Qwen-Image-2.1 single-stream block.

This module holds no arithmetic of the method: it only names the workloads
(their shapes, segment layouts and value distributions) and draws random
tensors for them. Both the CPU oracle and the CUDA path consume what it
returns; neither side imports the other.

Recipe (one stream per tensor, so any single tensor can be rebuilt alone):

* tensor ``(tag, index)`` of workload seed ``s`` is the concatenation of
  chunks of ``CHUNK`` standard normals (float32, numpy ``PCG64`` seeded with
  ``SeedSequence([s, TAG_ID[tag], index, chunk])``), multiplied in float32
  by the tag's standard deviation, plus 1 for the RMSNorm weights;
* hidden states ``x`` ~ N(0, 1) float32;
* modulation vectors ``[scale1 | gate1 | scale2 | gate2]`` ~ N(0, 0.1)
  float32, one set for the step (``mods_t``) and one for the t = 0 prefix
  (``mods0``);
* projection weights ~ N(0, fan_in^-1/2) (standard deviation), rounded to
  the workload's 16-bit type, float16 or bfloat16 (round to nearest even
  from the float32 draw) -- the oracle widens exactly these values;
  fan_in = dim for q, k, v, o, gate, up and mlp_hidden for down;
* per-head RMSNorm weights ``norm_q``, ``norm_k`` = 1 + N(0, 0.05) float32;
* latent tokens ~ N(0, 1) float32 [n, 64]; img_in weight ~ N(0, 64^-1/2)
  and proj_out weight ~ N(0, dim^-1/2), float32 (the page keeps f32 copies
  of both for its device path); final_scale ~ N(0, 0.1) float32;
* timestep weights t_lin1 [dim, 256], t_lin2 [dim, dim], modulation
  [4 dim, dim], norm_out [dim, dim] ~ N(0, fan_in^-1/2) float32, no biases.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

CHUNK = 1 << 22

TAG_ID = {
    "x_prefix": 1,
    "x_target": 2,
    "mods_t": 3,
    "mods0": 4,
    "wq": 10,
    "wk": 11,
    "wv": 12,
    "wo": 13,
    "wgate": 14,
    "wup": 15,
    "wdown": 16,
    "norm_q": 17,
    "norm_k": 18,
    "tok": 30,          # latent tokens of the target image block
    "w_in": 31,         # img_in
    "w_out": 32,        # proj_out
    "final_scale": 33,  # final modulation of norm_out
    "t_lin1": 34,       # timestep_embedder.linear_1
    "t_lin2": 35,       # timestep_embedder.linear_2
    "modulation": 36,   # modulation.1
    "norm_out": 37,     # norm_out.linear
    "op_test": 50,  # single-operation checks: index = a case number
    "sketch": 60,   # Gaussian sketch matrices of the parity statistics
}

# Segment kinds, as the library's C ABI numbers them.
TEXT = 0
IMAGE = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: model geometry, the prompt prefix of each
    sequence and the shared target image block."""

    name: str
    dim: int
    heads: int
    mlp_hidden: int
    layers: int
    prefixes: tuple  # per sequence: tuple of (kind, a, b) segments
    target: tuple  # (h, w) of the target image block
    head_dim: int = 128
    axes: tuple = (16, 56, 56)
    eps: float = 1e-6
    theta: float = 10000.0
    seed: int = 0
    dtype: str = "f16"  # 16-bit type of the weights and activation rows: "f16" or "bf16"

    @property
    def nseq(self) -> int:
        return len(self.prefixes)

    def segs(self, s: int = 0) -> list:
        """Segment list of sequence ``s``: its prefix then the target."""
        return list(self.prefixes[s]) + [(IMAGE, self.target[0], self.target[1])]

    @property
    def n_target(self) -> int:
        return self.target[0] * self.target[1]

    def prefix_rows(self, s: int = 0) -> int:
        tot = 0
        for kind, a, b in self.prefixes[s]:
            tot += a if kind == TEXT else a * b
        return tot


def _t(n):
    return (TEXT, n, 0)


def _i(h, w):
    return (IMAGE, h, w)


WORKLOADS = {
    # single block, dim 256 (2 heads), prefix Text(18), target Image(16,16)
    "tiny_block_d256": Workload("tiny_block_d256", 256, 2, 768, 1, ((_t(18),),), (16, 16)),
    # one full-width block, prefix Text(18), target Image(64,64)
    "block_d4096_n4096": Workload("block_d4096_n4096", 4096, 32, 12288, 1, ((_t(18),),), (64, 64)),
    # 32 blocks, prefix Text(18) + condition Image(64,64), target Image(64,64)
    "step32_cond4114_n4096": Workload(
        "step32_cond4114_n4096", 4096, 32, 12288, 32, ((_t(18), _i(64, 64)),), (64, 64)
    ),
    # 32 blocks, prefix Text(18), target Image(128,128)
    "step32_n16384": Workload("step32_n16384", 4096, 32, 12288, 32, ((_t(18),),), (128, 128)),
    # CFG pair: prefixes Text(18) and Text(1), shared target Image(32,32)
    "cfg_pair32_n1024": Workload(
        "cfg_pair32_n1024", 4096, 32, 12288, 32, ((_t(18),), (_t(1),)), (32, 32)
    ),
    # --- extra parity cases (small, several tiles, ragged tails) ---
    # 32 chained blocks at dim 256 with a mixed block-causal prefix
    "chain32_d256_mixed": Workload(
        "chain32_d256_mixed", 256, 2, 768, 32, ((_t(5), _i(4, 6), _t(3), _i(3, 2)),), (10, 13)
    ),
    # ragged: 130 target rows, 150-row prefix with a 12x11 image block
    "ragged_d512": Workload("ragged_d512", 512, 4, 1536, 2, ((_t(7), _i(12, 11), _t(11)),), (10, 13)),
    # CFG pair at dim 256, prefixes of different lengths
    "cfg_pair_d256": Workload("cfg_pair_d256", 256, 2, 768, 2, ((_t(18),), (_t(1),)), (9, 15)),
    # smallest target: one row, one-row prefix
    "single_row_d256": Workload("single_row_d256", 256, 2, 768, 1, ((_t(1),),), (1, 1)),
    # an odd head count (3 heads, dim 384): the qkv and O projections have
    # N = 1152 and 384, not multiples of 256, so they run 128-column tiles;
    # 4356 target rows make the qkv's last wave a partial one (162 tile
    # pairs on 76 clusters), split along K
    "heads3_d384_n4356": Workload("heads3_d384_n4356", 384, 3, 1024, 2, ((_t(18),),), (66, 66)),
    # one full-width block with the 4114-row condition prefix: every launch
    # has the shapes of one layer of step32_cond4114_n4096 (small profiling
    # captures of those kernels)
    "block_cond4114_n4096": Workload(
        "block_cond4114_n4096", 4096, 32, 12288, 1, ((_t(18), _i(64, 64)),), (64, 64)
    ),
    # --- bf16 weights and activation rows ---
    "tiny_block_d256_bf16": Workload("tiny_block_d256_bf16", 256, 2, 768, 1, ((_t(18),),), (16, 16),
                                     dtype="bf16"),
    "chain32_d256_mixed_bf16": Workload(
        "chain32_d256_mixed_bf16", 256, 2, 768, 32, ((_t(5), _i(4, 6), _t(3), _i(3, 2)),), (10, 13), dtype="bf16"
    ),
    "cfg_pair_d256_bf16": Workload("cfg_pair_d256_bf16", 256, 2, 768, 2, ((_t(18),), (_t(1),)), (9, 15),
                                   dtype="bf16"),
    "block_d4096_n4096_bf16": Workload("block_d4096_n4096_bf16", 4096, 32, 12288, 1, ((_t(18),),), (64, 64),
                                       dtype="bf16"),
    "step32_cond4114_n4096_bf16": Workload(
        "step32_cond4114_n4096_bf16", 4096, 32, 12288, 32, ((_t(18), _i(64, 64)),), (64, 64), dtype="bf16"
    ),
}


def _stream_chunk(seed: int, tag: str, index: int, chunk: int, count: int) -> np.ndarray:
    ss = np.random.SeedSequence([seed, TAG_ID[tag], index, chunk])
    return np.random.Generator(np.random.PCG64(ss)).standard_normal(count, dtype=np.float32)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def normal(seed: int, tag: str, index: int, count: int, std: float, out: np.ndarray | None = None,
           dtype=np.float32, offset: float = 0.0) -> np.ndarray:
    """``count`` draws of tensor (tag, index): f32 standard normals times
    f32(std), plus ``offset``, cast to ``dtype`` (into ``out`` if given)."""
    if out is None:
        out = np.empty(count, dtype=dtype)
    assert out.size == count and out.dtype == np.dtype(dtype)
    std32 = np.float32(std)
    off32 = np.float32(offset)
    nchunks = (count + CHUNK - 1) // CHUNK

    def one(c):
        lo = c * CHUNK
        hi = min(count, lo + CHUNK)
        z = _stream_chunk(seed, tag, index, c, hi - lo)
        z *= std32
        if offset != 0.0:
            z += off32
        out[lo:hi] = z.astype(dtype, copy=False)

    if nchunks <= 1:
        for c in range(nchunks):
            one(c)
    else:
        list(_pool().map(one, range(nchunks)))
    return out


def x_prefix(w: Workload, s: int = 0) -> np.ndarray:
    """Prefix hidden states of sequence ``s``: float32 [lp, dim], N(0, 1)."""
    lp = w.prefix_rows(s)
    return normal(w.seed, "x_prefix", s, lp * w.dim, 1.0).reshape(lp, w.dim)


def x_target(w: Workload) -> np.ndarray:
    """Target hidden states, shared by every sequence: float32 [n, dim]."""
    return normal(w.seed, "x_target", 0, w.n_target * w.dim, 1.0).reshape(w.n_target, w.dim)


def mods_t(w: Workload) -> np.ndarray:
    """Step modulation [scale1|gate1|scale2|gate2]: float32 [4·dim], N(0, 0.1)."""
    return normal(w.seed, "mods_t", 0, 4 * w.dim, 0.1)


LATENT_CHANNELS = 64


def tokens(w: Workload) -> np.ndarray:
    """Latent tokens of the target image: float32 [n, 64], N(0, 1)."""
    return normal(w.seed, "tok", 0, w.n_target * LATENT_CHANNELS, 1.0).reshape(w.n_target, LATENT_CHANNELS)


def w_in(w: Workload) -> np.ndarray:
    """img_in weight: float32 [dim, 64], N(0, 64^-1/2)."""
    return normal(w.seed, "w_in", 0, w.dim * LATENT_CHANNELS, LATENT_CHANNELS ** -0.5).reshape(w.dim, LATENT_CHANNELS)


def w_out(w: Workload) -> np.ndarray:
    """proj_out weight: float32 [64, dim], N(0, dim^-1/2)."""
    return normal(w.seed, "w_out", 0, LATENT_CHANNELS * w.dim, w.dim ** -0.5).reshape(LATENT_CHANNELS, w.dim)


def final_scale(w: Workload) -> np.ndarray:
    """Final modulation (norm_out scale) of the step: float32 [dim], N(0, 0.1)."""
    return normal(w.seed, "final_scale", 0, w.dim, 0.1)


TIMESTEP_CHANNELS = 256


def timestep_weights(w: Workload) -> dict:
    """t_lin1 [dim, 256], t_lin2 [dim, dim], modulation [4 dim, dim],
    norm_out [dim, dim]: float32, N(0, fan_in^-1/2)."""
    d = w.dim
    shapes = {"t_lin1": (d, TIMESTEP_CHANNELS), "t_lin2": (d, d), "modulation": (4 * d, d), "norm_out": (d, d)}
    return {k: normal(w.seed, k, 0, r * c, c ** -0.5).reshape(r, c) for k, (r, c) in shapes.items()}


def mods0(w: Workload) -> np.ndarray:
    """t = 0 modulation of the prefix: float32 [4·dim], N(0, 0.1)."""
    return normal(w.seed, "mods0", 0, 4 * w.dim, 0.1)


WEIGHT_TAGS = ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")


def weight_shape(w: Workload, tag: str) -> tuple:
    H, I = w.dim, w.mlp_hidden
    return {
        "wq": (H, H), "wk": (H, H), "wv": (H, H), "wo": (H, H),
        "wgate": (I, H), "wup": (I, H), "wdown": (H, I),
    }[tag]


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 values -> bfloat16 bit patterns (uint16), rounded to nearest
    even (the draws hold no NaN)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> the same values as float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def weight(w: Workload, layer: int, tag: str, out: np.ndarray | None = None) -> np.ndarray:
    """Projection weight of ``layer`` in nn.Linear layout [out, in], as the
    device stores it: float16 for f16 workloads, bfloat16 bit patterns
    (uint16) for bf16 workloads (into ``out`` if given)."""
    rows, cols = weight_shape(w, tag)
    flat = None if out is None else out.reshape(-1)
    if w.dtype == "bf16":
        z = normal(w.seed, tag, layer, rows * cols, cols ** -0.5)
        b = bf16_bits(z)
        if flat is not None:
            flat[:] = b
            b = flat
        return b.reshape(rows, cols)
    res = normal(w.seed, tag, layer, rows * cols, cols ** -0.5, out=flat, dtype=np.float16)
    return res.reshape(rows, cols)


def weight_values(w: Workload, layer: int, tag: str) -> np.ndarray:
    """The values of ``weight``: float16, or float32 holding the bfloat16
    values exactly."""
    a = weight(w, layer, tag)
    return bf16_values(a) if w.dtype == "bf16" else a


def norm_weight(w: Workload, layer: int, tag: str) -> np.ndarray:
    """Per-head RMSNorm weight ``norm_q``/``norm_k``: float32 [head_dim]."""
    return normal(w.seed, tag, layer, w.head_dim, 0.05, offset=1.0)


def layer_weights(w: Workload, layer: int) -> dict:
    """All weights of one layer (projection values as stored on the device:
    float16, or bfloat16 values as float32; float32 norms)."""
    d = {t: weight_values(w, layer, t) for t in WEIGHT_TAGS}
    d["norm_q"] = norm_weight(w, layer, "norm_q")
    d["norm_k"] = norm_weight(w, layer, "norm_k")
    return d


def op_tensor(seed: int, case: int, slot: int, shape, std: float = 1.0, offset: float = 0.0,
              dtype=np.float32) -> np.ndarray:
    """A seeded tensor for a single-operation check: stream (seed, case,
    slot) of the "op_test" tag."""
    count = int(np.prod(shape))
    return normal(seed * 1000003 + case, "op_test", slot, count, std, dtype=dtype, offset=offset).reshape(shape)


def sketch(rows: int, k: int, side: int) -> np.ndarray:
    """A seeded Gaussian sketch matrix float64 [k, rows] (N(0, 1) entries),
    used by the parity tests to reduce a [rows, cols] output X to the small
    matrix L X R^T (L = sketch(rows, k, 0), R = sketch(cols, k, 1)) whose
    relative L2 difference estimates that of the whole output. Random
    numbers only: stream (0, "sketch", rows * 4 + side) of the recipe."""
    return normal(0, "sketch", rows * 4 + side, k * rows, 1.0).astype(np.float64).reshape(k, rows)
