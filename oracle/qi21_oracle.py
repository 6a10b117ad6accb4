"""CPU oracle of the Qwen-Image-2.1 single-stream DiT block (prefill + step).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module. The CUDA
library never calls it, shares no code with it and has no fallback to it.

Source: the docs.rs page of ``cortiq_engine/qwen_image21.rs`` (v0.8.4),
the CPU-exact reference path. Each function names the item of that page it
restates. Precision: everything in float64 (stricter than the page's f32
activations and f32 host GEMM), except where the page fixes a float32 step
that changes values beyond rounding: the RoPE tables (``rope_tables``: f32
frequencies, f32 angle, f32 cos/sin). Matrix products use numpy's ``@``
(a library primitive) with no blocking or reordering of the definition.

Pinned by ``tests/test_oracle_pins.py`` (worked examples of the page's own
tests, closed forms, brute force and invariants). Helpers without a pin of
their own (``gated_add``, ``linear_row``) are pinned through the functions
that use them (the zero-gate identity, the closed-form blocks, the
timestep chain). The absolute values of a full-size block are parity
unpinned: the pages print no activations, so they rest on the pinned
pieces and on the invariants (prefill + step = joint forward under the
block-causal mask; blocks with Wq = Wk = 0 or Wv = 0 in closed form).
"""
from __future__ import annotations

import numpy as np

TEXT = 0
IMAGE = 1


# --------------------------------------------------------------- layout ----
# qwen_image21.rs, "Seg", "Qi21Layout" (total, prefix_len, target, validate,
# block_ids, positions).

def seg_len(seg) -> int:
    kind, a, b = seg
    return a if kind == TEXT else a * b


def total_rows(segs) -> int:
    return sum(seg_len(s) for s in segs)


def prefix_len(segs) -> int:
    """Rows before the target block (the last segment)."""
    return total_rows(segs) - seg_len(segs[-1])


def validate(segs) -> None:
    """The layout ends with a non-empty target image and has a non-empty
    prefix (qwen_image21.rs, Qi21Layout::validate)."""
    if not segs:
        raise ValueError("empty layout")
    kind, a, b = segs[-1]
    if kind != IMAGE or a <= 0 or b <= 0:
        raise ValueError("the layout must end with a non-empty target image block")
    if prefix_len(segs) == 0:
        raise ValueError("the prompt prefix is empty")


def block_ids(segs) -> np.ndarray:
    """Per row: -1 for text, else the running image-block id
    (qwen_image21.rs, Qi21Layout::block_ids)."""
    out = []
    bid = 0
    for kind, a, b in segs:
        if kind == TEXT:
            out += [-1] * a
        else:
            out += [bid] * (a * b)
            bid += 1
    return np.array(out, dtype=np.int32)


def positions(segs) -> np.ndarray:
    """(frame, h, w) RoPE positions of every row (qwen_image21.rs,
    Qi21Layout::positions): a text row sits at [p, p, p] and advances p by
    one; an image block of h x w rows holds the frame at p, centres row r on
    r - (h - floor(h/2)) and column c on c - (w - floor(w/2)) in raster
    order, then advances p by max(h, w)."""
    out = []
    p = 0
    for kind, a, b in segs:
        if kind == TEXT:
            for _ in range(a):
                out.append((p, p, p))
                p += 1
        else:
            h, w = a, b
            for r in range(h):
                for c in range(w):
                    out.append((p, r - (h - h // 2), c - (w - w // 2)))
            p += max(h, w)
    return np.array(out, dtype=np.int64).reshape(-1, 3)


def prefix_visibility(segs) -> np.ndarray:
    """Block-causal mask of the prefix as leading runs (qwen_image21.rs,
    Qi21Dit::prefill): prefix row i sees keys [0, end[i]) with end[i] = i+1
    for a text row and one past the last row of its own image block for an
    image row."""
    lp = prefix_len(segs)
    ids = block_ids(segs)[:lp]
    end = np.zeros(lp, dtype=np.uint32)
    for i in range(lp):
        if ids[i] < 0:
            end[i] = i + 1
        else:
            e = i + 1
            while e < lp and ids[e] == ids[i]:
                e += 1
            end[i] = e
    return end


def rope_tables(pos: np.ndarray, axes=(16, 56, 56), theta: float = 10000.0):
    """cos/sin tables [rows, head_dim/2] in pair order frame, h, w
    (qwen_image21.rs, rope_tables). The page fixes float32 here: the
    frequency of pair i of an axis of width d is 1 / f32(theta)^(2i/d), the
    angle is f32(position) * frequency, and cos/sin are taken in f32."""
    pos = np.asarray(pos, dtype=np.int64).reshape(-1, 3)
    freqs = []
    for d in axes:
        e = (2 * np.arange(d // 2, dtype=np.float32)) / np.float32(d)
        freqs.append(np.float32(1.0) / np.power(np.float32(theta), e, dtype=np.float32))
    cols = []
    for a, fr in enumerate(freqs):
        ang = pos[:, a].astype(np.float32)[:, None] * fr[None, :]
        cols.append(ang.astype(np.float32))
    ang = np.concatenate(cols, axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def target_rope(segs, axes=(16, 56, 56), theta=10000.0):
    """RoPE tables of the target rows at their positions after this
    sequence's own prefix (qwen_image21.rs, Qi21Dit::target_rope)."""
    pos = positions(segs)
    return rope_tables(pos[prefix_len(segs):], axes, theta)


# --------------------------------------------------------------- pieces ----

def silu(v):
    """v / (1 + e^-v) (qwen_image21.rs, silu)."""
    return v / (1.0 + np.exp(-v))


def layer_norm(x, eps):
    """Affine-free LayerNorm with biased variance over the last axis
    (qwen_image21.rs, layer_norm_into)."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps)


def norm_mod(x, scale, eps):
    """dst = LN(x) * (1 + scale) (qwen_image21.rs, Qi21Dit::norm_mod)."""
    return layer_norm(x, eps) * (1.0 + np.asarray(scale, dtype=np.float64))


def gated_add(x, y, gate_raw):
    """x + tanh(gate) * y (qwen_image21.rs, Qi21Dit::gated_add; the gate
    chunk is tanh-ed first, as block_cpu does)."""
    return x + np.tanh(np.asarray(gate_raw, dtype=np.float64)) * y


def rms_norm(v, w, eps):
    """Per-vector RMSNorm over the last axis times the weight as is
    (qwen_image21.rs, rms_norm_inplace)."""
    v = np.asarray(v, dtype=np.float64)
    ss = (v * v).mean(axis=-1, keepdims=True)
    return v / np.sqrt(ss + eps) * np.asarray(w, dtype=np.float64)


def rope_rotate(v, cos, sin):
    """Rotate the interleaved pairs (v[2j], v[2j+1]) of each head vector by
    the row's angle j: (a c - b s, a s + b c) (qwen_image21.rs,
    Qi21Dit::qk_norm_rope). v: [rows, heads, hd]; cos/sin: [rows, hd/2]."""
    a = v[..., 0::2]
    b = v[..., 1::2]
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    out = np.empty_like(v)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def qk_norm_rope(t, w, cos, sin, heads, head_dim, eps):
    """Per (row, head): RMSNorm * w over head_dim, then the interleaved
    RoPE (qwen_image21.rs, Qi21Dit::qk_norm_rope). t: [rows, heads*hd]."""
    rows = t.shape[0]
    v = np.asarray(t, dtype=np.float64).reshape(rows, heads, head_dim)
    v = rms_norm(v, w, eps)
    return rope_rotate(v, cos, sin).reshape(rows, heads * head_dim)


def masked_softmax(scores, visible):
    """Row softmax over the first visible[i] entries of row i, the rest
    exactly 0 (qwen_image21.rs, softmax_prefix)."""
    s = np.asarray(scores, dtype=np.float64)
    m = s.shape[1]
    keep = np.arange(m)[None, :] < np.asarray(visible, dtype=np.int64)[:, None]
    s = np.where(keep, s, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    p = np.where(keep, np.exp(s - mx), 0.0)
    return p / p.sum(axis=1, keepdims=True)


def attention(q, k, v, visible, heads, head_dim):
    """Per head: q * (1/sqrt(hd)), S = q k^T, masked softmax with query i
    seeing keys [0, visible[i]), O = P v (qwen_image21.rs,
    Qi21Dit::attention). q: [n, heads*hd]; k, v: [m, heads*hd]."""
    n = q.shape[0]
    m = k.shape[0]
    qh = np.asarray(q, dtype=np.float64).reshape(n, heads, head_dim)
    kh = np.asarray(k, dtype=np.float64).reshape(m, heads, head_dim)
    vh = np.asarray(v, dtype=np.float64).reshape(m, heads, head_dim)
    scale = 1.0 / np.sqrt(head_dim)
    out = np.empty((n, heads, head_dim), dtype=np.float64)
    for h in range(heads):
        s = (qh[:, h, :] * scale) @ kh[:, h, :].T
        p = masked_softmax(s, visible)
        out[:, h, :] = p @ vh[:, h, :]
    return out.reshape(n, heads * head_dim)


# ---------------------------------------------------------------- block ----

def block(x, W, mods, cos, sin, cfg, kv_prefix=None, visible=None, rows=None, lin=None):
    """One block on the query rows of x (qwen_image21.rs, Qi21Dit::block_cpu):

        xn = LN(x) (1 + s1); q, k, v = xn Wq^T, xn Wk^T, xn Wv^T
        q, k <- qk RMSNorm + RoPE
        o = attention(q, [k_prefix ++ k], [v_prefix ++ v], visible)
        x += tanh(g1) (o Wo^T)
        xn = LN(x) (1 + s2); x += tanh(g2) ((silu(xn Wg^T) * (xn Wu^T)) Wd^T)

    x: [M, H]; W: dict of the layer's weights (float16 or float64 arrays);
    mods: [4H] raw [s1|g1|s2|g2]; cos/sin: [M, hd/2] of the query rows;
    kv_prefix: optional (K, V) [lp, H] post-RoPE keys/values seen first;
    visible: [M] leading-run key counts (default: every key).

    rows: optional subset of query rows whose output is wanted. Keys and
    values are still formed from every row of x; the query-side work is
    restricted to these rows (each output row depends only on its own
    query and on all keys).

    lin: the projection a -> a W^T (default: the plain product; the FP8
    variant passes linear_fp8).

    Returns (x_out [len(rows) or M, H], k [M, H], v [M, H]) with k, v the
    block's own post-RoPE keys and values."""
    H, nh, hd, eps = cfg["dim"], cfg["heads"], cfg["head_dim"], cfg["eps"]
    f = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    x = f(x)
    mods = f(mods)
    s1, g1, s2, g2 = mods[:H], mods[H:2 * H], mods[2 * H:3 * H], mods[3 * H:]
    M = x.shape[0]
    sel = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    if lin is None:
        lin = lambda a, w: a @ f(w).T  # noqa: E731
    xn = norm_mod(x, s1, eps)
    k = qk_norm_rope(lin(xn, W["wk"]), W["norm_k"], cos, sin, nh, hd, eps)
    v = lin(xn, W["wv"])
    q = qk_norm_rope(lin(xn[sel], W["wq"]), W["norm_q"], f(cos)[sel], f(sin)[sel], nh, hd, eps)
    if kv_prefix is not None:
        ka = np.concatenate([f(kv_prefix[0]), k], axis=0)
        va = np.concatenate([f(kv_prefix[1]), v], axis=0)
    else:
        ka, va = k, v
    if visible is None:
        vis = np.full(len(sel), ka.shape[0], dtype=np.int64)
    else:
        vis = np.asarray(visible, dtype=np.int64)[sel]
    o = attention(q, ka, va, vis, nh, hd)
    xs = gated_add(x[sel], lin(o, W["wo"]), g1)
    xn2 = norm_mod(xs, s2, eps)
    hid = silu(lin(xn2, W["wgate"])) * lin(xn2, W["wup"])
    xs = gated_add(xs, lin(hid, W["wdown"]), g2)
    return xs, k, v


def cfg_of(w) -> dict:
    """Geometry dict of a synthetic workload."""
    return {"dim": w.dim, "heads": w.heads, "head_dim": w.head_dim, "eps": w.eps,
            "axes": tuple(w.axes), "theta": w.theta}


def prefill(x_prefix, weights, mods0, segs, cfg, keep_x=False, lin=None):
    """The prefix through every block with the t = 0 modulation and the
    block-causal mask, keeping each layer's own post-RoPE (K, V)
    (qwen_image21.rs, Qi21Dit::prefill, host loop).

    weights: list of per-layer weight dicts. Returns (cache, xs) with cache
    a list of (K, V) [lp, H] per layer and xs the hidden state after each
    block (if keep_x)."""
    validate(segs)
    lp = prefix_len(segs)
    pos = positions(segs)
    cos, sin = rope_tables(pos[:lp], cfg["axes"], cfg["theta"])
    vis = prefix_visibility(segs)
    x = np.asarray(x_prefix, dtype=np.float64)
    cache, xs = [], []
    for W in weights:
        x, k, v = block(x, W, mods0, cos, sin, cfg, None, vis, lin=lin)
        cache.append((k, v))
        if keep_x:
            xs.append(x)
    return cache, xs


def step(x_target, weights, mods, segs, cache, cfg, keep_x=False, lin=None):
    """The target rows through every block against [cached prefix, own rows]
    with every key visible (qwen_image21.rs, Qi21Dit::step_cpu, the block
    loop; the image embedding and the final projection are outside it).
    Returns (x_out, xs)."""
    validate(segs)
    lp = prefix_len(segs)
    x = np.asarray(x_target, dtype=np.float64)
    n = x.shape[0]
    cos, sin = target_rope(segs, cfg["axes"], cfg["theta"])
    vis = np.full(n, lp + n, dtype=np.int64)
    xs = []
    for layer, W in enumerate(weights):
        x, _, _ = block(x, W, mods, cos, sin, cfg, cache[layer], vis, lin=lin)
        if keep_x:
            xs.append(x)
    return x, xs


def joint_forward(x_prefix, x_target, weights, mods0, mods, segs, cfg):
    """The whole joint sequence [prefix; target] through every block with
    no cache: prefix rows modulated from t = 0 and target rows from t
    (causal_condition), prefix row i seeing keys [0, end[i]) and target rows
    seeing every key -- the block-causal mask of the page's module notes
    ("(q >= kv) or same_image_block"). Returns the target rows' output.

    The per-row modulation is a restatement, not a call of ``block``: each
    row takes LN(x)(1+s) and the two gates of its own modulation set."""
    validate(segs)
    H, nh, hd, eps = cfg["dim"], cfg["heads"], cfg["head_dim"], cfg["eps"]
    f = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    lp = prefix_len(segs)
    x = np.concatenate([f(x_prefix), f(x_target)], axis=0)
    T = x.shape[0]
    cos, sin = rope_tables(positions(segs), cfg["axes"], cfg["theta"])
    vis = np.concatenate([prefix_visibility(segs).astype(np.int64), np.full(T - lp, T, dtype=np.int64)])
    m = np.empty((T, 4 * H), dtype=np.float64)
    m[:lp] = f(mods0)
    m[lp:] = f(mods)
    s1, g1, s2, g2 = m[:, :H], m[:, H:2 * H], m[:, 2 * H:3 * H], m[:, 3 * H:]
    for W in weights:
        xn = layer_norm(x, eps) * (1.0 + s1)
        q = qk_norm_rope(xn @ f(W["wq"]).T, W["norm_q"], cos, sin, nh, hd, eps)
        k = qk_norm_rope(xn @ f(W["wk"]).T, W["norm_k"], cos, sin, nh, hd, eps)
        v = xn @ f(W["wv"]).T
        o = attention(q, k, v, vis, nh, hd)
        x = x + np.tanh(g1) * (o @ f(W["wo"]).T)
        xn = layer_norm(x, eps) * (1.0 + s2)
        hid = silu(xn @ f(W["wgate"]).T) * (xn @ f(W["wup"]).T)
        x = x + np.tanh(g2) * (hid @ f(W["wdown"]).T)
    return x[lp:]


def embed_image(tok, w_in):
    """img_in: latent tokens [n, in_channels] -> hidden states [n, dim],
    no bias (qwen_image21.rs, Qi21Dit::embed_image): x = tok W_in^T with
    W_in [dim, in_channels]."""
    return np.asarray(tok, dtype=np.float64) @ np.asarray(w_in, dtype=np.float64).T


def final_layer(x, final_scale, w_out, eps):
    """After the blocks: LN(x)(1 + final_scale), then proj_out [out, dim]
    with no bias (qwen_image21.rs, Qi21Dit::step_cpu, the last two
    statements; the device path passes fs = 1 + final_scale)."""
    return norm_mod(x, final_scale, eps) @ np.asarray(w_out, dtype=np.float64).T


def denoise(tok, w_in, weights, mods, final_scale, w_out, segs, cache, cfg):
    """One denoiser call: latent tokens -> velocity (qwen_image21.rs,
    Qi21Dit::step_cpu): embed_image, the blocks against the cached prefix,
    the final modulated LayerNorm and proj_out."""
    x = embed_image(tok, w_in)
    x, _ = step(x, weights, mods, segs, cache, cfg)
    return final_layer(x, final_scale, w_out, cfg["eps"])


# ------------------------------------------------------------ timestep ----
# qwen_image21.rs, Qi21Dit::temb and Qi21Dit::mods: the one shared modulation
# of a denoiser call, from the model input t in [0, 1].

TIMESTEP_CHANNELS = 256


def timestep_sinusoid(t):
    """[cos(a_i) | sin(a_i)], i < 128, a_i = (1000 t) f_i with
    f_i = exp(-ln(10000) i / 128); every step in float32 as the page fixes
    it (qwen_image21.rs, Qi21Dit::temb, the loop over HALF)."""
    half = TIMESTEP_CHANNELS // 2
    ts = np.float32(1000.0) * np.float32(t)
    i = np.arange(half, dtype=np.float32)
    f = np.exp(-np.log(np.float32(10000.0)) * i / np.float32(half))
    a = ts * f
    return np.concatenate([np.cos(a), np.sin(a)]).astype(np.float32)


def linear_row(w, x):
    """One vector through a bias-free nn.Linear [out, in]: f64 sums rounded
    to f32 per output (qwen_image21.rs, lin_row)."""
    return (np.asarray(w, dtype=np.float64) @ np.asarray(x, dtype=np.float64)).astype(np.float32)


def timestep_embed(t, t_lin1, t_lin2):
    """temb [dim] = t_lin2 silu(t_lin1 e(t)) (qwen_image21.rs, Qi21Dit::temb)."""
    h = silu(linear_row(t_lin1, timestep_sinusoid(t)).astype(np.float64)).astype(np.float32)
    return linear_row(t_lin2, h)


def timestep_mods(t, t_lin1, t_lin2, modulation, norm_out):
    """(mods [4 dim] raw [s1|g1|s2|g2], final_scale [dim]) of one timestep:
    both read s = silu(temb) (qwen_image21.rs, Qi21Dit::mods)."""
    s = silu(timestep_embed(t, t_lin1, t_lin2).astype(np.float64)).astype(np.float32)
    return linear_row(modulation, s), linear_row(norm_out, s)


# ----------------------------------------------------------------- FP8 ----
# A generic W8A8 variant of the four projections. The pages' device weights
# are 8- and 4-bit codecs whose formats they do not give, so this variant
# uses the OCP FP8 E4M3 format: every activation row and every weight row
# (output channel) is scaled by a power of two so that its largest
# magnitude fits 448, rounded to the nearest E4M3 value (ties to even,
# saturating), multiplied as codes with wide accumulation, and the two
# scales applied to the product. Powers of two keep scaling exact, so the
# rounding decision depends only on the value being quantised.

E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte (OCP FP8): sign bit 7, exponent bits 3..6
    with bias 7, mantissa bits 0..2; exponent 0 is subnormal (m 2^-9);
    0x7F / 0xFF are NaN, there is no infinity."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_grid():
    """(values, codes) of the 127 finite non-negative E4M3 values, in
    increasing order (codes 0x00 .. 0x7E)."""
    codes = np.arange(0x7F, dtype=np.int64)
    vals = np.array([e4m3_value(c) for c in codes], dtype=np.float64)
    return vals, codes


_E4M3_VALS, _E4M3_CODES = e4m3_grid()


def round_e4m3(a):
    """Round to the nearest E4M3 value, ties to the even code, magnitudes
    beyond 448 saturating to 448 (the satfinite conversion)."""
    a = np.asarray(a, dtype=np.float64)
    m = np.minimum(np.abs(a), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_VALS, m, side="left"), 1, len(_E4M3_VALS) - 1)
    lo = hi - 1
    vlo, vhi = _E4M3_VALS[lo], _E4M3_VALS[hi]
    dlo, dhi = m - vlo, vhi - m
    take_hi = (dhi < dlo) | ((dhi == dlo) & (_E4M3_CODES[hi] % 2 == 0))
    r = np.where(take_hi, vhi, vlo)
    r = np.where(m == 0.0, 0.0, r)
    return np.copysign(r, a)


def pow2_exp(amax):
    """Smallest integer e with amax <= 448 2^e (0 for amax = 0), from the
    binary exponent of amax: amax = f 2^p with f in [0.5, 1) and
    448 = 0.875 2^9."""
    amax = np.asarray(amax, dtype=np.float64)
    f, p = np.frexp(amax)
    e = np.where(f <= 0.875, p - 9, p - 8)
    return np.where(amax == 0.0, 0, e).astype(np.int64)


def quantize_rows(a):
    """(q, e): per row e = pow2_exp(max |a_row|) and q = round_e4m3(a 2^-e)
    (E4M3 values as floats)."""
    a = np.asarray(a, dtype=np.float64)
    e = pow2_exp(np.max(np.abs(a), axis=-1))
    q = round_e4m3(a * np.ldexp(1.0, -e)[..., None])
    return q, e


def linear_fp8(a, w):
    """a W^T with both operands quantised row-wise (activation rows, weight
    output channels): (q_a q_w^T) 2^(e_a + e_w)."""
    qa, ea = quantize_rows(a)
    qw, ew = quantize_rows(np.asarray(w, dtype=np.float64))
    return (qa @ qw.T) * np.ldexp(1.0, ea[:, None] + ew[None, :])


def mods_dev(mods, h):
    """[s1 | tanh g1 | s2 | tanh g2]: the gate chunks tanh-ed in f32, the
    scale chunks as they are (qi21.rs, mods_dev)."""
    m = np.asarray(mods, dtype=np.float32)[:4 * h].copy()
    m[h:2 * h] = np.tanh(m[h:2 * h])
    m[3 * h:4 * h] = np.tanh(m[3 * h:4 * h])
    return m


# ------------------------------------------------------------- FLOP count --

def step_flops(dim, mlp_hidden, layers, n_rows, visible_sum):
    """Algorithmic work of one pass: GEMM flops 2 M (4 H^2 + 3 H I) per
    layer plus attention 4 H sum_i visible(i) per layer (QK^T and PV over all
    heads). Returns (gemm_flops, attn_flops)."""
    g = 2.0 * n_rows * (4 * dim * dim + 3 * dim * mlp_hidden) * layers
    a = 4.0 * dim * float(visible_sum) * layers
    return g, a
