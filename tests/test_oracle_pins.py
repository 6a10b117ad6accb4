"""Pins of the CPU oracle against what the pages and the mathematics fix:
the page's own worked examples (tests/golden/), closed forms, brute force on
tiny inputs and invariants. No GPU."""
import json
import math
import os

import numpy as np
import pytest
from scipy import special as sp_special

from oracle import qi21_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _tiny_cfg(dim=8, heads=2, head_dim=4, axes=(2, 0, 2)):
    return {"dim": dim, "heads": heads, "head_dim": head_dim, "eps": 1e-6, "axes": axes, "theta": 10000.0}


def _rand_layer(rng, H, I, hd):
    return {
        "wq": rng.standard_normal((H, H)) / math.sqrt(H),
        "wk": rng.standard_normal((H, H)) / math.sqrt(H),
        "wv": rng.standard_normal((H, H)) / math.sqrt(H),
        "wo": rng.standard_normal((H, H)) / math.sqrt(H),
        "wgate": rng.standard_normal((I, H)) / math.sqrt(H),
        "wup": rng.standard_normal((I, H)) / math.sqrt(H),
        "wdown": rng.standard_normal((H, I)) / math.sqrt(I),
        "norm_q": 1.0 + 0.05 * rng.standard_normal(hd),
        "norm_k": 1.0 + 0.05 * rng.standard_normal(hd),
    }


# ------------------------------------------------------------ layout pins --

def test_positions_worked_examples():
    g = _golden("layout_examples.json")
    for case in g["cases"]:
        segs = [tuple(s) for s in case["segs"]]
        p = O.positions(segs)
        for r, want in case["positions"].items():
            assert p[int(r)].tolist() == want, (segs, r)
        for r, want in case.get("positions_frame", {}).items():
            assert p[int(r)][0] == want
        if "prefix_len" in case:
            assert O.prefix_len(segs) == case["prefix_len"]
        if "block_ids" in case:
            assert O.block_ids(segs).tolist() == case["block_ids"]


def test_positions_brute_force_rule():
    # A direct re-derivation from the rule: frame = running position, image
    # coordinates centred so that row h//2 ... sits at 0 - (h - h//2) + h//2.
    segs = [(0, 4, 0), (1, 5, 3), (0, 2, 0), (1, 2, 6), (1, 1, 1)]
    p = O.positions(segs)
    assert p.shape == (4 + 15 + 2 + 12 + 1, 3)
    # text rows 0..3 at [i, i, i]
    assert p[:4].tolist() == [[i, i, i] for i in range(4)]
    img = p[4:19]
    assert set(img[:, 0].tolist()) == {4}
    assert sorted(set(img[:, 1].tolist())) == [-3, -2, -1, 0, 1]  # h=5: r - 3
    assert sorted(set(img[:, 2].tolist())) == [-2, -1, 0]  # w=3: c - 2
    assert img[0].tolist() == [4, -3, -2] and img[1].tolist() == [4, -3, -1]  # raster order
    # next text resumes at 4 + max(5, 3) = 9
    assert p[19].tolist() == [9, 9, 9] and p[20].tolist() == [10, 10, 10]
    # Image(2,6) at frame 11, then Image(1,1) at 11 + 6 = 17
    assert p[21].tolist() == [11, -1, -3]
    assert p[-1].tolist() == [17, -1, -1]


def test_prefix_visibility_hand_cases():
    # condition-image prefix of the 32-layer workload: Text(18) + Image(64,64)
    segs = [(0, 18, 0), (1, 64, 64), (1, 64, 64)]
    vis = O.prefix_visibility(segs)
    assert len(vis) == 18 + 4096
    assert vis[:18].tolist() == list(range(1, 19))
    assert (vis[18:] == 4114).all()
    # mixed: Text5, Image(4,6), Text3, Image(3,2) | target
    segs = [(0, 5, 0), (1, 4, 6), (0, 3, 0), (1, 3, 2), (1, 2, 2)]
    vis = O.prefix_visibility(segs).tolist()
    assert vis == [1, 2, 3, 4, 5] + [29] * 24 + [30, 31, 32] + [38] * 6
    v = np.array(vis)
    assert (np.diff(v) >= 0).all() and v.min() >= 1 and v.max() <= len(vis)


def test_validate_rejects_bad_layouts():
    with pytest.raises(ValueError):
        O.validate([(0, 3, 0)])  # no target image
    with pytest.raises(ValueError):
        O.validate([(1, 2, 2)])  # empty prefix
    with pytest.raises(ValueError):
        O.validate([(0, 3, 0), (1, 0, 4)])  # empty target
    O.validate([(0, 1, 0), (1, 1, 1)])


# -------------------------------------------------------------- RoPE pins --

def test_rope_tables_unit_rotations_and_identity():
    # the page's own test: t2i(4, 2, 2) -> rows*64 entries, unit rotations,
    # position 0 -> identity
    segs = [(0, 4, 0), (1, 2, 2)]
    c, s = O.rope_tables(O.positions(segs), (16, 56, 56), 10000.0)
    assert c.size == O.total_rows(segs) * 64
    assert np.all(np.abs(c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2 - 1.0) < 1e-5)
    assert np.all(np.abs(c[0] - 1.0) < 1e-7)


def test_rope_tables_closed_form():
    # angle of pair j: frame axis for j < 8, h axis for 8 <= j < 36, w axis
    # after; frequency theta^(-2i/d) of the axis width d.
    pos = np.array([[0, 0, 0], [3, -1, -2], [82, 31, -32], [17, 5, 9]])
    c, s = O.rope_tables(pos, (16, 56, 56), 10000.0)
    for r, p in enumerate(pos):
        for j in range(64):
            if j < 8:
                ang = p[0] * 10000.0 ** (-2 * j / 16)
            elif j < 36:
                ang = p[1] * 10000.0 ** (-2 * (j - 8) / 56)
            else:
                ang = p[2] * 10000.0 ** (-2 * (j - 36) / 56)
            # f32 frequency and angle: |err| <= a few ulp of the angle
            tol = 4e-7 * max(1.0, abs(ang)) + 2e-7
            assert abs(c[r, j] - math.cos(ang)) < tol, (r, j)
            assert abs(s[r, j] - math.sin(ang)) < tol, (r, j)


def test_rope_rotation_sign_and_pairing():
    # rotating e_{2j} by angle a gives cos a at 2j and sin a at 2j+1
    hd = 8
    ang = np.array([[0.3, -1.1, 2.0, 0.7]])
    cos, sin = np.cos(ang), np.sin(ang)
    for j in range(4):
        v = np.zeros((1, 1, hd))
        v[0, 0, 2 * j] = 1.0
        out = O.rope_rotate(v, cos, sin)[0, 0]
        want = np.zeros(hd)
        want[2 * j] = math.cos(ang[0, j])
        want[2 * j + 1] = math.sin(ang[0, j])
        np.testing.assert_allclose(out, want, atol=1e-15)


def test_rope_norm_preservation():
    rng = np.random.default_rng(1)
    segs = [(0, 18, 0), (1, 8, 8)]
    c, s = O.rope_tables(O.positions(segs), (16, 56, 56), 10000.0)
    v = rng.standard_normal((c.shape[0], 3, 128))
    out = O.rope_rotate(v, c, s)
    n0 = np.linalg.norm(v, axis=-1)
    n1 = np.linalg.norm(out, axis=-1)
    # the f32 tables are unit rotations within 1e-5 (relative norm change
    # is bounded by half of that)
    assert np.max(np.abs(n1 / n0 - 1.0)) < 1e-6 * 10


# -------------------------------------------------------------- norm pins --

def test_layer_norm_closed_form():
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    eps = 1e-6
    want = (x - 2.5) / math.sqrt(1.25 + eps)
    np.testing.assert_allclose(O.layer_norm(x, eps), want, rtol=0, atol=1e-15)
    # modulated: LN(x)(1 + s)
    s = np.array([0.5, -1.0, 0.0, 2.0])
    np.testing.assert_allclose(O.norm_mod(x, s, eps), want * (1 + s), atol=1e-15)
    rng = np.random.default_rng(0)
    y = O.layer_norm(rng.standard_normal((5, 300)) * 3 + 7, 1e-6)
    assert np.max(np.abs(y.mean(axis=1))) < 1e-12
    assert np.max(np.abs(y.var(axis=1) - 1.0)) < 1e-5


def test_rms_norm_closed_form():
    v = np.array([[3.0, 4.0]])
    w = np.array([1.0, 2.0])
    r = math.sqrt(12.5 + 1e-6)
    np.testing.assert_allclose(O.rms_norm(v, w, 1e-6), [[3 / r, 8 / r]], atol=1e-15)
    # weight used as is (not 1 + w): w = 0 gives 0
    assert np.all(O.rms_norm(v, np.zeros(2), 1e-6) == 0)


def test_silu_and_mods_dev_example():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(30.0) - 30.0) < 1e-10
    assert abs(O.silu(-30.0)) < 1e-10
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    g = _golden("mods_dev_example.json")
    m = np.array(g["mods"], dtype=np.float32)
    d = O.mods_dev(m, g["h"])
    for i in g["unchanged"]:
        assert d[i] == m[i]
    for i, v in g["tanh_of"].items():
        assert d[int(i)] == np.tanh(np.float32(v))


# --------------------------------------------------------- attention pins --

def _brute_attention(q, k, v, visible, heads, hd):
    n, m = q.shape[0], k.shape[0]
    out = np.zeros((n, heads * hd))
    for h in range(heads):
        for i in range(n):
            sc = []
            for j in range(visible[i]):
                dot = 0.0
                for d in range(hd):
                    dot += (q[i, h * hd + d] / math.sqrt(hd)) * k[j, h * hd + d]
                sc.append(dot)
            mx = max(sc)
            e = [math.exp(x - mx) for x in sc]
            den = math.fsum(e)
            for d in range(hd):
                out[i, h * hd + d] = math.fsum(e[j] * v[j, h * hd + d] for j in range(visible[i])) / den
    return out


def test_attention_brute_force():
    rng = np.random.default_rng(3)
    heads, hd = 2, 16
    n, m = 6, 11
    q = rng.standard_normal((n, heads * hd))
    k = rng.standard_normal((m, heads * hd))
    v = rng.standard_normal((m, heads * hd))
    visible = [1, 3, 3, 7, 11, 11]
    got = O.attention(q, k, v, visible, heads, hd)
    want = _brute_attention(q, k, v, visible, heads, hd)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_masked_softmax_rows_and_zeros():
    rng = np.random.default_rng(4)
    s = rng.standard_normal((5, 9)) * 5
    vis = [1, 2, 5, 9, 9]
    p = O.masked_softmax(s, vis)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-12
    for i, vv in enumerate(vis):
        assert np.all(p[i, vv:] == 0.0)
        assert np.all(p[i, :vv] > 0.0)


def test_attention_special_cases():
    rng = np.random.default_rng(5)
    heads, hd = 2, 8
    k = np.tile(rng.standard_normal((1, heads * hd)), (7, 1))  # all keys equal
    v = rng.standard_normal((7, heads * hd))
    q = rng.standard_normal((3, heads * hd))
    vis = [2, 5, 7]
    o = O.attention(q, k, v, vis, heads, hd)
    for i, vv in enumerate(vis):
        np.testing.assert_allclose(o[i], v[:vv].mean(axis=0), atol=1e-13)
    o1 = O.attention(q, rng.standard_normal((7, heads * hd)), v, [1, 1, 1], heads, hd)
    for i in range(3):
        np.testing.assert_allclose(o1[i], v[0], atol=1e-15)


# -------------------------------------------------------------- block pins --

def test_block_identity_when_gates_are_zero():
    rng = np.random.default_rng(6)
    cfg = _tiny_cfg()
    H, I = 8, 12
    W = _rand_layer(rng, H, I, cfg["head_dim"])
    x = rng.standard_normal((5, H)).astype(np.float32)
    mods = rng.standard_normal(4 * H) * 0.1
    mods[H:2 * H] = 0.0
    mods[3 * H:] = -0.0
    pos = np.array([[i, i, i] for i in range(5)])
    c, s = O.rope_tables(pos, cfg["axes"], cfg["theta"])
    out, _, _ = O.block(x, W, mods, c, s, cfg)
    assert np.array_equal(out, x.astype(np.float64))


def test_block_closed_form_zero_qk():
    # Wq = Wk = 0: q = k = 0 after RMSNorm, every visible score is 0, so the
    # attention averages the visible values. Wgate = 0 makes silu(0) = 0 and
    # the FFN adds nothing. Written out with explicit loops (nn.Linear: out_r
    # = sum_c W[r, c] in_c).
    rng = np.random.default_rng(7)
    cfg = _tiny_cfg()
    H, I = 8, 12
    W = _rand_layer(rng, H, I, cfg["head_dim"])
    W["wq"][:] = 0
    W["wk"][:] = 0
    W["wgate"][:] = 0
    x = rng.standard_normal((6, H))
    mods = rng.standard_normal(4 * H) * 0.5
    vis = [1, 2, 2, 4, 6, 6]
    pos = np.array([[i, i, i] for i in range(6)])
    c, s = O.rope_tables(pos, cfg["axes"], cfg["theta"])
    out, k, _ = O.block(x, W, mods, c, s, cfg, None, vis)
    assert np.all(k == 0)
    eps = cfg["eps"]
    s1, g1 = mods[:H], mods[H:2 * H]
    xn = []
    for r in range(6):
        mu = math.fsum(x[r]) / H
        var = math.fsum((x[r, c_] - mu) ** 2 for c_ in range(H)) / H
        xn.append([(x[r, c_] - mu) / math.sqrt(var + eps) * (1 + s1[c_]) for c_ in range(H)])
    vrow = [[math.fsum(W["wv"][o, c_] * xn[r][c_] for c_ in range(H)) for o in range(H)] for r in range(6)]
    for i in range(6):
        ob = [math.fsum(vrow[j][o] for j in range(vis[i])) / vis[i] for o in range(H)]
        for o in range(H):
            proj = math.fsum(W["wo"][o, c_] * ob[c_] for c_ in range(H))
            want = x[i, o] + math.tanh(g1[o]) * proj
            assert abs(out[i, o] - want) < 1e-12, (i, o)


def test_block_closed_form_ffn_only():
    # Wv = 0: the attention output is 0 and the block is the FFN residual
    # x + tanh(g2) Wd (silu(Wg xn2) * (Wu xn2)) with xn2 = LN(x)(1 + s2).
    rng = np.random.default_rng(8)
    cfg = _tiny_cfg()
    H, I = 8, 12
    W = _rand_layer(rng, H, I, cfg["head_dim"])
    W["wv"][:] = 0
    x = rng.standard_normal((3, H))
    mods = rng.standard_normal(4 * H) * 0.5
    pos = np.array([[i, i, i] for i in range(3)])
    c, s = O.rope_tables(pos, cfg["axes"], cfg["theta"])
    out, _, _ = O.block(x, W, mods, c, s, cfg)
    eps = cfg["eps"]
    s2, g2 = mods[2 * H:3 * H], mods[3 * H:]
    for r in range(3):
        mu = math.fsum(x[r]) / H
        var = math.fsum((x[r, c_] - mu) ** 2 for c_ in range(H)) / H
        xn = [(x[r, c_] - mu) / math.sqrt(var + eps) * (1 + s2[c_]) for c_ in range(H)]
        gt = [math.fsum(W["wgate"][o, c_] * xn[c_] for c_ in range(H)) for o in range(I)]
        up = [math.fsum(W["wup"][o, c_] * xn[c_] for c_ in range(H)) for o in range(I)]
        hid = [gt[o] / (1 + math.exp(-gt[o])) * up[o] for o in range(I)]
        for o in range(H):
            d = math.fsum(W["wdown"][o, c_] * hid[c_] for c_ in range(I))
            assert abs(out[r, o] - (x[r, o] + math.tanh(g2[o]) * d)) < 1e-12


def test_block_qk_path_against_explicit_loops():
    # q/k path: RMSNorm * w then RoPE, checked element by element on one
    # row against a loop restatement (catches a wrong pair order or sign).
    rng = np.random.default_rng(9)
    heads, hd = 2, 8
    t = rng.standard_normal((2, heads * hd))
    w = 1 + 0.1 * rng.standard_normal(hd)
    ang = rng.standard_normal((2, hd // 2))
    cos, sin = np.cos(ang), np.sin(ang)
    got = O.qk_norm_rope(t, w, cos, sin, heads, hd, 1e-6)
    for r in range(2):
        for h in range(heads):
            v = t[r, h * hd:(h + 1) * hd]
            inv = 1 / math.sqrt(math.fsum(a * a for a in v) / hd + 1e-6)
            u = [v[d] * inv * w[d] for d in range(hd)]
            for j in range(hd // 2):
                a, b = u[2 * j], u[2 * j + 1]
                assert abs(got[r, h * hd + 2 * j] - (a * cos[r, j] - b * sin[r, j])) < 1e-13
                assert abs(got[r, h * hd + 2 * j + 1] - (a * sin[r, j] + b * cos[r, j])) < 1e-13


def test_block_row_subset_equals_full():
    rng = np.random.default_rng(10)
    cfg = _tiny_cfg(dim=16, heads=2, head_dim=8, axes=(2, 2, 4))
    H, I = 16, 24
    W = _rand_layer(rng, H, I, 8)
    x = rng.standard_normal((9, H))
    mods = rng.standard_normal(4 * H) * 0.2
    segs = [(0, 3, 0), (1, 3, 3)]
    c, s = O.rope_tables(O.positions(segs)[3:], cfg["axes"], cfg["theta"])
    kvp = (rng.standard_normal((3, H)), rng.standard_normal((3, H)))
    full, k, v = O.block(x, W, mods, c, s, cfg, kvp, None)
    rows = [0, 4, 8]
    sub, k2, v2 = O.block(x, W, mods, c, s, cfg, kvp, None, rows=rows)
    np.testing.assert_allclose(sub, full[rows], rtol=0, atol=1e-13)
    np.testing.assert_array_equal(k, k2)


@pytest.mark.parametrize("segs", [
    [(0, 4, 0), (1, 3, 3)],
    [(0, 3, 0), (1, 2, 3), (0, 2, 0), (1, 4, 2)],
])
def test_prefill_plus_step_equals_joint_forward(segs):
    # The prefix never attends to the target and never sees t, so running
    # the prefix once (keeping K/V) and the target against the cache equals
    # the joint forward under the block-causal mask on the target rows.
    rng = np.random.default_rng(11)
    cfg = _tiny_cfg(dim=16, heads=2, head_dim=8, axes=(2, 2, 4))
    H, I = 16, 24
    layers = [_rand_layer(rng, H, I, 8) for _ in range(3)]
    lp = O.prefix_len(segs)
    n = O.seg_len(segs[-1])
    xp = rng.standard_normal((lp, H))
    xt = rng.standard_normal((n, H))
    m0 = rng.standard_normal(4 * H) * 0.3
    mt = rng.standard_normal(4 * H) * 0.3
    cache, _ = O.prefill(xp, layers, m0, segs, cfg)
    got, _ = O.step(xt, layers, mt, segs, cache, cfg)
    want = O.joint_forward(xp, xt, layers, m0, mt, segs, cfg)
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel < 1e-12


def test_flop_accounting_reproduces_measured_classes():
    g = _golden("measured_classes_1024.json")
    n, lp, L, H, I = g["rows"], g["prefix"], g["layers"], g["dim"], g["mlp_hidden"]
    c = g["classes"]
    flops = {
        "qkv": 2 * n * 3 * H * H * L,
        "o": 2 * n * H * H * L,
        "gateup": 2 * n * 2 * H * I * L,
        "down": 2 * n * H * I * L,
        "flash": 4 * H * n * (lp + n) * L,
    }
    for k, f in flops.items():
        tf = f / (c[k]["ms"] * 1e-3) / 1e12
        assert abs(tf - c[k]["tflops"]) < 1.0, (k, tf)
    gemm, attn = O.step_flops(H, I, L, n, n * (lp + n))
    assert gemm == sum(flops[k] for k in ("qkv", "o", "gateup", "down"))
    assert attn == flops["flash"]


# ------------------------------------------------------ embed / final pins --

def test_embed_image_closed_form():
    # nn.Linear layout: x[r][c] = sum_k tok[r][k] W[c][k]
    tok = np.array([[1.0, 2.0, 0.0], [0.0, -1.0, 3.0]])
    W = np.array([[1.0, 0.0, 0.0], [0.0, 1.0, 0.0], [1.0, 1.0, 1.0], [2.0, 0.0, -1.0]])
    want = np.array([[1.0, 2.0, 3.0, 2.0], [0.0, -1.0, 2.0, -3.0]])
    np.testing.assert_array_equal(O.embed_image(tok, W), want)


def test_final_layer_closed_form_and_constant_rows():
    eps = 1e-6
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    fs = np.array([0.5, -1.0, 0.0, 1.0])
    W = np.array([[1.0, 1.0, 1.0, 1.0], [0.0, 0.0, 0.0, 2.0]])
    ln = (x[0] - 2.5) / math.sqrt(1.25 + eps)
    xn = ln * (1.0 + fs)
    want = [[xn.sum(), 2.0 * xn[3]]]
    np.testing.assert_allclose(O.final_layer(x, fs, W, eps), want, atol=1e-14)
    # a constant row normalises to zero whatever the scale and weight
    c = np.full((2, 8), 3.25)
    rng = np.random.default_rng(12)
    assert np.all(O.final_layer(c, rng.standard_normal(8), rng.standard_normal((5, 8)), eps) == 0.0)


def test_denoise_composes_embed_step_final():
    rng = np.random.default_rng(13)
    cfg = _tiny_cfg(dim=16, heads=2, head_dim=8, axes=(2, 2, 4))
    H, I, C = 16, 24, 5
    layers = [_rand_layer(rng, H, I, 8) for _ in range(2)]
    segs = [(0, 3, 0), (1, 2, 3)]
    lp, n = O.prefix_len(segs), O.seg_len(segs[-1])
    tok = rng.standard_normal((n, C))
    w_in = rng.standard_normal((H, C))
    w_out = rng.standard_normal((C, H))
    fsc = rng.standard_normal(H) * 0.1
    m0, mt = rng.standard_normal(4 * H) * 0.2, rng.standard_normal(4 * H) * 0.2
    cache, _ = O.prefill(rng.standard_normal((lp, H)), layers, m0, segs, cfg)
    got = O.denoise(tok, w_in, layers, mt, fsc, w_out, segs, cache, cfg)
    x = tok @ w_in.T
    for l, W in enumerate(layers):
        x, _, _ = O.block(x, W, mt, *O.target_rope(segs, cfg["axes"], cfg["theta"]), cfg, cache[l], None)
    want = O.layer_norm(x, cfg["eps"]) * (1 + fsc) @ w_out.T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------- timestep pins --
# qwen_image21.rs, Qi21Dit::temb / Qi21Dit::mods.

def test_timestep_sinusoid_at_zero_and_closed_form():
    # t = 0: every angle is 0, so the cos half is 1 and the sin half 0 exactly
    e0 = O.timestep_sinusoid(0.0)
    assert e0.shape == (256,) and e0.dtype == np.float32
    np.testing.assert_array_equal(e0, np.r_[np.ones(128), np.zeros(128)].astype(np.float32))
    # t = 0.001 gives 1000 t = 1: frequency i is 10000^(-i/128), a geometric
    # ladder from 1 down to 10000^(-127/128); cos first, then sin
    e = O.timestep_sinusoid(0.001).astype(np.float64)
    f = np.array([10000.0 ** (-i / 128.0) for i in range(128)])
    np.testing.assert_allclose(e[:128], np.cos(f), atol=2e-6)
    np.testing.assert_allclose(e[128:], np.sin(f), atol=2e-6)
    assert abs(e[0] - 0.5403023058681398) < 1e-6 and abs(e[128] - 0.8414709848078965) < 1e-6
    # the unit circle, per frequency, at any t
    for t in (0.0, 0.37, 1.0):
        v = O.timestep_sinusoid(t).astype(np.float64)
        np.testing.assert_allclose(v[:128] ** 2 + v[128:] ** 2, 1.0, atol=1e-6)
    # at t = 1 the slowest frequency is 10000^(-127/128) (angle ~0.1075 rad)
    v = O.timestep_sinusoid(1.0).astype(np.float64)
    a = 1000.0 * 10000.0 ** (-127 / 128)
    assert abs(v[127] - np.cos(a)) < 1e-5 and abs(v[255] - np.sin(a)) < 1e-5


def _perm(n, seed):
    p = np.random.default_rng(seed).permutation(n)
    m = np.zeros((n, n), np.float32)
    m[np.arange(n), p] = 1.0
    return m, p


def _silu_ref(v):
    v = np.asarray(v, np.float64)
    return v * sp_special.expit(v)


def test_timestep_mods_through_permutations():
    # with permutation weights every linear is a gather, so the result has a
    # closed form: mods chunk c = (c + 1) silu(silu(silu(e)[p1])[p2])[p3]
    # where the weights pick columns p; a transposed weight would apply the
    # inverse permutation and fail
    dim = 256
    P1, p1 = _perm(dim, 1)
    P2, p2 = _perm(dim, 2)
    P3, p3 = _perm(dim, 3)
    mod = np.concatenate([(c + 1) * P3 for c in range(4)]).astype(np.float32)
    nout = (-2.0 * P2).astype(np.float32)
    t = 0.731
    e = O.timestep_sinusoid(t).astype(np.float64)
    temb = _silu_ref(e[p1])[p2]
    s = _silu_ref(temb)
    mods, fs = O.timestep_mods(t, P1, P2, mod, nout)
    np.testing.assert_allclose(O.timestep_embed(t, P1, P2), temb, rtol=1e-6, atol=1e-7)
    for c in range(4):
        np.testing.assert_allclose(mods[c * dim:(c + 1) * dim], (c + 1) * s[p3], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(fs, -2.0 * s[p2], rtol=1e-6, atol=1e-7)


def test_timestep_mods_brute_force_tiny():
    # dim 4: plain Python sums over the 256 sinusoid channels
    rng = np.random.default_rng(5)
    dim = 4
    W1 = rng.standard_normal((dim, 256)).astype(np.float32) / 16
    W2 = rng.standard_normal((dim, dim)).astype(np.float32)
    Wm = rng.standard_normal((4 * dim, dim)).astype(np.float32)
    Wn = rng.standard_normal((dim, dim)).astype(np.float32)
    t = 0.25
    e = [float(v) for v in O.timestep_sinusoid(t)]
    sl = lambda v: v / (1.0 + math.exp(-v))
    h = [sl(math.fsum(float(W1[r, k]) * e[k] for k in range(256))) for r in range(dim)]
    temb = [math.fsum(float(W2[r, k]) * h[k] for k in range(dim)) for r in range(dim)]
    s = [sl(v) for v in temb]
    mods = [math.fsum(float(Wm[r, k]) * s[k] for k in range(dim)) for r in range(4 * dim)]
    fs = [math.fsum(float(Wn[r, k]) * s[k] for k in range(dim)) for r in range(dim)]
    got_m, got_f = O.timestep_mods(t, W1, W2, Wm, Wn)
    np.testing.assert_allclose(got_m, mods, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(got_f, fs, rtol=1e-5, atol=1e-6)


# ------------------------------------------------------------ FP8 pins ----
# OCP FP8 E4M3 (the generic 8-bit variant of the projections).

def test_e4m3_decode_known_codes():
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in known.items():
        assert O.e4m3_value(c) == v, hex(c)
    assert math.isnan(O.e4m3_value(0x7F)) and math.isnan(O.e4m3_value(0xFF))
    vals, codes = O.e4m3_grid()
    assert len(vals) == 127 and np.all(np.diff(vals) > 0) and vals[-1] == 448.0
    # 3 mantissa bits: 8 values per binade above the subnormals
    assert np.sum((vals >= 1.0) & (vals < 2.0)) == 8


def test_round_e4m3_ties_saturation_and_grid():
    vals, _ = O.e4m3_grid()
    # grid values are fixed points, with either sign
    np.testing.assert_array_equal(O.round_e4m3(vals), vals)
    np.testing.assert_array_equal(O.round_e4m3(-vals), -vals)
    # ties go to the even code: 1.0625 between 1.0 (0x38) and 1.125 (0x39)
    assert O.round_e4m3(1.0625) == 1.0
    # 1.1875 between 1.125 (0x39) and 1.25 (0x3A)
    assert O.round_e4m3(1.1875) == 1.25
    # 2^-10 is halfway between 0 and the smallest subnormal 2^-9
    assert O.round_e4m3(2.0 ** -10) == 0.0
    assert O.round_e4m3(2.0 ** -10 * 1.0001) == 2.0 ** -9
    # off a tie, the nearer neighbour
    assert O.round_e4m3(1.0624) == 1.0 and O.round_e4m3(1.0626) == 1.125
    # saturation (no infinity): everything beyond 448 clamps to 448
    np.testing.assert_array_equal(O.round_e4m3([449.0, 464.0, 1e9, -1e9]), [448.0, 448.0, 448.0, -448.0])
    # the result is always a grid value and the nearest one
    rng = np.random.default_rng(0)
    a = rng.standard_normal(20000) * np.exp2(rng.uniform(-12, 9, 20000))
    r = O.round_e4m3(a)
    assert np.all(np.isin(np.abs(r), vals))
    best = np.min(np.abs(np.abs(a)[:, None] - vals[None, :]), axis=1)
    inside = np.abs(a) <= 448.0
    np.testing.assert_allclose(np.abs(np.abs(r) - np.abs(a))[inside], best[inside], rtol=0, atol=0)


def test_pow2_exp_minimal():
    assert O.pow2_exp(448.0) == 0 and O.pow2_exp(448.0000001) == 1
    assert O.pow2_exp(224.0) == -1 and O.pow2_exp(1.0) == -8 and O.pow2_exp(0.0) == 0
    rng = np.random.default_rng(1)
    a = np.exp2(rng.uniform(-20, 20, 5000))
    e = O.pow2_exp(a)
    assert np.all(a <= 448.0 * np.exp2(e)) and np.all(a > 448.0 * np.exp2(e - 1.0))


def test_linear_fp8_exact_on_grid_and_error_bound():
    rng = np.random.default_rng(2)
    vals, _ = O.e4m3_grid()
    # rows already on the grid, each with one element at 448: no rounding,
    # scale 1, so the product is the plain one
    a = rng.choice(vals, size=(5, 33)) * rng.choice([-1.0, 1.0], size=(5, 33))
    w = rng.choice(vals, size=(7, 33)) * rng.choice([-1.0, 1.0], size=(7, 33))
    a[:, 0] = 448.0
    w[:, 3] = -448.0
    np.testing.assert_array_equal(O.linear_fp8(a, w), a @ w.T)
    # scaling by powers of two commutes with quantisation
    np.testing.assert_array_equal(O.linear_fp8(a * 8.0, w / 4.0), (a @ w.T) * 2.0)
    # generic inputs: every element within half a grid step (relative 2^-4)
    x = rng.standard_normal((16, 64))
    q, e = O.quantize_rows(x)
    deq = q * np.exp2(e)[:, None]
    big = np.abs(x) >= 2.0 ** -6 * np.exp2(e)[:, None]
    assert np.all(np.abs(deq - x)[big] <= np.abs(x)[big] * 2.0 ** -4 + 1e-300)
