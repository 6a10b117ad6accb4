"""Per-operation parity of the CUDA kernels against the CPU oracle, through
the library's single-operation entry points (qi21_op_*). Inputs are seeded
(synthetic.qi21_inputs.op_tensor); expected values come from oracle/ only.

Tolerances (derived from the arithmetic, f16 unit roundoff u = 2^-11):
  - f16 outputs: |gpu - ref| <= 2u |ref| + atol, atol a few u of the
    output scale (one rounding of the stored value plus f32 arithmetic);
  - f32 GEMM outputs: rel L2 <= 1e-5 (f32 accumulation of K products);
  - attention: rel L2 <= 2e-3 (P rounded to f16 before P V, f32 sums).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from oracle import qi21_oracle as O  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu

U16 = 2.0 ** -11


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert q.device_status() == 0, "a kernel gave up waiting"


# ------------------------------------------------------------------ rows ----

def test_mods_prep():
    for case, dim in enumerate([256, 4096]):
        m = S.op_tensor(1, case, 0, (4 * dim,), 0.5)
        md = torch.empty(4 * dim, dtype=torch.float32, device="cuda")
        q.op_mods_prep(T(m), md)
        np.testing.assert_allclose(host(md), O.mods_dev(m, dim), rtol=0, atol=2e-7)


# row counts above the resident CTA count make each CTA walk several rows
@pytest.mark.parametrize("rows,dim", [(1, 128), (130, 512), (37, 4096), (3, 8192), (0, 256), (2000, 4096),
                                      (700, 8192), (4099, 1024)])
def test_rowop_norm(rows, dim):
    x = S.op_tensor(2, dim, 0, (rows, dim), 3.0, offset=0.5)
    sc = S.op_tensor(2, dim, 1, (dim,), 0.1)
    xd = T(x)
    xn = torch.empty((rows, dim), dtype=torch.float16, device="cuda")
    q.op_rowop(xd, T(sc), xn=xn)
    if rows == 0:
        return
    ref = O.norm_mod(x, sc, 1e-6)
    got = host(xn).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * U16 * np.abs(ref) + 4 * U16)
    np.testing.assert_array_equal(host(xd), x)  # x untouched without y


@pytest.mark.parametrize("rows,dim", [(5, 256), (64, 4096), (1500, 4096)])
def test_rowop_gate_and_norm(rows, dim):
    x = S.op_tensor(3, dim, 0, (rows, dim), 1.0)
    y = S.op_tensor(3, dim, 1, (rows, dim), 1.0)
    gt = np.tanh(S.op_tensor(3, dim, 2, (dim,), 0.3))
    sc = S.op_tensor(3, dim, 3, (dim,), 0.1)
    xd = T(x)
    xn = torch.empty((rows, dim), dtype=torch.float16, device="cuda")
    q.op_rowop(xd, T(sc), xn=xn, y=T(y), gate_t=T(gt))
    x1 = O.gated_add(x, y, np.arctanh(gt.astype(np.float64)))
    np.testing.assert_allclose(host(xd), x1, rtol=1e-6, atol=1e-6)
    ref = O.norm_mod(x1, sc, 1e-6)
    got = host(xn).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * U16 * np.abs(ref) + 4 * U16)


@pytest.mark.parametrize("rows,heads", [(1, 1), (33, 2), (300, 32)])
def test_qkrope(rows, heads):
    H = heads * 128
    panel = S.op_tensor(4, rows * heads, 0, (rows, 3 * H), 2.0).astype(np.float16)
    nq = S.op_tensor(4, rows * heads, 1, (128,), 0.05, offset=1.0)
    nk = S.op_tensor(4, rows * heads, 2, (128,), 0.05, offset=1.0)
    segs = [(0, 7, 0), (1, 9, 11), (1, rows, 1)]
    pos = O.positions(segs)[-rows:]
    cs, sn = O.rope_tables(pos)
    pd = T(panel)
    q.op_qkrope(pd, heads, T(nq), T(nk), T(cs), T(sn))
    got = host(pd)
    p64 = panel.astype(np.float64)
    rq = O.qk_norm_rope(p64[:, :H], nq, cs, sn, heads, 128, 1e-6)
    rk = O.qk_norm_rope(p64[:, H:2 * H], nk, cs, sn, heads, 128, 1e-6)
    for g, r in ((got[:, :H], rq), (got[:, H:2 * H], rk)):
        g = g.astype(np.float64)
        assert np.all(np.abs(g - r) <= 2 * U16 * np.abs(r) + 8 * U16)
    np.testing.assert_array_equal(got[:, 2 * H:], panel[:, 2 * H:])  # v untouched


def test_kvcopy_exact():
    rows, H = 77, 512
    panel = S.op_tensor(5, 0, 0, (rows, 3 * H), 1.0).astype(np.float16)
    kv = torch.zeros((rows, 2 * H), dtype=torch.float16, device="cuda")
    q.op_kvcopy(T(panel), kv)
    np.testing.assert_array_equal(host(kv), panel[:, H:])


# ------------------------------------------------------------------ GEMM ----

GEMM_SHAPES = [
    (1, 128, 64), (18, 256, 256), (128, 384, 64), (130, 768, 256), (300, 1536, 512),
    (257, 128, 768), (513, 256, 4096), (4114, 512, 256),
]


def _ab(case, M, N, K):
    A = S.op_tensor(6, case, 0, (M, K), 1.0).astype(np.float16)
    Bw = S.op_tensor(6, case, 1, (N, K), K ** -0.5).astype(np.float16)
    return A, Bw


@pytest.mark.parametrize("shape", GEMM_SHAPES)
def test_gemm_f32_and_f16(shape):
    M, N, K = shape
    A, Bw = _ab(M * 7 + N, M, N, K)
    ref = A.astype(np.float64) @ Bw.astype(np.float64).T
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.op_gemm(q.EPI_F32, T(A), T(Bw), out)
    got = host(out)
    assert rel_l2(got, ref) < 1e-5
    assert np.max(np.abs(got - ref)) < 1e-3
    out16 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    q.op_gemm(q.EPI_F16, T(A), T(Bw), out16)
    g16 = host(out16).astype(np.float64)
    assert np.all(np.abs(g16 - ref) <= U16 * np.abs(ref) + 1e-3)


@pytest.mark.parametrize("shape", [(18, 256, 256), (300, 512, 1536), (129, 4096, 4096)])
def test_gemm_residual_gate(shape):
    M, N, K = shape
    A, Bw = _ab(M + 3 * N, M, N, K)
    x0 = S.op_tensor(7, M, 0, (M, N), 1.0)
    gt = np.tanh(S.op_tensor(7, M, 1, (N,), 0.1))
    xd = T(x0)
    q.op_gemm(q.EPI_RESID, T(A), T(Bw), xd, gate_t=T(gt))
    ref = x0 + gt.astype(np.float64) * (A.astype(np.float64) @ Bw.astype(np.float64).T)
    got = host(xd)
    assert rel_l2(got, ref) < 1e-6
    assert np.max(np.abs(got - ref)) < 1e-4


def _interleave_w13(G, Up):
    """The documented w13 layout: 128-row slices [gate 64 rows | up 64 rows]."""
    I, H = G.shape
    out = np.empty((2 * I, H), G.dtype)
    for j in range(I // 64):
        out[128 * j:128 * j + 64] = G[64 * j:64 * j + 64]
        out[128 * j + 64:128 * j + 128] = Up[64 * j:64 * j + 64]
    return out


@pytest.mark.parametrize("M,I,K", [(18, 192, 256), (130, 768, 256), (300, 1536, 512), (257, 12288, 4096)])
def test_gemm_swiglu(M, I, K):
    A = S.op_tensor(8, M, 0, (M, K), 1.0).astype(np.float16)
    G = S.op_tensor(8, M, 1, (I, K), K ** -0.5).astype(np.float16)
    Up = S.op_tensor(8, M, 2, (I, K), K ** -0.5).astype(np.float16)
    W = _interleave_w13(G, Up)
    out = torch.empty((M, I), dtype=torch.float16, device="cuda")
    q.op_gemm(q.EPI_SWIGLU, T(A), T(W), out)
    a = A.astype(np.float64)
    ref = O.silu(a @ G.astype(np.float64).T) * (a @ Up.astype(np.float64).T)
    got = host(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * U16 * np.abs(ref) + 2e-3)
    assert rel_l2(got, ref) < 1e-3


def test_gemm_full_width_sampled_rows():
    # the qkv projection at full size (M 4096, N 12288, K 4096): sampled
    # rows against f64 dot products
    M, N, K = 4096, 12288, 4096
    A, Bw = _ab(999, M, N, K)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    q.op_gemm(q.EPI_F16, T(A), T(Bw), out)
    rows = np.array([0, 1, 127, 128, 2047, 2048, 4000, 4094, 4095])
    got = out[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    ref = A[rows].astype(np.float64) @ Bw.astype(np.float64).T
    assert np.all(np.abs(got - ref) <= U16 * np.abs(ref) + 1e-3)


# ------------------------------------------------------------- attention ----

def _attn_case(case, heads, nq, n_own, n_pre, vis=None):
    H = heads * 128
    panel = S.op_tensor(9, case, 0, (n_own, 3 * H), 1.0).astype(np.float16)
    kvp = S.op_tensor(9, case, 1, (max(n_pre, 1), 2 * H), 1.0).astype(np.float16)[:n_pre]
    out = torch.full((nq, H), float("nan"), dtype=torch.float16, device="cuda")
    visd = None if vis is None else T(np.asarray(vis, np.int32))
    q.op_attention(T(panel), heads, out, nq, n_own, kv_pre=T(kvp) if n_pre else None, n_pre=n_pre, vis=visd)
    p = panel.astype(np.float64)
    kv = kvp.astype(np.float64)
    K = np.concatenate([kv[:, :H], p[:, H:2 * H]], axis=0)
    V = np.concatenate([kv[:, H:], p[:, 2 * H:]], axis=0)
    v = np.full(nq, n_pre + n_own) if vis is None else np.minimum(np.asarray(vis), n_pre + n_own)
    ref = O.attention(p[:nq, :H], K, V, v, heads, 128)
    return host(out).astype(np.float64), ref


@pytest.mark.parametrize("heads,nq,n_own,n_pre", [
    (2, 130, 130, 18),      # step: 18-row prefix + 130 own keys, ragged tiles
    (2, 256, 256, 18),
    (1, 1, 1, 0),           # a single key
    (2, 64, 64, 4114),      # a long cache, block boundary inside the cache
    (4, 200, 200, 63),      # prefix/panel boundary one short of a key block
    (32, 129, 129, 1),
    (2, 100, 100, 64),      # cache of exactly one 64-key box: a block of cache and panel boxes
    (2, 5, 5, 70),          # padded cache boxes, then a panel box reaching past the panel
    (3, 300, 300, 191),
    (2, 140, 140, 129),
])
def test_attention_step_mode(heads, nq, n_own, n_pre):
    got, ref = _attn_case(nq * 31 + n_pre, heads, nq, n_own, n_pre)
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) < 2e-3
    assert np.max(np.abs(got - ref)) < 1e-2


@pytest.mark.parametrize("segs", [
    [(0, 5, 0), (1, 4, 6), (0, 3, 0), (1, 3, 2), (1, 1, 1)],
    [(0, 18, 0), (1, 16, 16), (0, 5, 0), (1, 2, 2)],
    [(0, 130, 0), (1, 1, 1)],          # purely causal text
    [(1, 12, 11), (0, 7, 0), (1, 1, 1)],  # image first: bidirectional block of 132
])
def test_attention_prefill_mask(segs):
    vis = O.prefix_visibility(segs).astype(np.int64)
    lp = len(vis)
    got, ref = _attn_case(lp, 2, lp, lp, 0, vis=vis)
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) < 2e-3
    assert np.max(np.abs(got - ref)) < 1e-2
    # a text query must not see later keys: first row attends to key 0 only
    H = 256
    panel = S.op_tensor(9, lp, 0, (lp, 3 * H), 1.0).astype(np.float16)
    if vis[0] == 1:
        np.testing.assert_allclose(got[0], panel[0, 2 * H:].astype(np.float64), atol=2 * U16 * 4)


def _expected_parts(epi, M, N, K, clusters):
    """The documented part count of qi21_op_gemm_split with ample scratch:
    the tiles of a partial last wave (pairs of 256 rows x BN columns) split
    into the largest power of two <= min(clusters // tail tiles, k-blocks,
    cap), cap 2 for SWIGLU (128-column owners; on a 128-column tile the
    second part only contributes), else min(8, BN / 32)."""
    bn = 256 if N % 256 == 0 else 128
    pairs = ((M + 127) // 128 + 1) // 2 * (N // bn)
    rem = pairs % clusters
    if pairs <= clusters or rem == 0:
        return 1
    cap = 2 if epi == "swiglu" else min(8, bn // 32)
    lim = min(cap, clusters // rem, K // 64)
    p = 1
    while p * 2 <= lim:
        p *= 2
    return p


def _split_case(epi, dtype, M, N, K, seed):
    A = S.op_tensor(11, seed, 0, (M, K), 1.0).astype(np.float32)
    Bw = S.op_tensor(11, seed, 1, (N, K), K ** -0.5).astype(np.float32)
    if dtype == "bf16":
        A, Bw = S.bf16_values(S.bf16_bits(A)), S.bf16_values(S.bf16_bits(Bw))
        tA, tB = T(A).to(torch.bfloat16), T(Bw).to(torch.bfloat16)
    else:
        A, Bw = A.astype(np.float16), Bw.astype(np.float16)
        tA, tB = T(A), T(Bw)
    return A, Bw, tA, tB


# (epilogue, operand type, M, N, K): tail tiles of 4, 16, 28 and 14 pairs
# (parts 8, 4, 2 and 4 on 76 resident clusters), a 128-column tile, SWIGLU
# at its cap of two parts (two owners on 256-column tiles; one owner and
# one contributor on 128-column tiles)
SPLIT_CASES = [
    ("resid", "f16", 2500, 2048, 1024),
    ("f32", "f16", 5788, 1024, 768),
    ("f16", "f16", 3251, 2048, 512),
    ("swiglu", "f16", 2500, 2048, 1024),
    ("resid", "bf16", 2500, 1152, 512),
    ("swiglu", "bf16", 2500, 1152, 512),
    ("swiglu", "f16", 3251, 2048, 512),
    ("resid", "f16", 4096, 4096, 4096),
]


@pytest.mark.parametrize("epi,dtype,M,N,K", SPLIT_CASES)
def test_gemm_k_split_tail(epi, dtype, M, N, K):
    # the K-split tail against the oracle's f64 products; against the
    # unsplit GEMM (the same sums in another order: f32 rounding apart); two
    # split runs bit-identical; with no room for partials it is the unsplit
    # GEMM bit for bit
    clusters = torch.cuda.get_device_properties(0).multi_processor_count // 2
    A, Bw, tA, tB = _split_case(epi, dtype, M, N, K, M + N + K)
    E = {"resid": q.EPI_RESID, "f32": q.EPI_F32, "f16": q.EPI_F16, "swiglu": q.EPI_SWIGLU}[epi]
    scratch = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    cols = N // 2 if epi == "swiglu" else N
    odt = torch.float32 if epi in ("resid", "f32") else tA.dtype
    x0 = S.op_tensor(11, M, 2, (M, cols), 1.0) if epi == "resid" else None
    gt = T(np.tanh(S.op_tensor(11, M, 3, (N,), 0.1))) if epi == "resid" else None

    def run(split, room=64 << 20):
        out = T(x0) if epi == "resid" else torch.zeros((M, cols), dtype=odt, device="cuda")
        if split:
            parts = q.op_gemm_split(E, tA, tB, out, scratch[:room], gate_t=gt)
        else:
            q.op_gemm(E, tA, tB, out, gate_t=gt)
            parts = 1
        return host(out.float()).astype(np.float64), parts

    got, parts = run(True)
    assert parts == _expected_parts(epi, M, N, K, clusters)
    rows = np.arange(M) if M * N * K <= 8e9 else np.array([0, 1, 255, 256, 2047, 3840, 3968, 4095])
    a = A[rows].astype(np.float64)
    if epi == "swiglu":
        G, Up = np.empty((N // 2, K)), np.empty((N // 2, K))
        for j in range(N // 128):  # the interleaved plane: 64 gate rows, then 64 up rows
            G[64 * j:64 * j + 64] = Bw[128 * j:128 * j + 64]
            Up[64 * j:64 * j + 64] = Bw[128 * j + 64:128 * j + 128]
        ref = O.silu(a @ G.T) * (a @ Up.T)
    else:
        ref = a @ Bw.astype(np.float64).T
        if epi == "resid":
            ref = x0[rows] + np.tanh(S.op_tensor(11, M, 3, (N,), 0.1)).astype(np.float64) * ref
    g = got[rows]
    u = U16 if dtype == "f16" else 2.0 ** -8
    if epi in ("resid", "f32"):
        assert rel_l2(g, ref) < 1e-5
    else:
        assert np.all(np.abs(g - ref) <= 2 * u * np.abs(ref) + 2e-3)
    plain, _ = run(False)
    if epi in ("resid", "f32"):
        assert np.max(np.abs(got - plain)) <= 1e-5 * np.max(np.abs(plain))
    else:  # one output rounding apart, plus the f32 reordering of O(1) sums
        assert np.all(np.abs(got - plain) <= 2 * u * np.abs(plain) + 1e-5)
    again, _ = run(True)
    np.testing.assert_array_equal(again, got)
    none, p1 = run(True, room=4096)
    assert p1 == 1
    np.testing.assert_array_equal(none, plain)


def test_gemm_split_rejects_bad_scratch():
    A, Bw, tA, tB = _split_case("f16", "f16", 256, 256, 64, 1)
    out = torch.empty((256, 256), dtype=torch.float16, device="cuda")
    scratch = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    for bad in (scratch[:100], scratch[16:]):
        with pytest.raises(q.Qi21Error) as e:
            q.op_gemm_split(q.EPI_F16, tA, tB, out, bad)
        assert e.value.code == -8
