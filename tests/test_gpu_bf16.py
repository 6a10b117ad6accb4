"""The bf16 path (qi21_geom.dtype = QI21_DTYPE_BF16) against the CPU oracle,
through the C ABI: the single operations with bf16 operands and outputs,
and whole blocks with the weights rounded to bf16 (the oracle widens
exactly those values, as for f16).

Tolerances follow from bf16's unit roundoff u = 2^-8 (8 significant bits):
one rounding of a stored value has a relative RMS error of u / sqrt(3)
(2.3e-3), against 2.8e-4 for f16.
  - 16-bit outputs element-wise: |gpu - ref| <= 2u |ref| + a few u of the
    output scale (one rounding plus f32 arithmetic);
  - f32 GEMM outputs: rel L2 <= 1e-5 (the operands are exact bf16 values,
    f32 accumulation), as for f16;
  - attention: two bf16 roundings in sequence (P before P V, the stored
    output) give ~3.2e-3 RMS: rel L2 <= 8e-3;
  - blocks: the hidden state after a block within rel L2 2e-3 (the bar; the
    f32 residual carries most of it), the block's own contribution within
    3e-2 (a few bf16 roundings, ~8x the f16 figure), the K/V cache within
    6e-3 (two roundings: the modulated-LN row and the stored K / V).
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from blockcheck import DeviceRun, end_to_end, host, rel_l2, sample_rows, teacher_forced_layer  # noqa: E402
from oracle import qi21_oracle as O  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu

UB = 2.0 ** -8
TOL = (2e-3, 3e-2, 6e-3)


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def TB(a):
    """A bf16 CUDA tensor holding the bf16 rounding of float array a."""
    bits = S.bf16_bits(np.asarray(a, np.float32))
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def rb(a):
    """The bf16 rounding of a, as float64 (what the device holds)."""
    return S.bf16_values(S.bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert q.device_status() == 0, "a kernel gave up waiting"


# ------------------------------------------------------------------ rows ----

@pytest.mark.parametrize("rows,dim", [(1, 128), (130, 512), (2000, 4096), (700, 8192)])
def test_rowop_norm_bf16(rows, dim):
    x = S.op_tensor(12, dim, 0, (rows, dim), 3.0, offset=0.5)
    sc = S.op_tensor(12, dim, 1, (dim,), 0.1)
    xn = torch.empty((rows, dim), dtype=torch.bfloat16, device="cuda")
    q.op_rowop(T(x), T(sc), xn=xn)
    ref = O.norm_mod(x, sc, 1e-6)
    got = host(xn).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * UB * np.abs(ref) + 4 * UB * 2 ** -3)


@pytest.mark.parametrize("rows,heads", [(33, 2), (300, 32)])
def test_qkrope_bf16(rows, heads):
    H = heads * 128
    panel = rb(S.op_tensor(13, rows * heads, 0, (rows, 3 * H), 2.0))
    nq = S.op_tensor(13, rows * heads, 1, (128,), 0.05, offset=1.0)
    nk = S.op_tensor(13, rows * heads, 2, (128,), 0.05, offset=1.0)
    segs = [(0, 7, 0), (1, 9, 11), (1, rows, 1)]
    cs, sn = O.rope_tables(O.positions(segs)[-rows:])
    pd = TB(panel)
    q.op_qkrope(pd, heads, T(nq), T(nk), T(cs), T(sn))
    got = host(pd).astype(np.float64)
    rq = O.qk_norm_rope(panel[:, :H], nq, cs, sn, heads, 128, 1e-6)
    rk = O.qk_norm_rope(panel[:, H:2 * H], nk, cs, sn, heads, 128, 1e-6)
    for g, r in ((got[:, :H], rq), (got[:, H:2 * H], rk)):
        assert np.all(np.abs(g - r) <= 2 * UB * np.abs(r) + 4 * UB * 2 ** -3)
    np.testing.assert_array_equal(got[:, 2 * H:], panel[:, 2 * H:])  # v untouched


def test_kvcopy_bf16_exact():
    rows, H = 77, 512
    panel = TB(S.op_tensor(14, 0, 0, (rows, 3 * H), 1.0))
    kv = torch.zeros((rows, 2 * H), dtype=torch.bfloat16, device="cuda")
    q.op_kvcopy(panel, kv)
    assert torch.equal(kv.view(torch.int16), panel[:, H:].contiguous().view(torch.int16))


# ------------------------------------------------------------------ GEMM ----

@pytest.mark.parametrize("shape", [(1, 128, 64), (130, 768, 256), (513, 256, 4096), (4114, 512, 256)])
def test_gemm_bf16_f32_and_store(shape):
    M, N, K = shape
    A = rb(S.op_tensor(15, M + N, 0, (M, K), 1.0))
    Bw = rb(S.op_tensor(15, M + N, 1, (N, K), K ** -0.5))
    ref = A @ Bw.T
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.op_gemm(q.EPI_F32, TB(A), TB(Bw), out)
    got = host(out)
    assert rel_l2(got, ref) < 1e-5
    out16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    q.op_gemm(q.EPI_F16, TB(A), TB(Bw), out16)
    g16 = host(out16).astype(np.float64)
    assert np.all(np.abs(g16 - ref) <= UB * np.abs(ref) + 1e-3)


@pytest.mark.parametrize("shape", [(18, 256, 256), (300, 512, 1536), (129, 4096, 4096)])
def test_gemm_bf16_residual_gate(shape):
    M, N, K = shape
    A = rb(S.op_tensor(16, M, 0, (M, K), 1.0))
    Bw = rb(S.op_tensor(16, M, 1, (N, K), K ** -0.5))
    x0 = S.op_tensor(16, M, 2, (M, N), 1.0)
    gt = np.tanh(S.op_tensor(16, M, 3, (N,), 0.1))
    xd = T(x0)
    q.op_gemm(q.EPI_RESID, TB(A), TB(Bw), xd, gate_t=T(gt))
    ref = x0 + gt.astype(np.float64) * (A @ Bw.T)
    got = host(xd)
    assert rel_l2(got, ref) < 1e-6
    assert np.max(np.abs(got - ref)) < 1e-4


def _interleave_w13(G, Up):
    I, H = G.shape
    out = np.empty((2 * I, H), G.dtype)
    for j in range(I // 64):
        out[128 * j:128 * j + 64] = G[64 * j:64 * j + 64]
        out[128 * j + 64:128 * j + 128] = Up[64 * j:64 * j + 64]
    return out


@pytest.mark.parametrize("M,I,K", [(130, 768, 256), (257, 12288, 4096)])
def test_gemm_bf16_swiglu(M, I, K):
    A = rb(S.op_tensor(17, M, 0, (M, K), 1.0))
    G = rb(S.op_tensor(17, M, 1, (I, K), K ** -0.5))
    Up = rb(S.op_tensor(17, M, 2, (I, K), K ** -0.5))
    out = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    q.op_gemm(q.EPI_SWIGLU, TB(A), TB(_interleave_w13(G, Up)), out)
    ref = O.silu(A @ G.T) * (A @ Up.T)
    got = host(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * UB * np.abs(ref) + 2e-3)


# ------------------------------------------------------------- attention ----

def _attn_case(case, heads, nq, n_own, n_pre, vis=None):
    H = heads * 128
    panel = rb(S.op_tensor(18, case, 0, (n_own, 3 * H), 1.0))
    kvp = rb(S.op_tensor(18, case, 1, (max(n_pre, 1), 2 * H), 1.0))[:n_pre]
    out = torch.full((nq, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    visd = None if vis is None else T(np.asarray(vis, np.int32))
    q.op_attention(TB(panel), heads, out, nq, n_own, kv_pre=TB(kvp) if n_pre else None, n_pre=n_pre, vis=visd)
    K = np.concatenate([kvp[:, :H], panel[:, H:2 * H]], axis=0)
    V = np.concatenate([kvp[:, H:], panel[:, 2 * H:]], axis=0)
    v = np.full(nq, n_pre + n_own) if vis is None else np.minimum(np.asarray(vis), n_pre + n_own)
    ref = O.attention(panel[:nq, :H], K, V, v, heads, 128)
    return host(out).astype(np.float64), ref


@pytest.mark.parametrize("heads,nq,n_own,n_pre", [
    (2, 130, 130, 18), (1, 1, 1, 0), (2, 64, 64, 4114), (4, 200, 200, 63), (2, 5, 5, 70),
])
def test_attention_bf16_step_mode(heads, nq, n_own, n_pre):
    got, ref = _attn_case(nq * 31 + n_pre, heads, nq, n_own, n_pre)
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) < 8e-3
    assert np.max(np.abs(got - ref)) < 8e-2


def test_attention_bf16_prefill_mask():
    segs = [(0, 18, 0), (1, 16, 16), (0, 5, 0), (1, 2, 2)]
    vis = O.prefix_visibility(segs).astype(np.int64)
    lp = len(vis)
    got, ref = _attn_case(lp, 2, lp, lp, 0, vis=vis)
    assert rel_l2(got, ref) < 8e-3
    assert np.max(np.abs(got - ref)) < 8e-2


# ---------------------------------------------------------------- blocks ----

@pytest.mark.parametrize("name", ["tiny_block_d256_bf16", "cfg_pair_d256_bf16", "chain32_d256_mixed_bf16"])
def test_bf16_blocks_end_to_end_and_teacher_forced(name):
    w = S.WORKLOADS[name]
    run = DeviceRun(w)
    assert run.kv(0, 0).dtype == torch.bfloat16
    cfg = O.cfg_of(w)
    weights = [S.layer_weights(w, l) for l in range(w.layers)]
    worst = end_to_end(run, weights, cfg, TOL)
    print(f"{name}: worst end-to-end block rel L2 {worst:.2e}")
    for s in range(w.nseq):
        for l in range(w.layers):
            teacher_forced_layer(run, l, s, weights[l], cfg, TOL)


def test_bf16_full_width_block_sampled():
    w = S.WORKLOADS["block_d4096_n4096_bf16"]
    run = DeviceRun(w)
    cfg = O.cfg_of(w)
    e, d = teacher_forced_layer(run, 0, 0, S.layer_weights(w, 0), cfg, TOL,
                                rows_step=sample_rows(w.n_target, 1))
    print(f"block_d4096_n4096_bf16: step rel L2 {e:.2e}, delta {d:.2e}")


def test_bf16_32_layers_condition_prefix_sampled():
    # the 32-layer step with the 4114-row condition prefix, bf16 weights:
    # teacher-forced layers 0 and 31 on sampled rows, the output finite
    w = S.WORKLOADS["step32_cond4114_n4096_bf16"]
    run = DeviceRun(w)
    cfg = O.cfg_of(w)
    rows = sample_rows(w.n_target, 2)
    for l in (0, 31):
        e, d = teacher_forced_layer(run, l, 0, S.layer_weights(w, l), cfg, TOL,
                                    rows_pre=sample_rows(w.prefix_rows(0), 3), rows_step=rows)
        print(f"step32_cond4114_n4096_bf16 layer {l}: step rel L2 {e:.2e}, delta {d:.2e}")
    assert np.all(np.isfinite(host(run.out)))
    assert q.count_nonfinite(run.kv(0, 31)) == 0
    del run
    torch.cuda.empty_cache()


def test_bf16_geometry_refuses_f16_planes_and_fp8():
    w = S.WORKLOADS["tiny_block_d256_bf16"]
    g = D.geom_of(w)
    h = torch.zeros((256, 256), dtype=torch.float16, device="cuda")
    n = torch.ones(128, device="cuda")
    with pytest.raises(TypeError):
        q.pack_layer(g, h, h, h, h, h, h, h, n, n)
    assert q.workspace_bytes_fp8(g, 16) == 0
    assert q.load().qi21_geom_check(C.byref(g)) == 0
