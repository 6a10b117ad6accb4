"""Block-level parity of the CUDA prefill and step against the CPU oracle,
through the C ABI (qi21_prefill / qi21_step / qi21_step_batch).

Bar: rel L2 <= 2e-3 of every block output (the hidden state after the
block) against the oracle on the same seeded inputs, both end to end (each
side runs its own chain) and teacher-forced (the oracle's block l is fed
the GPU's input of block l and the GPU's cache of layer l). The block's own
contribution x_out - x_in, which the residual would otherwise dilute, is
held to rel L2 <= 1e-2 and the K/V cache to rel L2 <= 2e-3.

Small workloads run the whole oracle; the full-width workloads (dim 4096)
check sampled layers and sampled rows (block outputs are row-independent
given every key), which the oracle computes row by row, plus exact
properties that hold at any size.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from blockcheck import DeviceRun, end_to_end, host, rel_l2, sample_rows, teacher_forced_layer  # noqa: E402
from oracle import qi21_oracle as O  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu

X_TOL = 2e-3
DELTA_TOL = 1e-2
KV_TOL = 2e-3


TOL = (X_TOL, DELTA_TOL, KV_TOL)


def _teacher_forced_layer(run, layer, s, W, cfg, rows_pre=None, rows_step=None):
    return teacher_forced_layer(run, layer, s, W, cfg, TOL, rows_pre=rows_pre, rows_step=rows_step)


SMALL = ["tiny_block_d256", "chain32_d256_mixed", "ragged_d512", "cfg_pair_d256", "single_row_d256",
         "heads3_d384_n4356"]


@pytest.mark.parametrize("name", SMALL)
def test_small_workload_end_to_end_and_teacher_forced(name):
    w = S.WORKLOADS[name]
    run = DeviceRun(w)
    cfg = O.cfg_of(w)
    weights = [S.layer_weights(w, l) for l in range(w.layers)]
    end_to_end(run, weights, cfg, TOL)
    for s in range(w.nseq):
        for l in range(w.layers):
            _teacher_forced_layer(run, l, s, weights[l], cfg)


def test_zero_gates_give_the_identity_exactly():
    w = S.WORKLOADS["ragged_d512"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    H = w.dim
    m = S.mods_t(w).copy()
    m[H:2 * H] = 0.0
    m[3 * H:] = 0.0
    dw.mods_t = D.to_dev(m)
    out = dw.step()
    np.testing.assert_array_equal(host(out), np.concatenate([S.x_target(w)] * w.nseq))


def test_cfg_batch_equals_single_steps_exactly():
    w = S.WORKLOADS["cfg_pair_d256"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    both = host(dw.step()).copy()
    n = w.n_target
    for s in range(w.nseq):
        out = torch.empty((n, w.dim), device="cuda")
        q.step(dw.g, dw.layers, dw.caches[s], dw.x_target[s * n:(s + 1) * n].contiguous(), out, dw.mods_t, dw.ws)
        np.testing.assert_array_equal(host(out), both[s * n:(s + 1) * n])


def test_step_in_place_and_repeatable():
    w = S.WORKLOADS["tiny_block_d256"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    a = host(dw.step()).copy()
    x = dw.x_target.clone()
    q.step(dw.g, dw.layers, dw.caches[0], x, x, dw.mods_t, dw.ws)
    np.testing.assert_array_equal(host(x), a)
    b = host(dw.step())
    np.testing.assert_array_equal(a, b)


def test_step_rejects_unfilled_cache_and_small_workspace():
    w = S.WORKLOADS["tiny_block_d256"]
    dw = D.DeviceWorkload(w)
    with pytest.raises(q.Qi21Error) as e:
        dw.step()
    assert e.value.code == -7
    dw.prefill_all()
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.Qi21Error) as e:
        q.step(dw.g, dw.layers, dw.caches[0], dw.x_target, dw.x_out, dw.mods_t, small)
    assert e.value.code == -8


# ------------------------------------------------------------ full width ----

_sample_rows = sample_rows


def test_block_d4096_n4096_sampled():
    w = S.WORKLOADS["block_d4096_n4096"]
    run = DeviceRun(w)
    cfg = O.cfg_of(w)
    W = S.layer_weights(w, 0)
    rows = _sample_rows(w.n_target, 1)
    e, d = _teacher_forced_layer(run, 0, 0, W, cfg, rows_step=rows)
    print(f"block_d4096_n4096: step rel L2 {e:.2e}, delta {d:.2e}")


@pytest.fixture(scope="module")
def layers32():
    w = S.WORKLOADS["step32_cond4114_n4096"]
    g = D.geom_of(w)
    layers = D.upload_layers(w, g)
    yield layers
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,layers_checked", [
    ("step32_cond4114_n4096", (0, 1, 31)),
    ("step32_n16384", (0, 31)),
    ("cfg_pair32_n1024", (0, 31)),
])
def test_full_width_32_layers_sampled(name, layers_checked, layers32):
    w = S.WORKLOADS[name]
    run = DeviceRun(w, layers=layers32)
    cfg = O.cfg_of(w)
    rows = _sample_rows(w.n_target, 2)
    for l in layers_checked:
        W = S.layer_weights(w, l)
        for s in range(w.nseq):
            lp = w.prefix_rows(s)
            rows_pre = _sample_rows(lp, 3) if lp > 256 else None
            e, d = _teacher_forced_layer(run, l, s, W, cfg, rows_pre=rows_pre, rows_step=rows)
            print(f"{name} layer {l} seq {s}: step rel L2 {e:.2e}, delta {d:.2e}")
    out = host(run.out)
    assert np.all(np.isfinite(out))
    del run
    torch.cuda.empty_cache()


def test_a_bad_later_layer_enqueues_nothing():
    # every layer is validated and every tensor map encoded before the first
    # launch: a misaligned plane in layer 3 of 32 is refused with no kernel
    # launched and the output untouched
    import ctypes as C

    from diffusion_transformer_denoiser_qi21_gb300 import _binding as B
    w = S.WORKLOADS["chain32_d256_mixed"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    torch.cuda.synchronize()
    arr = (B.Layer * w.layers)()
    for i, l in enumerate(dw.layers):
        arr[i] = l.c
    arr[3].w13 = arr[3].w13 + 2  # 2-byte aligned
    out = torch.full_like(dw.x_target, float("nan"))
    _, before = q.profile_read()
    rc = q.load().qi21_step(C.byref(dw.g), arr, dw.caches[0].handle, dw.x_target.data_ptr(), out.data_ptr(),
                            dw.mods_t.data_ptr(), None, dw.ws.data_ptr(), dw.ws.numel(), None)
    assert rc == -1 and b"layer 3" in q.load().qi21_last_error()
    torch.cuda.synchronize()
    _, after = q.profile_read()
    assert after == before
    assert torch.isnan(out).all()


@pytest.mark.parametrize("name", ["ragged_d512", "chain32_d256_mixed", "tiny_block_d256_bf16"])
def test_prefill_cache_rows_are_the_panel_k_v_bits(name):
    # the qkv epilogue of a prefill stores each k and v value into the panel
    # and into the layer's cache row; the last layer stops after it, so the
    # workspace still holds that layer's panel: its K|V columns and the cache
    # of the last layer agree bit for bit
    w = S.WORKLOADS[name]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    torch.cuda.synchronize()
    H, lp = w.dim, dw.caches[0].lp

    def a256(v):
        return (v + 255) // 256 * 256

    off = a256(lp * H * 4) + a256(lp * H * 2)  # x [lp][H] f32, xn [lp][H], then the panel [lp][3H]
    panel = dw.ws[off:off + lp * 3 * H * 2].view(torch.int16).view(lp, 3 * H)
    kv = dw.caches[0].layer_tensor(w.layers - 1).view(torch.int16)
    assert torch.equal(kv, panel[:, H:])


def test_tiny_block_against_the_unrounded_f32_weights():
    # for information: the device runs the f16-rounded weights (the bar is
    # against the oracle on exactly those); the oracle on the unrounded f32
    # draws shows what the weight rounding itself moves (about 2^-11 / sqrt(3)
    # of each weight, spread over the block's projections)
    w = S.WORKLOADS["tiny_block_d256"]
    run = DeviceRun(w, keep_prefill_x=False)
    cfg = O.cfg_of(w)
    W32 = {}
    for tag in S.WEIGHT_TAGS:
        r, c = S.weight_shape(w, tag)
        W32[tag] = S.normal(w.seed, tag, 0, r * c, c ** -0.5).reshape(r, c)
    W32["norm_q"] = S.norm_weight(w, 0, "norm_q")
    W32["norm_k"] = S.norm_weight(w, 0, "norm_k")
    segs = w.segs(0)
    cache, _ = O.prefill(S.x_prefix(w), [W32], S.mods0(w), segs, cfg)
    ref32, _ = O.step(S.x_target(w), [W32], S.mods_t(w), segs, cache, cfg)
    cache16, _ = O.prefill(S.x_prefix(w), [S.layer_weights(w, 0)], S.mods0(w), segs, cfg)
    ref16, _ = O.step(S.x_target(w), [S.layer_weights(w, 0)], S.mods_t(w), segs, cache16, cfg)
    got = host(run.out)
    x0 = S.x_target(w).astype(np.float64)
    e32 = rel_l2(got, ref32)
    d32 = rel_l2(got - x0, ref32 - x0)
    print(f"tiny_block_d256 vs oracle on f32 weights: block rel L2 {e32:.2e}, delta {d32:.2e}; "
          f"vs f16-rounded weights {rel_l2(got, ref16):.2e}; the two oracles differ by {rel_l2(ref16, ref32):.2e}")
    assert np.isfinite(e32) and e32 < 2e-3
