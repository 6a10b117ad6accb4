"""The optional non-finite refusal (qi21_set_checks / QI21_CHECK_FINITE) and
the scan behind it (qi21_count_nonfinite), the page's "a non-finite velocity
is declined" rule of its device step (gpu_wgpu/qi21.rs, step).

The counts are integers decided by exponent bits: compared exactly with
numpy's isfinite on the same host values.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu

ERR_NONFINITE = -10


@pytest.fixture(autouse=True)
def _clean():
    prev = q.set_checks(0)
    yield
    q.set_checks(prev)
    assert q.device_status() == 0


def _planted(n, dtype, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(n).astype(dtype)
    if n:
        k = max(1, n // 997)
        idx = rng.choice(n, size=min(n, k), replace=False)
        bad = np.array([np.nan, np.inf, -np.inf], dtype)
        a[idx] = bad[rng.integers(0, 3, size=idx.size)]
        # the largest finite values must not count
        big = np.finfo(dtype).max
        a[rng.integers(0, n, size=min(n, 3))] = big
        a[0] = a[0] if n < 5 else -big
    return a


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 4096, 1000003])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_count_nonfinite_exact(dtype, n, offset):
    a = _planted(n + offset, dtype, n * 7 + offset)
    t = torch.from_numpy(a).cuda()[offset:]  # offset views: unaligned heads
    want = int(np.count_nonzero(~np.isfinite(a[offset:])))
    assert q.count_nonfinite(t) == want


def test_count_nonfinite_nan_payloads_and_subnormals():
    bits = np.array([0x7fc00001, 0xffc00000, 0x7f800001, 0x7f800000, 0xff800000, 0x00000001, 0x7f7fffff,
                     0x80800000], np.uint32)
    t = torch.from_numpy(bits.view(np.float32)).cuda()
    assert q.count_nonfinite(t) == 5
    h = np.array([0x7c01, 0xfe00, 0x7c00, 0xfc00, 0x0001, 0x7bff, 0x8400], np.uint16)
    assert q.count_nonfinite(torch.from_numpy(h.view(np.float16)).cuda()) == 4


def _tiny():
    w = S.WORKLOADS["tiny_block_d256"]
    dw = D.DeviceWorkload(w)
    io = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (S.tokens(w), S.w_in(w), S.w_out(w),
                                                                      S.final_scale(w))]
    return w, dw, io


def test_checks_pass_on_finite_work_and_refuse_planted_values():
    w, dw, (tok, w_in, w_out, fs) = _tiny()
    out = torch.empty((w.n_target, 64), device="cuda")
    assert q.set_checks(q.CHECK_FINITE) == 0
    dw.prefill_all()
    dw.step()
    q.denoise(dw.g, dw.layers, dw.caches[0], tok, w_in, dw.mods_t, fs, w_out, out, dw.ws)
    assert q.count_nonfinite(out) == 0
    # an infinite proj_out weight: the velocity is refused
    w_bad = w_out.clone()
    w_bad[5, 17] = float("inf")
    with pytest.raises(q.Qi21Error) as ei:
        q.denoise(dw.g, dw.layers, dw.caches[0], tok, w_in, dw.mods_t, fs, w_bad, out, dw.ws)
    assert ei.value.code == ERR_NONFINITE
    # a NaN in the step's input: the hidden state is refused
    x_bad = dw.x_target.clone()
    x_bad[3, 9] = float("nan")
    with pytest.raises(q.Qi21Error) as ei:
        dw.step(x_in=x_bad)
    assert ei.value.code == ERR_NONFINITE
    # a NaN in the prefix: the cache is refused
    dw.x_prefix[0][2, 1] = float("nan")
    with pytest.raises(q.Qi21Error) as ei:
        dw.prefill_all()
    assert ei.value.code == ERR_NONFINITE
    # the checks off: the same calls are accepted (asynchronously)
    q.set_checks(0)
    dw.prefill_all()
    q.denoise(dw.g, dw.layers, dw.caches[0], tok, w_in, dw.mods_t, fs, w_bad, out, dw.ws)
    torch.cuda.synchronize()
    assert q.count_nonfinite(out) > 0


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    # a wait that nothing ends: the kernel gives up after its limit (~2 s),
    # raises the status word and returns; no fault, the context stays usable
    import time
    assert q.device_status() == 0
    t0 = time.monotonic()
    q.selftest_wait_timeout()
    torch.cuda.synchronize()
    dt = time.monotonic() - t0
    assert 1.0 < dt < 30.0, dt
    assert q.device_status() != 0
    assert q.device_status() == 0  # read and cleared
    a = _planted(4096, np.float32, 11)
    assert q.count_nonfinite(torch.from_numpy(a).cuda()) == int(np.count_nonzero(~np.isfinite(a)))
    w, dw, _ = _tiny()
    dw.prefill_all()
    dw.step()
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["tiny_block_d256", "tiny_block_d256_bf16"])
def test_amax_probe_records_the_stored_maxima(name):
    # QI21_CHECK_AMAX: the largest |value| stored at each 16-bit site of a
    # pass (the page's AMAX probe). A one-layer step leaves its qkv panel,
    # attention output, second LayerNorm rows and SwiGLU rows in the
    # workspace: their maxima equal the recorded ones exactly; the first
    # LayerNorm's rows are overwritten, so attn-in is checked against the
    # oracle within one rounding of the 16-bit type.
    from oracle import qi21_oracle as O
    from synthetic import device as D
    w = S.WORKLOADS[name]
    dw = D.DeviceWorkload(w)
    q.amax_read(reset=True)
    prev = q.set_checks(q.CHECK_AMAX)
    try:
        dw.prefill_all()
        pre = q.amax_read(reset=True)
        _, l0 = q.profile_read()
        dw.step()
        got = q.amax_read(reset=True)
        _, l1 = q.profile_read()
    finally:
        q.set_checks(prev)
    # the prefill of one layer stops after the qkv projection
    assert pre["attn-in"] > 0 and pre["qkv"] > 0
    assert pre["attn-out"] == 0 and pre["ffn-in"] == 0 and pre["hidden"] == 0
    assert l1["misc"] - l0["misc"] == 1 + 5  # the modulation prep and five probes
    M, H, I = w.n_target, w.dim, w.mlp_hidden

    def a256(v):
        return (v + 255) // 256 * 256

    xn = a256(M * H * 4)
    panel = xn + a256(M * H * 2)
    att = panel + a256(M * 3 * H * 2)
    hid = att + a256(M * H * 2)
    dt = q.dtype_of(dw.g)

    def mx(off, count):
        return float(dw.ws[off:off + count * 2].view(dt).float().abs().max())

    assert got["ffn-in"] == mx(xn, M * H)
    assert got["qkv"] == mx(panel, M * 3 * H)
    assert got["attn-out"] == mx(att, M * H)
    assert got["hidden"] == mx(hid, M * I)
    ref = float(np.abs(O.norm_mod(S.x_target(w), S.mods_t(w)[:H], w.eps)).max())
    u = 2.0 ** (-8 if w.dtype == "bf16" else -11)
    assert abs(got["attn-in"] - ref) <= 2 * u * ref
    assert all(v == 0 for v in q.amax_read(reset=False).values())
    # with the flag off nothing is probed
    _, l2 = q.profile_read()
    dw.step()
    _, l3 = q.profile_read()
    assert l3["misc"] - l2["misc"] == 1
    assert all(v == 0 for v in q.amax_read(reset=False).values())
