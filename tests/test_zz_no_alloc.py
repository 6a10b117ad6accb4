"""The allocation-free step, qi21_step_noalloc, against the ordinary step.

Some callers cannot allocate device memory: their memory belongs to another
allocator and they have no buffer to lend, or they run under a
no-allocation rule after start-up because cudaMalloc can synchronise the
device and stall other streams. qi21_step_noalloc serves them from a static
device scratch inside the library. Through the C ABI, this checks that two
calls in a row give exactly the block output of qi21_step with a caller
workspace (the same kernels on the same inputs: bit for bit, so a stale
scratch would show) and the oracle's within the block bar, that a warm call
allocates no device memory, and that a step too large for the scratch is
refused with QI21_ERR_WORKSPACE.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from oracle import qi21_oracle as O  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu

X_TOL = 2e-3


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_noalloc_step_matches_the_workspace_step_twice():
    w = S.WORKLOADS["ragged_d512"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    ref = dw.step().cpu().numpy().copy()
    cfg = O.cfg_of(w)
    weights = [S.layer_weights(w, l) for l in range(w.layers)]
    cache, _ = O.prefill(S.x_prefix(w), weights, S.mods0(w), w.segs(0), cfg)
    oracle_out, _ = O.step(S.x_target(w), weights, S.mods_t(w), w.segs(0), cache, cfg)
    for _ in range(2):
        out = torch.full_like(dw.x_target, float("nan"))
        q.step_noalloc(dw.g, dw.layers, dw.caches[0], dw.x_target, out, dw.mods_t)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        np.testing.assert_array_equal(got, ref)
        assert _rel(got, oracle_out) <= X_TOL
    assert q.device_status() == 0


def test_noalloc_step_allocates_no_device_memory():
    w = S.WORKLOADS["tiny_block_d256"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    out = torch.empty_like(dw.x_target)
    q.step_noalloc(dw.g, dw.layers, dw.caches[0], dw.x_target, out, dw.mods_t)  # warm: first call per device
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        q.step_noalloc(dw.g, dw.layers, dw.caches[0], dw.x_target, out, dw.mods_t)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert q.device_status() == 0


def test_noalloc_step_refuses_a_step_larger_than_its_scratch():
    w = S.WORKLOADS["block_d4096_n4096"]
    g = D.geom_of(w)
    cache = q.KVCache(g, w.segs(0))
    assert q.workspace_bytes(g, cache.n) > (32 << 20)
    dummy = torch.zeros(1, device="cuda")
    with pytest.raises(q.Qi21Error) as e:
        q.step_noalloc(g, [], cache, dummy, dummy, dummy)
    assert e.value.code == -8
    assert "static scratch" in str(e.value)
