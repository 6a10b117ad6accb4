"""Several host threads calling the library at once, each on its own CUDA
stream, in a fresh process: the first calls of the GEMM, attention and row
kernels (one-time set-up of kernel attributes, tensor-map encoder, SM
count) happen concurrently. Every result must equal, bit for bit, the
result of the same call made afterwards from one thread (the kernels are
deterministic), and no kernel may report a give-up.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import diffusion_transformer_denoiser_qi21_gb300 as q

    rng = np.random.default_rng(5)
    def dev(shape, dtype, scale=1.0):
        return torch.from_numpy((scale * rng.standard_normal(shape)).astype(dtype)).cuda()

    H = 256
    A = dev((300, 512), np.float16)
    B = dev((256, 512), np.float16)
    g_out = torch.empty((300, 256), dtype=torch.float32, device="cuda")
    xr = dev((300, 256), np.float32)
    Br = dev((256, 512), np.float16, 0.05)
    gate = dev((256,), np.float32, 0.3)
    panel = dev((130, 3 * H), np.float16)
    kv = dev((18, 2 * H), np.float16)
    a_out = torch.empty((130, H), dtype=torch.float16, device="cuda")
    x = dev((700, 1024), np.float32)
    sc = dev((1024,), np.float32, 0.1)
    xn = torch.empty((700, 1024), dtype=torch.float16, device="cuda")
    x_res0 = xr.clone()
    torch.cuda.synchronize()

    def job_gemm(s):
        q.op_gemm(1, A, B, g_out, stream=s)
    def job_resid(s):
        q.op_gemm(2, A, Br, xr, gate_t=gate, stream=s)
    def job_attn(s):
        q.op_attention(panel, 2, a_out, 130, 130, kv_pre=kv, n_pre=18, stream=s)
    def job_rowop(s):
        q.op_rowop(x, sc, xn=xn, stream=s)
    jobs = [job_gemm, job_resid, job_attn, job_rowop]
    errors = []
    start = threading.Barrier(len(jobs))
    def run(job):
        try:
            s = torch.cuda.Stream()
            start.wait()
            job(s)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(repr(e))
    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert q.device_status() == 0
    got = [g_out.clone(), xr.clone(), a_out.clone(), xn.clone()]

    xr.copy_(x_res0)
    for job in jobs:
        job(None)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    want = [g_out, xr, a_out, xn]
    for i, (a, b) in enumerate(zip(got, want)):
        assert torch.equal(a, b), i
        assert torch.isfinite(a.float()).all(), i
    print("OK")
""").replace("ROOT", repr(ROOT))


def test_concurrent_first_calls_from_threads():
    r = subprocess.run([sys.executable, "-c", SCRIPT], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.strip().endswith("OK")
