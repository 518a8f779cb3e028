"""The bounded-wait (timeout) path of the kernels, on the GPU, without a fault.

Every wait inside the kernels gives up after a wall-clock budget, raises the
CTA's abort flag, and every role winds down: the TMA producer lets its copies
in flight land, the MMA thread waits for its MMAs, TMEM is freed, and the
kernel sets the device status word that ``fa_get_last_device_status`` turns
into FA_ERR_TIMEOUT. A test-only variant of the library (built separately
with ``-DFA_TEST_SKIP_ARRIVE``, never part of ``libfa.so``) makes that happen
on purpose: the forward's producer never loads the last V tile of its key
stream, and the backward's producers never load the last query step of an
item (the d = 64 kernel: of each CTA's first item, after which it loads
nothing more), so the issuing warps' waits run out after the variant's 20 ms
budget. Each test checks that the call returns, that the status says
FA_ERR_TIMEOUT (once: reading it clears it), and that the same process then
runs the product library's forward and backward with results matching the
oracle, i.e. the context is intact.
"""

import ctypes
import math
import time

import numpy as np
import pytest

import synthetic_inputs as si
from oracle import dense

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def timeout_lib():
    from exact_io_aware_33_gb300 import build as b
    return fa.load_library(b.build_timeout_test_variant())


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("d", [64, 128])
def test_wait_runs_out_and_the_context_survives(timeout_lib, d):
    B, H, N, scale = 1, 1, 256, 1.0 / math.sqrt(d)
    x = si.make_small(B, H, N, d, seed=3100 + d, with_grad=True)
    g = {n: t.cuda() for n, t in x.items()}
    o = torch.empty_like(g["q"])
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK

    t0 = time.perf_counter()
    rc = timeout_lib.fa_fwd_stream(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(o), _p(lse), B, H, N, d, 0,
                                   scale, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_OK  # launched; the failure shows in the status word
    status = timeout_lib.fa_get_last_device_status()  # synchronises the device
    elapsed = time.perf_counter() - t0
    assert status == fa.FA_ERR_TIMEOUT
    assert elapsed < 10.0, f"the wind-down took {elapsed:.2f} s"
    assert timeout_lib.fa_get_last_device_status() == fa.FA_OK  # read once, then cleared
    # the product library's status word is separate and untouched
    assert fa.fa_get_last_device_status() == fa.FA_OK

    # the context still works: a normal forward and backward in the same process
    torch.cuda.synchronize()
    o2, lse2 = fa.fa_fwd(g["q"], g["k"], g["v"], causal=False, scale=scale)
    grads = fa.fa_bwd(g["q"], g["k"], g["v"], o2, lse2, g["do"], causal=False, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = dense.forward(x["q"], x["k"], x["v"], False, scale)
    err = np.abs(o2.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.abs(lse2.cpu().double().numpy() - lse_ref).max() <= 1e-3
    refs = dense.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], False, scale)
    for got, ref in zip(grads, refs):
        gg = got.float().cpu().double().numpy()
        assert np.abs(gg - ref).max() / np.abs(ref).max() <= 5e-2


@pytest.mark.parametrize("d", [64, 128])
def test_backward_wait_runs_out_and_the_context_survives(timeout_lib, d):
    # d = 64: the persistent pipelined kernel; d = 128: the sequential one.
    # N = 384 causal gives items of 3, 2 and 1 query steps per head.
    B, H, N, scale = 1, 2, 384, 1.0 / math.sqrt(d)
    x = si.make_small(B, H, N, d, seed=3200 + d, with_grad=True)
    g = {n: t.cuda() for n, t in x.items()}
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], causal=True, scale=scale)  # product library
    grads = [torch.empty_like(g["q"]) for _ in range(3)]
    ws_bytes = timeout_lib.fa_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK

    t0 = time.perf_counter()
    rc = timeout_lib.fa_bwd_stream(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(o), _p(lse), _p(g["do"]),
                                   _p(grads[0]), _p(grads[1]), _p(grads[2]), B, H, N, d, 1, scale, _p(ws),
                                   ws_bytes, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_OK
    status = timeout_lib.fa_get_last_device_status()
    elapsed = time.perf_counter() - t0
    assert status == fa.FA_ERR_TIMEOUT
    assert elapsed < 10.0, f"the wind-down took {elapsed:.2f} s"
    assert timeout_lib.fa_get_last_device_status() == fa.FA_OK
    assert fa.fa_get_last_device_status() == fa.FA_OK

    # the product library's backward in the same process, against the oracle
    got = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = dense.forward(x["q"], x["k"], x["v"], True, scale)
    refs = dense.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], True, scale)
    for t, ref in zip(got, refs):
        gg = t.float().cpu().double().numpy()
        assert np.abs(gg - ref).max() / np.abs(ref).max() <= 5e-2


@pytest.mark.parametrize("d,dv,window", [(128, 64, 0), (64, 128, 0), (128, 128, 200)])
def test_forward_ex_wait_runs_out_and_the_context_survives(timeout_lib, d, dv, window):
    # The persistent two-tile forward's other forms: P in columns of its own
    # (d_v = 64), d = 64 with d_v = 128, and a window (tiles starting at
    # different key tiles); causal, N = 512.
    from oracle import general
    B, H, N, scale = 1, 2, 512, 1.0 / math.sqrt(d)
    gen = torch.Generator().manual_seed(3300 + d + dv + window)
    x = {"q": torch.randn(B, H, N, d, generator=gen).to(torch.bfloat16),
         "k": torch.randn(B, H, N, d, generator=gen).to(torch.bfloat16),
         "v": torch.randn(B, H, N, dv, generator=gen).to(torch.bfloat16)}
    g = {n: t.cuda() for n, t in x.items()}
    o = torch.empty(B, H, N, dv, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK

    t0 = time.perf_counter()
    rc = timeout_lib.fa_fwd_ex(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(o), _p(lse), B, H, N, N, d, dv, 1,
                               window, scale, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_OK
    status = timeout_lib.fa_get_last_device_status()
    elapsed = time.perf_counter() - t0
    assert status == fa.FA_ERR_TIMEOUT
    assert elapsed < 10.0, f"the wind-down took {elapsed:.2f} s"
    assert timeout_lib.fa_get_last_device_status() == fa.FA_OK
    assert fa.fa_get_last_device_status() == fa.FA_OK

    # the product library's forward in the same process, against the oracle
    o2, lse2 = fa.fa_fwd_ex(g["q"], g["k"], g["v"], causal=True, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = general.forward(x["q"], x["k"], x["v"], True, scale, window)
    err = np.abs(o2.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.abs(lse2.cpu().double().numpy() - lse_ref).max() <= 1e-3
