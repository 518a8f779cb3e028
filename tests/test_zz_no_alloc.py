"""fa_bwd_noalloc: the backward with the library's built-in scratch array.

Some callers cannot allocate device memory on this path -- a framework that
owns all device memory and forbids libraries to allocate, or a serving loop
that must not call cudaMalloc while it runs. fa_bwd_noalloc serves them by
keeping its workspace in a fixed-size device array inside the library. This
file checks, through the C ABI, that two calls in a row give what the
workspace-taking entry point gives (within the backward's tolerance, with
dK and dV bitwise equal since each has one writer per element), that the
Python binding's wrapper with caller-provided outputs does the same, and
that a problem too large for the array is refused without a launch. It is collected
last so that a failure here leaves every other test already run; it also
passes on its own in a fresh process.
"""

import ctypes
import math

import numpy as np
import pytest

import synthetic_inputs as si

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

REL_MAX = 5e-2  # the backward gate used by the parity tests


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _rel(got, ref):
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    return float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-3))


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 333, 64, True), (1, 2, 256, 128, False)])
def test_two_calls_match_the_workspace_entry_point(B, H, N, d, causal):
    lib = fa.load_library()
    scale = 1.0 / math.sqrt(d)
    x = {k: t.cuda() for k, t in si.make_small(B, H, N, d, seed=77 + N, with_grad=True).items()}
    o, lse = fa.fa_fwd(x["q"], x["k"], x["v"], causal=causal, scale=scale)
    ref = fa.fa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    outs = []
    for _ in range(2):
        dq, dk, dv = (torch.full_like(x["q"], float("nan")) for _ in range(3))
        rc = lib.fa_bwd_noalloc(_p(x["q"]), _p(x["k"]), _p(x["v"]), _p(o), _p(lse), _p(x["do"]),
                                _p(dq), _p(dk), _p(dv), B, H, N, d, int(causal), scale,
                                ctypes.c_void_p(stream.cuda_stream))
        assert rc == fa.FA_OK, fa.fa_strerror(rc)
        torch.cuda.synchronize()
        outs.append((dq, dk, dv))
    assert lib.fa_get_last_device_status() == fa.FA_OK
    for dq, dk, dv in outs:
        assert torch.isfinite(dq.float()).all()
        assert _rel(dq, ref[0]) <= REL_MAX
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    # the two calls agree with each other as well (dQ up to atomic ordering)
    assert _rel(outs[1][0], outs[0][0]) <= REL_MAX


def test_python_wrapper_with_preallocated_outputs():
    # the binding's fa_bwd_noalloc (shape checks, caller-provided outputs,
    # device and stream handling) gives what fa_bwd gives
    B, H, N, d, causal = 1, 3, 300, 64, True
    x = {k: t.cuda() for k, t in si.make_small(B, H, N, d, seed=5, with_grad=True).items()}
    o, lse = fa.fa_fwd(x["q"], x["k"], x["v"], causal=causal)
    ref = fa.fa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal=causal)
    outs = tuple(torch.full_like(x["q"], float("nan")) for _ in range(3))
    got = fa.fa_bwd_noalloc(x["q"], x["k"], x["v"], o, lse, x["do"], causal=causal, dq=outs[0],
                            dk=outs[1], dv=outs[2], stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert all(g is t for g, t in zip(got, outs))
    assert _rel(got[0], ref[0]) <= REL_MAX
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_problem_larger_than_the_scratch_is_refused():
    lib = fa.load_library()
    B, H, N, d = 4, 32, 8192, 64
    assert lib.fa_bwd_workspace_bytes(B, H, N, d) > fa.FA_BWD_NOALLOC_MAX_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")  # never read: refused first
    p = _p(t)
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 1, 0.125, ctypes.c_void_p(0))
    assert rc == fa.FA_ERR_WORKSPACE
