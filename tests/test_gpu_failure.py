"""Device-side failure path: a bounded wait that runs out.

The dense attention kernel is run through a test hook that limits every
device wait to 1 ms and makes its Q load warp withhold the first Q tile, so
the first S product waits for a barrier that nothing completes.  The kernel
must return on its own, report FOCUS_ERR_TIMEOUT through the workspace's
error word, and leave the context and the workspace usable: the next normal
call on the same workspace matches the oracle.  Nothing here faults, traps or
hangs the GPU: every wait in the kernel is bounded.
"""
import time

import numpy as np
import pytest

import oracle.focus_ref as ref
from learned_group_sparse_focus_gb300 import synth
from _helpers import to_dev, to_host, TOL_BF16_MAX, TOL_BF16_MEAN

FOCUS_ERR_INVALID_ARG = 1
FOCUS_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def fz():
    from learned_group_sparse_focus_gb300 import focus
    return focus


def test_wait_limit_hook_checks_its_arguments(fz):
    # rejected before any device work: wait limit 0 or above one second
    p = fz.make_params(B=1, H=2, H_kv=1, n=300, d=128, D=64, d_g=32, K=4, A=1, w=300)
    lib = fz.lib()
    import ctypes
    for bad in (0, 1_000_000_001):
        st = lib.focus_test_attention_wait_limit(ctypes.byref(p), 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1 << 30,
                                                 bad, None)
        assert st == FOCUS_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("n,H,H_kv,d", [(700, 2, 1, 128), (300, 4, 2, 64)])
def test_wait_runs_out_and_the_next_call_is_correct(fz, n, H, H_kv, d):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    wl = synth.Workload("t", B=1, H=H, H_kv=H_kv, n=n, d=d, D=64, d_g=32, K=4, w=n, A=1, dtype="bf16",
                        groups="uniform", seed=77 + n)
    x = synth.draw(wl, parts=("attn",))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace(p)
    Q, K, V = (to_dev(x[k], "bf16") for k in ("Q", "K", "V"))
    O = torch.zeros_like(Q)
    torch.cuda.synchronize()
    t0 = time.time()
    fz.focus_test_attention_wait_limit(p, Q, K, V, O, ws, wait_ns=1_000_000)
    assert fz.focus_check_errors(ws) == FOCUS_ERR_TIMEOUT
    elapsed = time.time() - t0
    assert elapsed < 5.0, elapsed           # the kernel gave up on its own
    assert fz.focus_check_errors(ws) == 0   # the report cleared the word
    # the same workspace and context serve a normal call
    fz.focus_dense_causal_fwd(p, Q, K, V, O, None, ws)
    assert fz.focus_check_errors(ws) == 0
    g = np.zeros((1, 1, n), dtype=np.int32)
    want, _ = ref.attention(x["Q"], x["K"], x["V"], g, n, wl.scale, 1)
    diff = np.abs(to_host(O) - want)
    assert diff.max() <= TOL_BF16_MAX and diff.mean() <= TOL_BF16_MEAN, (diff.max(), diff.mean())
