"""Bounded device waits: a call whose first kernel waits on a flag that nothing
sets (the variant word's test hook) must come back, report a device timeout
through aircache_get_error, leave every later kernel of the call idle, and
leave the workspace usable: the next call on it compresses as a fresh one does.
The failure is made on the host side of the contract (a flag no kernel writes,
a short limit); nothing faults or hangs the GPU."""
import numpy as np
import pytest
import torch

from lvlm_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lvlm_kv_cache_gb300 import build

    build.build()
    from lvlm_kv_cache_gb300 import aircache

    aircache.lib()
    return aircache


def _problem(A, wl, **kw):
    s = wl.spec
    return A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha,
                     s.r, **kw)


def test_wait_expiry_reported_and_workspace_reusable(A):
    wl = W.make("7b", device="cuda", layers=3)
    good = _problem(A, wl)
    hooked = _problem(A, wl, wait_test=True)
    ref = A.compress(good)
    torch.cuda.synchronize()
    ws = good.new_workspace()
    assert hooked.workspace_size() == good.workspace_size()
    for _ in range(2):
        with pytest.raises(A.AirCacheError) as e:
            A.compress(hooked, ws=ws)
        assert e.value.status == A.ERR_DEVICE_TIMEOUT
        out = A.compress(good, ws=ws)  # the same workspace, now without the hook
        torch.cuda.synchronize()
        for key in ("iv", "keep", "out_offsets"):
            assert torch.equal(out[key], ref[key]), key
        for l in range(good.L):  # each layer's selection (entries past keep are not written)
            kp = int(ref["keep"][l])
            assert torch.equal(out["idx"][l, :kp], ref["idx"][l, :kp])
        n = int(ref["out_offsets"][-1])
        assert torch.equal(out["out_k"][:n], ref["out_k"][:n])
        assert torch.equal(out["out_v"][:n], ref["out_v"][:n])
