"""moe_forward_static_scratch: the MoE block for callers that cannot allocate device memory.

Such callers (code running during another thread's global-mode graph capture, plugins
whose host framework owns all device memory, paths that cannot take cudaMalloc's
implicit synchronisation) get the same block with its scratch in the library's fixed
32 MiB device array instead of a workspace.  This file runs last so that a failure here
leaves every other test already run.  It calls the entry point through the C ABI and
checks it against moe_forward on two calls in a row: both run the same kernels on the
same inputs, so the outputs must agree bit for bit.
"""
import ctypes

import pytest

torch = pytest.importorskip("torch")

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_routing_grouped_router_gb300 import build
    build.build()
    import top_routing_grouped_router_gb300 as m
    return m


def _ptr(t):
    return None if t is None else t.data_ptr()


def _static_call(moe, L, out, ids, w):
    L_ = moe.lib()
    q4 = ctypes.byref(L.q4) if L.q4 is not None else None
    return L_.moe_forward_static_scratch(ctypes.byref(L.shape), _ptr(L.x), _ptr(L.w_router), _ptr(L.b_router),
                                         _ptr(L.w_gate), _ptr(L.w_up), _ptr(L.w_down), q4, _ptr(out), _ptr(ids),
                                         _ptr(w), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["tiny", "decode8", "decode64z", "decode48q"])
def test_static_scratch_matches_workspace_forward_twice(moe, name):
    from top_routing_grouped_router_gb300.device import upload
    inp = synth.make_inputs(name)
    L = upload(inp)
    T, H, k = inp.T, inp.H, inp.k
    ref = torch.empty((T, H), dtype=L.out_dtype(), device="cuda")
    ref_ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = L.new_workspace()
    moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, ref, ref_ids, ref_w,
                    workspace=ws)
    for _ in range(2):
        out = torch.full((T, H), float("nan"), dtype=L.out_dtype(), device="cuda")
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        assert _static_call(moe, L, out, ids, w) == 0
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        assert torch.equal(w, ref_w)
        assert torch.equal(out, ref)
    assert moe.moe_read_device_error(ws) == 0
    # the static array's error word is readable too, and no call recorded an error
    assert moe.moe_static_scratch_read_error() == 0


def test_static_scratch_rejects_shapes_beyond_its_size(moe):
    s = moe.make_shape(4096, 2048, 128, 8, 768)
    assert moe.moe_workspace_size(s) > (32 << 20)
    fake = 1 << 20  # never dereferenced: the size check fails before anything is enqueued
    rc = moe.lib().moe_forward_static_scratch(ctypes.byref(s), fake, fake, None, fake, fake, fake, None, fake,
                                              None, None, None)
    assert rc == -4  # MOE_ERR_WORKSPACE
