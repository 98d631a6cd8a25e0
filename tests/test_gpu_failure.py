"""GPU: the bounded-wait failure path of the tensor-core expert kernels.

Every wait inside those kernels gives up after a wall-time limit, records MOE_ERR_DEVICE
in the workspace error word, and lets the CTA finish the copies and MMAs it already
issued, free its tensor memory and exit.  The test shortens the limit to 50 ms and makes
the down tiles wait for a publication count that nothing ever reaches (a host-side
injection through moe_debug_set_waits: no invalid memory, no trap), then checks that the
call returns promptly with the error recorded, that the CUDA context is still usable, and
that the next ordinary call on the same workspace is correct: bit-identical to a call
made before the failure and within tolerance of the oracle."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth

pytestmark = pytest.mark.gpu

from parity import NEAR_TIE, rel_err, to_f64, tolerance  # noqa: E402


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_routing_grouped_router_gb300 import build
    build.build()
    oracle.build()
    import top_routing_grouped_router_gb300 as m
    return m


def _forward(moe, L, ws):
    out = torch.full((L.T, L.shape.H), float("nan"), dtype=L.out_dtype(), device="cuda")
    ids = torch.full((L.T, L.shape.k), -1, dtype=torch.int32, device="cuda")
    moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, out, ids,
                    workspace=ws)
    return out, ids


# bf16 decode (tensor-core kernel), 4-bit decode and a large 4-bit batch (the 4-bit kernel's
# two tile shapes) and a large bf16 batch (several token chunks per expert)
@pytest.mark.parametrize("name,T", [("decode8", None), ("decode48q", None), ("decode48q", 200), ("decode8", 600)])
def test_bounded_wait_runs_out_and_the_next_call_is_correct(moe, name, T):
    from top_routing_grouped_router_gb300.device import upload
    inp = synth.make_inputs(name, T=T)
    L = upload(inp)
    ws = L.new_workspace()
    ref, ref_ids = _forward(moe, L, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_error(ws) == 0

    moe.moe_debug_set_waits(50_000_000, 1 << 20)  # 50 ms; down tiles wait for a count nothing reaches
    try:
        t0 = time.perf_counter()
        _forward(moe, L, ws)
        torch.cuda.synchronize()  # raises if the context was lost
        dt = time.perf_counter() - t0
    finally:
        moe.moe_debug_set_waits()
    assert moe.moe_read_device_error(ws) == -7  # MOE_ERR_DEVICE
    assert dt < 5.0, f"the failing call took {dt:.2f} s"

    # the same workspace, the default limit: correct again
    out, ids = _forward(moe, L, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_error(ws) == 0
    assert torch.equal(ids, ref_ids)
    assert torch.equal(out, ref)
    toks = np.arange(min(inp.T, 24), dtype=np.int32)
    r = oracle.forward_tokens(inp, toks)
    keep = r["tie_margin"] >= NEAR_TIE
    err = rel_err(to_f64(out)[toks][keep], r["out"][keep])
    assert err <= tolerance(inp), err
