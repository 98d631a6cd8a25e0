"""GPU: bucketed CUDA-graph decode (moe_graphs_* of the C ABI).

Every step of T tokens must give, bit for bit, the live rows of moe_forward on the
zero-padded batch of its bucket, and those rows must match the oracle within the bf16
tolerance."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth

pytestmark = pytest.mark.gpu

import top_routing_grouped_router_gb300 as moe  # noqa: E402
from top_routing_grouped_router_gb300.device import bf16_tensor_bits, upload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_routing_grouped_router_gb300 import build
    build.build()
    oracle.build()


def _padded_forward(L, x, T, B):
    s = moe.make_shape(B, L.shape.H, L.shape.E, L.shape.k, L.shape.I)
    xp = torch.zeros((B, L.shape.H), dtype=x.dtype, device=x.device)
    xp[:T] = x[:T]
    out = torch.empty_like(xp)
    ids = torch.empty((B, L.shape.k), dtype=torch.int32, device=x.device)
    ws = torch.zeros(moe.moe_workspace_size(s), dtype=torch.uint8, device=x.device)
    moe.moe_forward(s, xp, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, None, out, ids, workspace=ws)
    return out[:T], ids[:T]


@pytest.mark.parametrize("max_bs,steps", [(64, [1, 3, 8, 13, 33, 64, 8])])
def test_bucketed_graph_steps_equal_padded_forward_and_oracle(max_bs, steps):
    inp = synth.make_inputs("decode8", T=max_bs)
    L = upload(inp)
    g = moe.DecodeGraphs(L.shape, max_bs, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down)
    assert g.buckets == [1, 2, 4, 8, 16, 32, 48, 64]
    x = L.x
    for T in steps:
        out = torch.empty((T, inp.H), dtype=torch.bfloat16, device="cuda")
        ids = torch.empty((T, inp.k), dtype=torch.int32, device="cuda")
        g.run(T, x[:T], out, ids)
        g._stream.synchronize()
        B = g.bucket(T)
        ref_out, ref_ids = _padded_forward(L, x, T, B)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids), T
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), T
        toks = np.arange(min(T, 4))
        o = oracle.forward_tokens(inp, toks)
        got = synth.bf16_bits_to_f32(bf16_tensor_bits(out[:len(toks)]))
        keep = o["tie_margin"] >= 1e-5
        err = np.abs(got[keep] - o["out"][keep]).max() / np.abs(o["out"][keep]).max()
        assert err <= 1e-2, (T, err)
    g.close()


def test_graph_step_from_pinned_host_buffers_and_replay_is_deterministic():
    inp = synth.make_inputs("decode8", T=16)
    L = upload(inp)
    g = moe.DecodeGraphs(L.shape, 16, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down)
    T = 11
    xh = L.x[:T].cpu().pin_memory()
    outs = []
    for _ in range(2):
        oh = torch.empty((T, inp.H), dtype=torch.bfloat16).pin_memory()
        g.run(T, xh, oh)
        g._stream.synchronize()
        outs.append(oh)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref_out, _ = _padded_forward(L, L.x, T, 16)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), ref_out.cpu().view(torch.int16))
    with pytest.raises(moe.MoEError):
        g.run(17, xh, oh)  # larger than every bucket
    g.close()


def test_graph_step_from_pageable_and_unaligned_buffers_equals_the_aligned_step():
    """Buffers the device cannot address (pageable host memory) or whose address is not a
    multiple of 16 bytes take the copy-engine route around the bucket's graph; both must give
    the same bits as device buffers."""
    inp = synth.make_inputs("decode8", T=16)
    L = upload(inp)
    g = moe.DecodeGraphs(L.shape, 16, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down)
    T, H = 13, inp.H
    ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ref_ids = torch.empty((T, inp.k), dtype=torch.int32, device="cuda")
    g.run(T, L.x[:T], ref, ref_ids)
    # pageable host memory
    xh = L.x[:T].cpu()
    oh = torch.empty((T, H), dtype=torch.bfloat16)
    g.run(T, xh, oh)
    g._stream.synchronize()
    # device buffers 2 bytes past a 16-byte boundary
    xb = torch.empty(T * H + 1, dtype=torch.bfloat16, device="cuda")
    ob = torch.empty(T * H + 1, dtype=torch.bfloat16, device="cuda")
    xu, ou = xb[1:].view(T, H), ob[1:].view(T, H)
    assert xu.data_ptr() % 16 and ou.data_ptr() % 16
    xu.copy_(L.x[:T])
    torch.cuda.synchronize()
    ids = torch.empty((T, inp.k), dtype=torch.int32, device="cuda")
    g.run(T, xu, ou, ids)
    g._stream.synchronize()
    assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(ou.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(ids, ref_ids)
    g.close()


def test_graph_steps_with_4bit_weights_equal_padded_forward():
    """The bucket graphs of a 4-bit layer (prep, 4-bit decode kernel) from pinned host buffers:
    every step equals the live rows of moe_forward on the zero-padded batch."""
    inp = synth.make_inputs("decode48q", T=48)
    L = upload(inp)
    g = moe.DecodeGraphs(L.shape, 48, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4)
    for T in (48, 5, 20):
        B = g.bucket(T)
        xh = L.x[:T].cpu().pin_memory()
        oh = torch.empty((T, inp.H), dtype=torch.bfloat16).pin_memory()
        g.run(T, xh, oh)
        g._stream.synchronize()
        s = moe.make_shape(B, inp.H, inp.E, inp.k, inp.I, w=L.shape.w_dtype, q_block=L.shape.q_block)
        xp = torch.zeros((B, inp.H), dtype=torch.bfloat16, device="cuda")
        xp[:T] = L.x[:T]
        ref = torch.empty_like(xp)
        ws = torch.zeros(moe.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
        moe.moe_forward(s, xp, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, ref, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(oh.view(torch.int16), ref[:T].cpu().view(torch.int16)), T
    g.close()
