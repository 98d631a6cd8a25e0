"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, step by step,
on the seeded workloads at full size and on reduced, ragged and degenerate cases."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth

pytestmark = pytest.mark.gpu

from parity import check_layer, run_steps  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_routing_grouped_router_gb300 import build
    build.build()
    oracle.build()


def test_tiny_fp32_full():
    s, _ = check_layer(synth.make_inputs("tiny"), full_oracle=True)
    assert s["out_rel_err"] <= 1e-5


def test_decode8_full_size():
    check_layer(synth.make_inputs("decode8"), full_oracle=True)


def test_decode64_zipf_full_size_has_empty_experts():
    s, g = check_layer(synth.make_inputs("decode64z"), full_oracle=True)
    assert (g["counts"] == 0).sum() >= 1
    assert g["counts"].max() >= 32


def test_decode48_q4_full_size():
    check_layer(synth.make_inputs("decode48q"), full_oracle=True)


def test_prefill_q4_full_size():
    s, g = check_layer(synth.make_inputs("prefill4q"), full_oracle=False, n_sample_tokens=16, n_sample_rows=32,
                       target_experts=True, token_slice=64)
    assert g["counts"].sum() == 4096 * 8


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_prefill_full_size_layer(layer):
    s, g = check_layer(synth.make_inputs("prefill", layer=layer), full_oracle=False, n_sample_tokens=16,
                       n_sample_rows=32, target_experts=True, token_slice=64)
    assert g["counts"].sum() == 4096 * 8


@pytest.mark.parametrize("T,H,E,k,I,act,w,zipf", [
    (19, 72, 8, 2, 40, "f32", "f32", False),        # ragged everything, fp32
    (37, 2048, 128, 8, 768, "bf16", "bf16", False),  # odd token count at the decode shape
    (300, 512, 64, 6, 256, "bf16", "bf16", True),   # several permute chunks in one block
    (700, 256, 128, 8, 128, "bf16", "bf16", False),  # multi-block permute with a ragged last chunk
    (21, 256, 16, 4, 128, "bf16", "q4", False),      # 4-bit, two scale blocks per row
    (5, 128, 8, 8, 64, "bf16", "bf16", False),       # k == E: every expert, infinite margins
    (40, 256, 2, 2, 128, "bf16", "q4", False),       # 4-bit, 40 tokens per expert (one k-slab per down stage)
    (64, 384, 8, 2, 256, "bf16", "q4", True),        # 4-bit, skewed load, three row blocks of H
    (600, 512, 16, 4, 256, "bf16", "bf16", False),   # large batch: several token chunks per expert
    (1030, 512, 8, 2, 384, "bf16", "bf16", True),    # large batch, skewed load: ragged chunks
    (200, 256, 16, 4, 128, "bf16", "q4", False),     # 4-bit large batch: several 128-token chunks per expert
    (300, 512, 8, 2, 256, "bf16", "q4", True),       # 4-bit large batch, skewed load
    (37, 512, 16, 4, 256, "bf16", "q4", False),      # 4-bit decode on CUDA cores: 8 and 4 scale blocks per row
    (64, 64, 4, 2, 64, "bf16", "q4", True),          # 4-bit decode, one scale block per row, up to 64 tokens per expert
    (8, 256, 256, 8, 128, "bf16", "bf16", False),    # E = 256, the largest: 8 logits per lane, one-warp permutation
    (40, 256, 160, 6, 128, "bf16", "bf16", True),    # E = 160 (ragged over the lanes), five token groups
    (16, 256, 256, 4, 128, "bf16", "q4", False),     # 4-bit decode at E = 256
    (8, 4096, 32, 4, 256, "bf16", "bf16", False),    # H = 4096: two hidden-dim chunks per router thread, 32 down row blocks
    (8, 256, 16, 1, 128, "bf16", "bf16", False),     # top-1 routing at decode
    (12, 4096, 16, 2, 128, "bf16", "q4", False),     # 4-bit with 64 scale blocks per row: the generic kernels
])
def test_reduced_and_ragged_cases(T, H, E, k, I, act, w, zipf):
    inp = synth.make_custom(T, H, E, k, I, act=act, w=w, zipf=zipf, seed=T + E, name=f"custom{T}")
    # every y row and every token against the oracle: the second token chunk of an expert
    # with more than 256 rows, the split down chunks and the ragged last tiles included
    check_layer(inp, full_oracle=True)


def test_q4_non_affine_codebook_uses_generic_kernels():
    inp = synth.make_custom(12, 256, 8, 2, 128, act="bf16", w="q4", seed=17)
    rng = np.random.default_rng(4)
    inp.codebook = np.sort(rng.uniform(-1, 1, 16)).astype(np.float32)
    check_layer(inp, full_oracle=True)


def test_no_renormalisation():
    inp = synth.make_custom(12, 128, 16, 3, 64, act="f32", w="f32", seed=3, norm_topk=False)
    check_layer(inp, full_oracle=True)


def test_single_token():
    check_layer(synth.make_inputs("decode8", T=1), full_oracle=True)


def test_all_tokens_to_the_same_experts():
    inp = synth.make_custom(40, 256, 32, 4, 128, act="bf16", w="bf16", seed=5)
    bias = np.zeros(32, np.float32)
    bias[[3, 17, 22, 30]] = 40.0
    inp.b_router = bias
    s, g = check_layer(inp, full_oracle=True)
    assert sorted(np.nonzero(g["counts"])[0].tolist()) == [3, 17, 22, 30]
    assert (g["counts"][[3, 17, 22, 30]] == 40).all()


def test_exact_logit_ties_pick_the_lower_expert_first():
    # experts 5, 9 and 12 get expert 2's router row and bias, so their logits equal expert 2's
    # bit for bit on every token (same rows, same arithmetic); with k = 3 the tie straddles the
    # selection boundary, and the slots must hold 2, 5, 9 in that order, as in the oracle (a
    # tie goes to the lower expert index)
    import top_routing_grouped_router_gb300 as moe
    from top_routing_grouped_router_gb300.device import upload
    inp = synth.make_custom(16, 256, 32, 3, 128, act="bf16", w="bf16", seed=21)
    for e in (5, 9, 12):
        inp.w_router[e] = inp.w_router[2]
    bias = np.zeros(32, np.float32)
    bias[[2, 5, 9, 12]] = 8.0
    inp.b_router = bias
    L = upload(inp)
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((inp.T, inp.k), dtype=torch.int32, device="cuda")
    moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, None, out, ids,
                    workspace=L.new_workspace())
    torch.cuda.synchronize()
    ref = oracle.forward_tokens(inp, np.arange(inp.T))["ids"]
    assert (ref == np.array([2, 5, 9])).all()
    np.testing.assert_array_equal(ids.cpu().numpy(), ref)


def test_two_experts_take_every_token_of_a_large_batch():
    inp = synth.make_custom(777, 256, 16, 2, 128, act="bf16", w="bf16", seed=9)
    bias = np.zeros(16, np.float32)
    bias[[2, 11]] = 40.0
    inp.b_router = bias
    s, g = check_layer(inp, full_oracle=True)
    assert (g["counts"][[2, 11]] == 777).all()


def test_zero_tokens():
    import top_routing_grouped_router_gb300 as moe
    from top_routing_grouped_router_gb300.device import upload
    inp = synth.make_custom(0, 128, 8, 2, 64, act="bf16", w="bf16", seed=1)
    L = upload(inp)
    ws = L.new_workspace()
    counts = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((9,), -1, dtype=torch.int32, device="cuda")
    dummy = torch.empty(4, dtype=torch.int32, device="cuda")
    moe.moe_permute(L.shape, dummy, counts, offsets, dummy, dummy, ws)
    out = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L.shape, L.x if L.x.numel() else dummy, L.w_router, None, L.w_gate, L.w_up, L.w_down, None,
                    out, workspace=ws)
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == [0] * 8 and offsets.cpu().tolist() == [0] * 9


def test_forward_is_deterministic_and_graph_replay_is_bitwise_equal():
    import top_routing_grouped_router_gb300 as moe
    from top_routing_grouped_router_gb300.device import upload
    inp = synth.make_inputs("decode64z")
    L = upload(inp)
    ws = L.new_workspace()
    outs = []
    for _ in range(2):
        out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
        moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, out, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    g_out = torch.empty_like(outs[0])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, g_out,
                        workspace=ws)
    g_out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(g_out, outs[0])
    # replay again after changing the input in place: the graph reads the new tokens
    L.x.copy_(torch.flip(L.x, dims=[0]))
    graph.replay()
    eager = torch.empty_like(g_out)
    moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, eager, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(g_out, eager)
    assert torch.equal(eager, torch.flip(outs[0], dims=[0]))


def test_out_of_range_expert_id_is_recorded_not_trapped():
    import top_routing_grouped_router_gb300 as moe
    s = moe.make_shape(4, 128, 8, 2, 64)
    ws = torch.zeros(moe.moe_workspace_size(s), dtype=torch.uint8, device="cuda")
    ids = torch.tensor([[0, 1], [2, 8], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    counts = torch.empty(8, dtype=torch.int32, device="cuda")
    offsets = torch.empty(9, dtype=torch.int32, device="cuda")
    order = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    pos = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    moe.moe_permute(s, ids, counts, offsets, order, pos, ws)
    assert moe.moe_read_device_error(ws) == -7  # MOE_ERR_DEVICE
    assert moe.moe_read_device_error(ws) == 0
    assert counts.sum().item() == 7


@pytest.mark.parametrize("name,entry", [("decode8", "forward"), ("decode48q", "forward"), ("decode8", "rmsnorm"),
                                        ("decode48q", "rmsnorm")])
def test_chained_layers_read_the_previous_layers_output(name, entry):
    """Each call's kernels overlap the previous call's tail (programmatic dependent launch),
    so a kernel that read its inputs before waiting would see the previous layer's output
    half-written.  Layer l + 1 reads layer l's output as its tokens: the chain enqueued
    back to back must equal, bit for bit, the same chain with a synchronisation between
    calls."""
    import top_routing_grouped_router_gb300 as moe
    from top_routing_grouped_router_gb300.device import upload, to_device
    inp = synth.make_inputs(name)
    L = upload(inp)
    ws = L.new_workspace()
    gamma = to_device(synth.make_norm_weight(inp.H, inp.act, seed=7), "cuda")

    def chain(sync):
        x = L.x.clone()
        outs = []
        for _ in range(4):
            out = torch.empty_like(x)
            if entry == "rmsnorm":
                moe.moe_forward_rmsnorm(L.shape, x, gamma, 1e-6, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down,
                                        L.q4, out, workspace=ws)
            else:
                moe.moe_forward(L.shape, x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, out,
                                workspace=ws)
            if sync:
                torch.cuda.synchronize()
            outs.append(out)
            x = out
        torch.cuda.synchronize()
        return outs

    ref = chain(True)
    for _ in range(3):
        got = chain(False)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    assert moe.moe_read_device_error(ws) == 0
