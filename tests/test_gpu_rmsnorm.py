"""GPU parity of moe_forward_rmsnorm (pre-router RMSNorm + MoE block + residual) against
the oracle, on the fused decode path (T <= 64: the norm inside the router launch) and the
unfused path (a separate norm launch ahead of the tensor-core router)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth

pytestmark = pytest.mark.gpu

import top_routing_grouped_router_gb300 as moe  # noqa: E402
from top_routing_grouped_router_gb300.device import bf16_tensor_bits, to_device, upload  # noqa: E402
from parity import NEAR_TIE, rel_err, sample_tokens, to_f64  # noqa: E402

EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_routing_grouped_router_gb300 import build
    build.build()
    oracle.build()


def _run(inp, gamma, residual):
    L = upload(inp)
    g = to_device(gamma, "cuda")
    ws = L.new_workspace()
    T, H, k = inp.T, inp.H, inp.k
    dt = L.out_dtype()
    out = torch.empty((T, H), dtype=dt, device="cuda")
    xn = torch.empty((T, H), dtype=dt, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    moe.moe_forward_rmsnorm(L.shape, L.x, g, EPS, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, out,
                            add_residual=residual, x_norm_out=xn, expert_ids_out=ids, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_error(ws) == 0
    return L, ws, out, xn, ids


def _check(inp, full_oracle):
    gamma = synth.make_norm_weight(inp.H, inp.act, seed=inp.T)
    L, ws, out, xn, ids = _run(inp, gamma, residual=True)
    T, k = inp.T, inp.k
    # the normalised activations: the GPU rounds its fp32 value once, the oracle its double
    # value; a rounding boundary between the two can move an element by one unit in the
    # last place (bf16) or a few fp32 ulps
    xn_ref = oracle.rmsnorm(inp.x, gamma, EPS, inp.act)
    if inp.act == "bf16":
        got_bits = bf16_tensor_bits(xn).astype(np.int32)
        ref_bits = oracle.round_bf16(xn_ref).astype(np.int32)
        d = np.abs(got_bits - ref_bits)
        assert d.max() <= 1 and (d > 0).mean() < 1e-3, (d.max(), (d > 0).mean())
    else:
        np.testing.assert_allclose(xn.cpu().numpy(), xn_ref, rtol=2e-6, atol=1e-7)

    toks = np.arange(T) if full_oracle else sample_tokens(T, 12)
    if full_oracle:
        ref = oracle.forward_prenorm(inp, gamma, EPS, residual=True)
        o_out, o_ids, margin = ref["out"], ref["ids"], ref["tie_margin"]
    else:
        ref = oracle.forward_prenorm_tokens(inp, gamma, EPS, toks, residual=True)
        o_out, o_ids, margin = ref["out"], ref["ids"], ref["tie_margin"]
    keep = margin >= NEAR_TIE
    g_ids = ids.cpu().numpy()[toks]
    np.testing.assert_array_equal(np.sort(g_ids[keep], axis=1), np.sort(o_ids[keep], axis=1))
    g_out = to_f64(out)[toks]
    tol = 1e-5 if inp.act == "f32" else 1e-2
    assert rel_err(g_out[keep], o_out[keep]) <= tol

    # after the norm the block is moe_forward on xn: bit-identical without the residual
    _, _, out_nr, xn2, _ = _run(inp, gamma, residual=False)
    assert torch.equal(xn2, xn)
    ref_out = torch.empty_like(out_nr)
    ws2 = L.new_workspace()
    moe.moe_forward(L.shape, xn, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, ref_out, workspace=ws2)
    torch.cuda.synchronize()
    assert torch.equal(out_nr, ref_out)
    # and the residual is added before the single rounding
    hs = to_f64(L.x)
    d = np.abs(to_f64(out) - (hs + to_f64(out_nr)))
    scale = np.abs(hs + to_f64(out_nr)).max()
    assert d.max() <= (1e-6 if inp.act == "f32" else 8e-3) * scale


def test_rmsnorm_fused_decode_bf16():
    _check(synth.make_inputs("decode8"), full_oracle=True)


def test_rmsnorm_fused_decode_fp32_tiny():
    _check(synth.make_inputs("tiny"), full_oracle=True)


def test_rmsnorm_separate_launch_large_batch():
    _check(synth.make_custom(200, 1024, 64, 8, 512, seed=21, name="norm200"), full_oracle=False)


def test_rmsnorm_fused_decode_q4():
    _check(synth.make_inputs("decode48q"), full_oracle=False)
