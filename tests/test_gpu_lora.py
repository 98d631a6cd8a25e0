"""GPU parity of moe_forward_lora (LoRA adapters on the expert projections) against the
oracle, on the bf16 and 4-bit tensor-core paths (decode and large batches) and the
generic fp32 path; on the bf16 and 4-bit paths both with the fp32 adapters as given
(CUDA-core adapter products) and with a pack (tensor-core adapter products).  With B = 0 the result
must equal moe_forward bit for bit, which also checks the split launches the adapters
need."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth

pytestmark = pytest.mark.gpu

import top_routing_grouped_router_gb300 as moe  # noqa: E402
from top_routing_grouped_router_gb300.device import to_device, upload  # noqa: E402
from parity import NEAR_TIE, rel_err, sample_tokens, to_f64  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_routing_grouped_router_gb300 import build
    build.build()
    oracle.build()


_NAMES = ("a_gate", "b_gate", "a_up", "b_up", "a_down", "b_down")


def _dev_lora(lora, shape=None):
    t = {n: to_device(np.ascontiguousarray(lora[n], dtype=np.float32), "cuda") for n in _NAMES}
    s = moe.make_lora(lora["rank"], lora["scale"], *[t[n] for n in _NAMES])
    if shape is not None:
        s = moe.pack_lora(shape, s)
        t["pack"] = s.pack_tensor
    return s, t


def _run_lora(L, lora_s):
    ws = L.new_workspace()
    out = torch.empty((L.shape.T, L.shape.H), dtype=L.out_dtype(), device="cuda")
    ids = torch.empty((L.shape.T, L.shape.k), dtype=torch.int32, device="cuda")
    moe.moe_forward_lora(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, lora_s, out, ids,
                         workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_error(ws) == 0
    return out, ids


def _check(inp, rank, n_tok, packed=False):
    lora = synth.make_lora(inp.E, inp.H, inp.I, rank=rank, seed=inp.T + rank)
    L = upload(inp)
    lora_s, keep_alive = _dev_lora(lora, L.shape if packed else None)
    out, ids = _run_lora(L, lora_s)
    toks = np.arange(inp.T) if n_tok is None else sample_tokens(inp.T, n_tok)
    ref = oracle.forward_lora(inp, lora, toks)
    keep = ref["tie_margin"] >= NEAR_TIE
    g_ids = ids.cpu().numpy()[toks]
    np.testing.assert_array_equal(np.sort(g_ids[keep], axis=1), np.sort(ref["ids"][keep], axis=1))
    tol = 1e-5 if inp.act == "f32" else 1e-2
    err = rel_err(to_f64(out)[toks][keep], ref["out"][keep])
    assert err <= tol, err
    # the adapters matter: the base block differs from the LoRA result by more than the tolerance
    base = oracle.forward_tokens(inp, toks)["out"]
    assert rel_err(base[keep], ref["out"][keep]) > 5 * tol

    # B = 0: bit-identical to moe_forward (same tiles, same rounding; gate/up and down split)
    zero = dict(lora)
    for n in ("b_gate", "b_up", "b_down"):
        zero[n] = np.zeros_like(lora[n])
    zs, keep_alive2 = _dev_lora(zero, L.shape if packed else None)
    out0, ids0 = _run_lora(L, zs)
    ref0 = torch.empty_like(out0)
    ids_ref = torch.empty_like(ids0)
    moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, ref0, ids_ref,
                    workspace=L.new_workspace())
    torch.cuda.synchronize()
    assert torch.equal(ids0, ids_ref)
    assert torch.equal(out0.view(torch.int16) if out0.dtype == torch.bfloat16 else out0,
                       ref0.view(torch.int16) if ref0.dtype == torch.bfloat16 else ref0)


def test_lora_decode_bf16_rank16():
    _check(synth.make_inputs("decode8"), 16, None)


def test_lora_packed_decode_bf16_rank16():
    _check(synth.make_inputs("decode8"), 16, None, packed=True)


def test_lora_packed_mid_batch_bf16_rank7():
    # 64 tokens: 128-token tiles, two-slab down tiles, A-side tiles of partial chunks
    _check(synth.make_custom(64, 1024, 32, 4, 256, seed=45, name="lora64"), 7, 16, packed=True)


def test_lora_packed_single_token_rank1():
    # one token, rank 1: A-side tiles of a single row, the rest of each tile padding
    _check(synth.make_custom(1, 256, 8, 2, 128, seed=53, name="lora1"), 1, None, packed=True)


def test_lora_pack_is_ignored_off_the_bf16_path():
    # a pack passed with fp32 weights changes nothing: the fp32 path keeps fp32 adapters
    inp = synth.make_inputs("tiny")
    lora = synth.make_lora(inp.E, inp.H, inp.I, rank=4, seed=7)
    L = upload(inp)
    plain, keep = _dev_lora(lora)
    packed, keep2 = _dev_lora(lora, L.shape)
    a, _ = _run_lora(L, plain)
    b, _ = _run_lora(L, packed)
    assert torch.equal(a, b)


def test_lora_packed_large_batch_bf16_rank16():
    # 2048 assignments over 16 experts (128 per expert on average): 256-token gate/up tiles
    _check(synth.make_custom(512, 1024, 16, 4, 384, seed=51, name="lora512"), 16, 16, packed=True)


def test_lora_decode_q4_rank16():
    _check(synth.make_inputs("decode48q"), 16, 12)


def test_lora_packed_decode_q4_rank16():
    # 4-bit decode with a pack: A-side products on the tensor cores from the grouped-order rows
    _check(synth.make_inputs("decode48q"), 16, 12, packed=True)


def test_lora_packed_q4_odd_row_blocks_rank5():
    # H = 384: an odd count of 128-row blocks (a 128-row down tile at the end of each expert)
    _check(synth.make_custom(40, 384, 16, 4, 256, w="q4", seed=47, name="lora40q"), 5, 16, packed=True)


def test_lora_packed_large_batch_q4_rank16():
    _check(synth.make_custom(200, 256, 16, 4, 128, w="q4", seed=43, name="lora200q"), 16, 16, packed=True)


def test_lora_fp32_generic_path_rank4():
    _check(synth.make_inputs("tiny"), 4, None)


def test_lora_large_batch_bf16_rank8():
    _check(synth.make_custom(300, 512, 16, 4, 256, seed=41, name="lora300"), 8, 16)


def test_lora_packed_large_batch_bf16_rank8():
    _check(synth.make_custom(300, 512, 16, 4, 256, seed=41, name="lora300"), 8, 16, packed=True)


def test_lora_large_batch_q4_rank16():
    _check(synth.make_custom(200, 256, 16, 4, 128, w="q4", seed=43, name="lora200q"), 16, 16)


def test_pack_layout_is_the_documented_hi_lo_split():
    # the pack's bytes against the layout moe.h documents, built here from the fp32 adapters:
    # hi = bf16(v), lo = bf16(v - hi) (nearest even), rows / columns past the rank zero
    E, H, I, r = 4, 128, 128, 5
    shape = moe.make_shape(8, H, E, 2, I)
    lora = synth.make_lora(E, H, I, rank=r, seed=3)
    s, keep = _dev_lora(lora, shape)
    got = s.pack_tensor.cpu().numpy().view(np.uint16)

    def split(v):
        v = np.asarray(v, dtype=np.float32)
        hi = synth.bf16_bits(v)
        lo = synth.bf16_bits(v - synth.bf16_bits_to_f32(hi))
        return hi, lo

    al = lambda b: (b + 255) // 256 * 256
    off_ah = al(E * 64 * H * 2) // 2
    off_bgu = off_ah + al(E * 32 * I * 2) // 2
    off_bd = off_bgu + al(E * I * 128 * 2) // 2
    ax = np.zeros((E, 64, H), np.uint16)
    ah = np.zeros((E, 32, I), np.uint16)
    bgu = np.zeros((E * I, 128), np.uint16)
    bd = np.zeros((E * H, 64), np.uint16)
    for name, base in (("a_gate", 0), ("a_up", 16)):
        hi, lo = split(lora[name])  # [E][r][H]
        ax[:, base:base + r] = hi
        ax[:, 32 + base:32 + base + r] = lo
    hi, lo = split(lora["a_down"])
    ah[:, :r] = hi
    ah[:, 16:16 + r] = lo
    for name, col in (("b_gate", 0), ("b_up", 64)):
        hi, lo = split(lora[name].reshape(E * I, r))
        bgu[:, col:col + r] = hi
        bgu[:, col + 16:col + 16 + r] = hi
        bgu[:, col + 32:col + 32 + r] = lo
    hi, lo = split(lora["b_down"].reshape(E * H, r))
    bd[:, :r] = hi
    bd[:, 16:16 + r] = hi
    bd[:, 32:32 + r] = lo
    np.testing.assert_array_equal(got[:E * 64 * H].reshape(ax.shape), ax)
    np.testing.assert_array_equal(got[off_ah:off_ah + E * 32 * I].reshape(ah.shape), ah)
    np.testing.assert_array_equal(got[off_bgu:off_bgu + E * I * 128].reshape(bgu.shape), bgu)
    np.testing.assert_array_equal(got[off_bd:off_bd + E * H * 64].reshape(bd.shape), bd)


def test_pack_for_4bit_weights_keeps_the_grouped_column_order():
    # with 4-bit weights the pack's A columns follow the 4-bit path's order of x and h: stored
    # position p of every 8-column group holds column (0,4,1,5,2,6,3,7)[p]; the B slabs are
    # those of the bf16 pack
    E, H, I, r = 4, 128, 128, 5
    lora = synth.make_lora(E, H, I, rank=r, seed=3)
    plain, keep = _dev_lora(lora, moe.make_shape(8, H, E, 2, I))
    grouped, keep2 = _dev_lora(lora, moe.make_shape(8, H, E, 2, I, w="q4", q_block=64))
    a = plain.pack_tensor.cpu().numpy().view(np.uint16)
    b = grouped.pack_tensor.cpu().numpy().view(np.uint16)
    assert a.shape == b.shape
    al = lambda n: (n + 255) // 256 * 256
    n_ax, n_ah = E * 64 * H, E * 32 * I
    off_ah = al(n_ax * 2) // 2
    order = np.array([0, 4, 1, 5, 2, 6, 3, 7])
    perm = lambda n: (np.arange(n).reshape(-1, 8)[:, order]).reshape(-1)
    np.testing.assert_array_equal(b[:n_ax].reshape(E * 64, H), a[:n_ax].reshape(E * 64, H)[:, perm(H)])
    np.testing.assert_array_equal(b[off_ah:off_ah + n_ah].reshape(E * 32, I),
                                  a[off_ah:off_ah + n_ah].reshape(E * 32, I)[:, perm(I)])
    off_bgu = off_ah + al(n_ah * 2) // 2
    np.testing.assert_array_equal(b[off_bgu:], a[off_bgu:])
