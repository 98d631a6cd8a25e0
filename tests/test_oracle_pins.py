"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against a hand-derived worked example (tests/golden),
a closed form, an invariant, a brute-force formulation or an independent library
routine (numpy matmul, numpy stable argsort, scipy softmax), chosen so that a
plausible slip anywhere in the oracle (a dropped bias, a wrong SiLU sign, a
transposed operand, a wrong nibble, an unstable sort, a missing renormalisation,
a wrong tie-break) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth


def _inputs_from_json(d):
    s = d["shape"]
    f = lambda a: np.ascontiguousarray(np.array(a, dtype=np.float32))
    return synth.MoEInputs(name="golden", T=s["T"], H=s["H"], E=s["E"], k=s["k"], I=s["I"], act="f32", w="f32",
                           norm_topk=s["norm_topk"], q_block=64, x=f(d["x"]), w_router=f(d["w_router"]),
                           b_router=None, w_gate=f(d["w_gate"]), w_up=f(d["w_up"]), w_down=f(d["w_down"]))


def _x64(inp):
    return synth.bf16_bits_to_f32(inp.x).astype(np.float64) if inp.act == "bf16" else inp.x.astype(np.float64)


def _w64(inp, a):
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def _silu(z):
    return z / (1.0 + np.exp(-z))


# ---------------------------------------------------------------- golden worked examples

def test_golden_worked_example_full_block(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "worked_routing_expert.json")))
    inp = _inputs_from_json(d)
    r = oracle.forward(inp)
    ex = d["expect"]
    np.testing.assert_array_equal(r["logits"], ex["logits"])
    np.testing.assert_array_equal(r["ids"], ex["ids"])
    np.testing.assert_allclose(r["weights"], ex["weights"], rtol=1e-15)
    np.testing.assert_array_equal(r["tie_margin"], ex["tie_margin"])
    for name in ("counts", "offsets", "order", "pos"):
        np.testing.assert_array_equal(r[name], ex[name])
    for e, yv in ex["y_by_expert"].items():
        _, y = oracle.expert_mlp(inp, np.array([1.0]), int(e))
        assert y[0] == pytest.approx(yv, rel=1e-15, abs=1e-300)
    np.testing.assert_allclose(r["out"], ex["out"], rtol=1e-15)


def test_golden_permutations(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "worked_permutation.json")))
    for c in d["cases"]:
        counts, offsets, order, pos = oracle.permute(np.array(c["ids"], np.int32), c["E"])
        for name, got in (("counts", counts), ("offsets", offsets), ("order", order), ("pos", pos)):
            np.testing.assert_array_equal(got, c[name], err_msg=f"{c['name']}:{name}")


def test_golden_q4_decoding(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "worked_q4_decode.json")))
    rows, cols, qb = d["rows"], d["cols"], d["q_block"]
    codes = np.zeros((1, rows, cols // 2), np.uint8)
    for b, v in d["bytes"].items():
        codes[0, 0, int(b)] = v
    scales = np.array(d["scales_bf16_bits"], np.uint16).reshape(1, rows, cols // qb)
    z = np.zeros((1, 1), np.float32)
    inp = synth.MoEInputs(name="q4", T=1, H=cols, E=1, k=1, I=rows, act="f32", w="q4", norm_topk=True,
                          q_block=qb, x=z, w_router=z, b_router=None, w_gate=codes, w_up=codes,
                          w_down=np.zeros((1, cols, rows // 2 if rows > 1 else 1), np.uint8),
                          gate_scales=scales, up_scales=scales, down_scales=scales,
                          codebook=synth.uniform_codebook16())
    for item in d["expect"]:
        assert oracle.weight_at(inp, "gate", 0, 0, item["col"]) == pytest.approx(item["value"], rel=1e-15)


# ---------------------------------------------------------------- step A: router logits

@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_router_logits_equal_numpy_matmul_with_bias(act):
    inp = synth.make_custom(7, 40, 6, 2, 12, act=act, w="f32", zipf=True, seed=11)
    got = oracle.router_logits(inp)
    want = _x64(inp) @ _w64(inp, inp.w_router).T + inp.b_router.astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- step B: softmax, top-k, renormalise

def test_topk_equals_full_sort_prefix():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((50, 16))
    ids, w, m = oracle.select_topk(logits, 5)
    for t in range(50):
        full = sorted(range(16), key=lambda e: (-logits[t, e], e))
        assert list(ids[t]) == full[:5]
        assert m[t] == logits[t, full[4]] - logits[t, full[5]]


def test_topk_ties_prefer_lower_index_and_report_zero_margin():
    logits = np.array([[0.5, 2.0, 2.0, 1.0, 2.0, -1.0]])
    ids, w, m = oracle.select_topk(logits, 2)
    assert list(ids[0]) == [1, 2]
    assert m[0] == 0.0
    np.testing.assert_allclose(w[0], [0.5, 0.5], rtol=1e-15)


def test_weights_sum_to_one_and_descend():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((64, 32)) * 3
    ids, w, _ = oracle.select_topk(logits, 8)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_k_equals_E_is_full_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((9, 8)) * 4
    ids, w, m = oracle.select_topk(logits, 8)
    full = scipy_special.softmax(logits, axis=1)
    for t in range(9):
        np.testing.assert_allclose(w[t], full[t, ids[t]], rtol=1e-13)
        assert sorted(ids[t]) == list(range(8))
    assert np.all(np.isinf(m))


def test_no_renorm_k1_is_max_softmax_probability():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((12, 10))
    ids, w, _ = oracle.select_topk(logits, 1, norm_topk=False)
    full = scipy_special.softmax(logits, axis=1)
    np.testing.assert_array_equal(ids[:, 0], logits.argmax(axis=1))
    np.testing.assert_allclose(w[:, 0], full.max(axis=1), rtol=1e-13)


def test_no_renorm_weights_are_softmax_entries():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((5, 12))
    ids, w, _ = oracle.select_topk(logits, 3, norm_topk=False)
    full = scipy_special.softmax(logits, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, ids.astype(np.int64), axis=1), rtol=1e-13)


# ---------------------------------------------------------------- steps C, D: histogram, scan, permutation

@pytest.mark.parametrize("A,E,seed", [(0, 4, 0), (1, 4, 1), (64, 128, 2), (512, 128, 3), (3000, 8, 4)])
def test_permutation_matches_stable_argsort_and_bincount(A, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, A).astype(np.int32)
    counts, offsets, order, pos = oracle.permute(ids, E)
    np.testing.assert_array_equal(counts, np.bincount(ids, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == A
    np.testing.assert_array_equal(offsets[1:], np.cumsum(counts))
    np.testing.assert_array_equal(order, np.argsort(ids, kind="stable"))
    np.testing.assert_array_equal(np.sort(order), np.arange(A))
    np.testing.assert_array_equal(pos[order], np.arange(A))
    assert np.all(np.diff(ids[order]) >= 0)


def test_permutation_rejects_out_of_range_ids():
    with pytest.raises(RuntimeError):
        oracle.permute(np.array([0, 5], np.int32), 4)


# ---------------------------------------------------------------- steps E, F: expert SwiGLU MLP

def test_expert_closed_form_one_dim():
    # H = I = 1: y = SiLU(a x) * (b x) * c
    for a, b, c, x in [(0.7, -1.3, 2.0, 1.5), (-2.0, 0.5, -0.25, 3.0), (0.0, 4.0, 1.0, 2.0), (30.0, 1.0, 1.0, 1.0)]:
        w = lambda v: np.array([[[v]]], np.float32)
        inp = synth.MoEInputs(name="cf", T=1, H=1, E=1, k=1, I=1, act="f32", w="f32", norm_topk=True,
                              q_block=64, x=w(x)[0], w_router=w(0.0)[0], b_router=None,
                              w_gate=w(a), w_up=w(b), w_down=w(c))
        g = float(np.float32(a)) * float(np.float32(x))
        want = g / (1.0 + math.exp(-g)) * (float(np.float32(b)) * float(np.float32(x))) * float(np.float32(c))
        _, y = oracle.expert_mlp(inp, np.array([float(np.float32(x))]), 0)
        assert y[0] == pytest.approx(want, rel=1e-14, abs=1e-300)


@pytest.mark.parametrize("act,wdt", [("f32", "f32"), ("bf16", "bf16")])
def test_sparse_block_equals_dense_numpy_brute_force(act, wdt):
    # all E experts for every token with numpy matmuls (non-square H != I), masked by the top-k weights
    inp = synth.make_custom(11, 24, 5, 2, 10, act=act, w=wdt, seed=21)
    r = oracle.forward(inp)
    X = _x64(inp)
    logits = X @ _w64(inp, inp.w_router).T
    mask = np.zeros((inp.T, inp.E))
    for t in range(inp.T):
        order = sorted(range(inp.E), key=lambda e: (-logits[t, e], e))[: inp.k]
        p = np.exp(logits[t] - logits[t].max())
        p /= p.sum()
        mask[t, order] = p[order] / p[order].sum()
    dense = np.zeros((inp.T, inp.H))
    for e in range(inp.E):
        G = X @ _w64(inp, inp.w_gate[e]).T
        U = X @ _w64(inp, inp.w_up[e]).T
        Y = (_silu(G) * U) @ _w64(inp, inp.w_down[e]).T
        dense += mask[:, e:e + 1] * Y
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_sparse_equals_oracle_dense_masked_brute_force():
    inp = synth.make_inputs("tiny")
    sparse = oracle.forward(inp)["out"]
    dense = oracle.forward_dense(inp)
    assert np.abs(sparse - dense).max() <= 1e-12 * np.abs(dense).max()


def test_forward_tokens_equals_full_forward_rows():
    inp = synth.make_custom(13, 32, 6, 3, 8, act="bf16", w="bf16", zipf=True, seed=5)
    r = oracle.forward(inp)
    toks = [0, 5, 12, 7]
    s = oracle.forward_tokens(inp, toks)
    np.testing.assert_array_equal(s["ids"], r["ids"][toks])
    np.testing.assert_allclose(s["out"], r["out"][toks], rtol=1e-13, atol=1e-15)


def test_single_expert_top1_is_plain_swiglu_mlp():
    inp = synth.make_custom(6, 16, 1, 1, 12, act="f32", w="f32", seed=8)
    r = oracle.forward(inp)
    X = _x64(inp)
    want = (_silu(X @ _w64(inp, inp.w_gate[0]).T) * (X @ _w64(inp, inp.w_up[0]).T)) @ _w64(inp, inp.w_down[0]).T
    np.testing.assert_allclose(r["weights"], 1.0)
    np.testing.assert_allclose(r["out"], want, rtol=1e-13, atol=1e-14)


def test_zero_up_projection_gives_zero_output():
    inp = synth.make_custom(5, 16, 4, 2, 8, act="f32", w="f32", seed=9)
    inp.w_up = np.zeros_like(inp.w_up)
    assert np.all(oracle.forward(inp)["out"] == 0.0)


def test_unpermute_is_weighted_gather():
    rng = np.random.default_rng(10)
    T, k, H = 4, 3, 5
    ids = rng.integers(0, 3, (T, k)).astype(np.int32)
    _, _, order, pos = oracle.permute(ids, 3)
    y = rng.standard_normal((T * k, H))
    w = rng.random((T, k))
    out = oracle.unpermute(y, w, pos, T, k)
    want = np.stack([sum(w[t, j] * y[pos[t * k + j]] for j in range(k)) for t in range(T)])
    np.testing.assert_allclose(out, want, rtol=1e-15)


# ---------------------------------------------------------------- 4-bit weights

def test_q4_roundtrip_error_bound_and_extremes():
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((6, 128)) * 0.05).astype(np.float32)
    cb = synth.uniform_codebook16()
    codes, scales = synth.quantize_q4_rows(w, cb, 64)
    z = np.zeros((1, 1), np.float32)
    inp = synth.MoEInputs(name="q4", T=1, H=128, E=1, k=1, I=6, act="f32", w="q4", norm_topk=True, q_block=64,
                          x=z, w_router=z, b_router=None, w_gate=codes[None], w_up=codes[None],
                          w_down=np.zeros((1, 128, 3), np.uint8), gate_scales=scales[None],
                          up_scales=scales[None], down_scales=np.zeros((1, 128, 1), np.uint16), codebook=cb)
    s = synth.bf16_bits_to_f32(scales).astype(np.float64)
    for r in range(6):
        for c in range(128):
            got = oracle.weight_at(inp, "gate", 0, r, c)
            assert abs(got - w[r, c]) <= s[r, c // 64] / 15.0 * (1 + 1e-6)
        for b in range(2):
            blk = np.abs(w[r, 64 * b:64 * (b + 1)])
            c = 64 * b + int(blk.argmax())
            nib = (codes[r, c // 2] >> (4 * (c & 1))) & 15
            assert nib == (15 if w[r, c] > 0 else 0)


def test_q4_block_oracle_matches_dequantised_dense():
    inp = synth.make_custom(4, 128, 3, 2, 64, act="bf16", w="q4", seed=13)
    r = oracle.forward(inp)

    def deq(codes, scales):
        lo, hi = codes & 15, codes >> 4
        c = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.int64)
        c[..., 0::2], c[..., 1::2] = lo, hi
        s = np.repeat(synth.bf16_bits_to_f32(scales).astype(np.float64), 64, axis=-1)
        return inp.codebook.astype(np.float64)[c] * s

    Wg, Wu, Wd = deq(inp.w_gate, inp.gate_scales), deq(inp.w_up, inp.up_scales), deq(inp.w_down, inp.down_scales)
    X = _x64(inp)
    out = np.zeros((inp.T, inp.H))
    for t in range(inp.T):
        for j in range(inp.k):
            e = r["ids"][t, j]
            y = (_silu(Wg[e] @ X[t]) * (Wu[e] @ X[t])) @ Wd[e].T
            out[t] += r["weights"][t, j] * y
    np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- input recipe properties the tests rely on

def test_zipf_workload_leaves_experts_empty_and_is_skewed():
    inp = synth.make_custom(64, 256, 128, 8, 8, act="bf16", w="bf16", zipf=True, seed=2)
    counts = np.bincount(oracle.select_topk(oracle.router_logits(inp), 8)[0].reshape(-1), minlength=128)
    assert (counts == 0).sum() >= 1
    assert counts.max() >= 32


def test_bf16_widening_is_exact():
    vals = np.array([1.0, -2.5, 3.140625, 1e-30, -65280.0], np.float32)
    bits = synth.bf16_bits(vals)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(bits)[[0, 1, 2, 4]], vals[[0, 1, 2, 4]])
    z = np.zeros((1, 1), np.float32)
    x = bits[:1].reshape(1, 1)
    inp = synth.MoEInputs(name="b", T=1, H=1, E=1, k=1, I=1, act="bf16", w="f32", norm_topk=True, q_block=64,
                          x=x, w_router=synth.bf16_bits(np.array([[3.140625]], np.float32)), b_router=None,
                          w_gate=z[None], w_up=z[None], w_down=z[None])
    assert oracle.router_logits(inp)[0, 0] == 3.140625


# ---------------------------------------------------------------- pre-router RMSNorm

def test_rmsnorm_worked_example(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "worked_rmsnorm.json")))
    hs = np.array(d["hs"], dtype=np.float32)
    for r, gamma in enumerate(d["gamma_rows"]):
        xn = oracle.rmsnorm(hs[r:r + 1], np.array(gamma, dtype=np.float32), d["eps"], "f32")
        np.testing.assert_allclose(xn[0], d["expect"][r], rtol=1e-15, atol=0)


def test_rmsnorm_is_scale_invariant_and_unit_rms():
    rng = np.random.default_rng(5)
    hs = rng.standard_normal((3, 96)).astype(np.float32)
    gamma = np.ones(96, dtype=np.float32)
    a = oracle.rmsnorm(hs, gamma, 0.0, "f32")
    b = oracle.rmsnorm((hs * np.float32(4.0)).astype(np.float32), gamma, 0.0, "f32")  # exact power-of-2 scale
    np.testing.assert_allclose(a, b, rtol=1e-15, atol=0)
    np.testing.assert_allclose((a ** 2).mean(axis=1), 1.0, rtol=1e-13)
    # gamma scales each column; a zero row stays zero with eps > 0
    g2 = rng.uniform(0.5, 1.5, 96).astype(np.float32)
    np.testing.assert_allclose(oracle.rmsnorm(hs, g2, 0.0, "f32"), a * g2.astype(np.float64), rtol=1e-14)
    z = oracle.rmsnorm(np.zeros((1, 96), np.float32), g2, 1e-6, "f32")
    assert np.all(z == 0)
    # eps enters under the root: a row of ones with eps = 3 gives 1 / sqrt(1 + 3) = 0.5
    np.testing.assert_allclose(oracle.rmsnorm(np.ones((1, 8), np.float32), np.ones(8, np.float32), 3.0, "f32"), 0.5,
                               rtol=1e-15)


def test_round_bf16_is_nearest_even_from_double():
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30, -1.5, 0.0, 3.0 * 2 ** -20, 1 - 2 ** -10])
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even mantissa -> 1; 1 + 3*2^-8 -> 1 + 2^-6 (even);
    # just above a half rounds up; 1 - 2^-10 rounds up to 1
    assert oracle.round_bf16(v).tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xBFC0, 0x0000, 0x3640, 0x3F80]
    # away from ties it agrees with fp32 rounding followed by bf16 rounding
    w = np.random.default_rng(6).standard_normal(1000)
    np.testing.assert_array_equal(oracle.round_bf16(w), synth.bf16_bits(w.astype(np.float32)))


def test_prenorm_block_with_one_hidden_unit_has_a_closed_form():
    # H = 1: RMSNorm(h) * gamma = sign(h) * gamma (eps = 0), so with one expert (E = k = 1,
    # weight 1) and I = 1, out = h + SiLU(a x) * (b x) * c with x = sign(h) * gamma
    inp = synth.MoEInputs(name="h1", T=2, H=1, E=1, k=1, I=1, act="f32", w="f32", norm_topk=True, q_block=64,
                          x=np.array([[-0.75], [2.5]], np.float32), w_router=np.array([[1.0]], np.float32),
                          b_router=None, w_gate=np.array([[[0.625]]], np.float32), w_up=np.array([[[1.5]]], np.float32),
                          w_down=np.array([[[-2.0]]], np.float32))
    gamma = np.array([1.25], np.float32)
    r = oracle.forward_prenorm(inp, gamma, 0.0, residual=True)
    for t, h in enumerate([-0.75, 2.5]):
        x = math.copysign(1.25, h)
        expect = h + (0.625 * x / (1 + math.exp(-0.625 * x))) * (1.5 * x) * (-2.0)
        assert abs(r["out"][t, 0] - expect) < 1e-12
    r0 = oracle.forward_prenorm(inp, gamma, 0.0, residual=False)
    np.testing.assert_allclose(r["out"] - r0["out"], inp.x.astype(np.float64), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- LoRA on the experts

def _lora_zero_b(l):
    z = dict(l)
    for n in ("b_gate", "b_up", "b_down"):
        z[n] = np.zeros_like(l[n])
    return z


def test_lora_with_zero_b_is_the_base_block():
    inp = synth.make_custom(6, 64, 8, 2, 32, act="f32", w="f32", seed=31)
    lora = _lora_zero_b(synth.make_lora(8, 64, 32, rank=4, seed=1))
    a = oracle.forward_lora(inp, lora)
    b = oracle.forward_tokens(inp, np.arange(6))
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["ids"], b["ids"])


def test_lora_equals_the_merged_weights():
    # integer-valued weights and adapters with scale 1/2: W + scale * B A is exact in fp32, so the
    # oracle on merged weights (a plain numpy matmul builds them) must agree to double rounding;
    # a transposed A or B, a wrong scale or an adapter on the wrong projection would not
    rng = np.random.default_rng(7)
    E, H, I, r, T, k = 4, 16, 8, 3, 5, 2
    ints = lambda *sh: rng.integers(-2, 3, size=sh).astype(np.float32)
    inp = synth.MoEInputs(name="lora", T=T, H=H, E=E, k=k, I=I, act="f32", w="f32", norm_topk=True, q_block=64,
                          x=(ints(T, H) / 4).astype(np.float32), w_router=ints(E, H), b_router=None,
                          w_gate=ints(E, I, H), w_up=ints(E, I, H), w_down=ints(E, H, I))
    lora = dict(rank=r, scale=0.5, a_gate=ints(E, r, H), b_gate=ints(E, I, r), a_up=ints(E, r, H),
                b_up=ints(E, I, r), a_down=ints(E, r, I), b_down=ints(E, H, r))
    merged = synth.MoEInputs(**{**inp.__dict__})
    merged.w_gate = (inp.w_gate + 0.5 * np.matmul(lora["b_gate"], lora["a_gate"])).astype(np.float32)
    merged.w_up = (inp.w_up + 0.5 * np.matmul(lora["b_up"], lora["a_up"])).astype(np.float32)
    merged.w_down = (inp.w_down + 0.5 * np.matmul(lora["b_down"], lora["a_down"])).astype(np.float32)
    a = oracle.forward_lora(inp, lora)
    b = oracle.forward_tokens(merged, np.arange(T))
    np.testing.assert_array_equal(a["ids"], b["ids"])
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-12, atol=1e-12 * np.abs(b["out"]).max())
    # and the adapters do change the result
    c = oracle.forward_tokens(inp, np.arange(T))
    assert np.abs(c["out"] - a["out"]).max() > 1e-3
