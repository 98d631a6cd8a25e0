"""Seeded synthetic inputs for the sparse Mixture-of-Experts block.

This module only *draws* inputs: activations, router weights, router bias and
expert weights, in the storage formats the MoE block consumes (fp32, bf16 bit
patterns, or 4-bit codes with bf16 block scales).  It holds none of the block's
arithmetic: no routing, no softmax, no expert MLP, no dequantisation.  Both the
CPU oracle and the CUDA path read the arrays produced here, and nothing else is
shared between them.

Workloads (all Qwen3-30B-A3B-style MoE layers, hidden H, E experts, top-k,
expert intermediate I; "N(0, 1/fan_in)" means std = 1/sqrt(fan_in) with
fan_in = H for the router, gate and up projections and I for the down
projection):

* ``tiny``      T=16, H=64, E=8, k=2, I=32, fp32 everywhere.
* ``decode8``   T=8, H=2048, E=128, k=8, I=768, bf16.
* ``decode64z`` T=64, same shape, bf16, with a router bias so that expert
                popularity follows Zipf(s=1.1) over a seeded permutation of the
                experts (skewed load, some experts empty).
* ``decode48q`` T=48, same shape, bf16 activations, expert weights as 4-bit
                codes into a 16-entry uniform codebook on [-1, 1] with one bf16
                absmax scale per 64 contiguous input-dim elements.
* ``prefill``   T=4096, same shape, bf16, four independent layers (separate
                weights and separate inputs).

Random numbers come from numpy's PCG64 seeded through ``SeedSequence`` with a
fixed word list per tensor (and per expert for expert weights), so every tensor
and every expert slab is reproducible on its own, on any host.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Optional

import numpy as np

__all__ = [
    "WORKLOADS", "MoEInputs", "make_inputs", "make_custom", "bf16_bits", "bf16_bits_to_f32",
    "uniform_codebook16", "quantize_q4_rows", "zipf_router_bias",
]

# name -> (T, H, E, k, I, act dtype, weight dtype, zipf bias, layers, seed)
WORKLOADS = {
    "tiny":      dict(T=16,   H=64,   E=8,   k=2, I=32,  act="f32",  w="f32",  zipf=False, layers=1, seed=0),
    "decode8":   dict(T=8,    H=2048, E=128, k=8, I=768, act="bf16", w="bf16", zipf=False, layers=1, seed=1),
    "decode64z": dict(T=64,   H=2048, E=128, k=8, I=768, act="bf16", w="bf16", zipf=True,  layers=1, seed=2),
    "decode48q": dict(T=48,   H=2048, E=128, k=8, I=768, act="bf16", w="q4",   zipf=False, layers=1, seed=3),
    "prefill":   dict(T=4096, H=2048, E=128, k=8, I=768, act="bf16", w="bf16", zipf=False, layers=4, seed=4),
    "prefill4q": dict(T=4096, H=2048, E=128, k=8, I=768, act="bf16", w="q4",   zipf=False, layers=1, seed=5),
}

_TENSOR_IDS = {"x": 1, "w_router": 2, "gate": 3, "up": 4, "down": 5, "perm": 6}
Q_BLOCK = 64
ZIPF_S = 1.1


def _rng(*words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(w) for w in words])))


def bf16_bits(f32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (round to nearest, ties to even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to fp32."""
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform_codebook16() -> np.ndarray:
    """The fixed 16-entry codebook: c_j = -1 + 2j/15 for j = 0..15 (uniform on [-1, 1], endpoints included)."""
    return np.array([-1.0 + 2.0 * j / 15.0 for j in range(16)], dtype=np.float32)


def quantize_q4_rows(w: np.ndarray, codebook: np.ndarray, q_block: int = Q_BLOCK):
    """Encode rows of fp32 weights [rows, cols] as 4-bit codes plus one bf16 absmax scale per block.

    Storage format (what the MoE block consumes):
      * scales[r, b] = bf16(max |w[r, b*q_block:(b+1)*q_block]|)
      * code = index j of the codebook entry nearest to w / scale (ties -> lower j;
      the codebook must be strictly increasing)
      * codes packed row-major [rows, cols/2] bytes, element 2i in the low nibble,
        element 2i+1 in the high nibble.
    """
    rows, cols = w.shape
    assert cols % q_block == 0 and cols % 2 == 0
    blocks = w.reshape(rows, cols // q_block, q_block)
    scale_bits = bf16_bits(np.abs(blocks).max(axis=2))
    scale = bf16_bits_to_f32(scale_bits).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    t = (blocks / safe[:, :, None]).reshape(rows, cols).astype(np.float32)
    cb = np.asarray(codebook, dtype=np.float64)
    assert np.all(np.diff(cb) > 0), "codebook must be strictly increasing"
    # nearest entry of a sorted codebook: count the midpoints strictly below t
    # (t exactly on a midpoint -> the lower entry)
    mids = (cb[:-1] + cb[1:]) / 2.0
    codes = np.searchsorted(mids, t.astype(np.float64), side="left").astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale_bits


def zipf_router_bias(E: int, seed: int, s: float = ZIPF_S) -> np.ndarray:
    """Router bias b[perm[r-1]] = ln(r^-s / sum_{r'} r'^-s) for popularity rank r = 1..E (fp32).

    perm is a seeded random permutation of the experts, so the most popular
    expert is not expert 0.
    """
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    perm = _rng(seed, _TENSOR_IDS["perm"]).permutation(E)
    b = np.empty(E, dtype=np.float64)
    b[perm] = np.log(p)
    return b.astype(np.float32)


@dataclasses.dataclass
class MoEInputs:
    """One MoE layer's inputs in storage form.

    x        [T, H]            fp32 or bf16 bits (uint16)
    w_router [E, H]            same dtype as x
    b_router [E] fp32 or None
    w_gate   [E, I, H]         fp32 / bf16 bits / q4 codes uint8 [E, I, H/2]
    w_up     [E, I, H]         same as w_gate
    w_down   [E, H, I]         fp32 / bf16 bits / q4 codes uint8 [E, H, I/2]
    *_scales bf16 bits [E, rows, in/q_block] (q4 only)
    codebook fp32[16] (q4 only)
    """
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    act: str
    w: str
    norm_topk: bool
    q_block: int
    x: np.ndarray
    w_router: np.ndarray
    b_router: Optional[np.ndarray]
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray
    gate_scales: Optional[np.ndarray] = None
    up_scales: Optional[np.ndarray] = None
    down_scales: Optional[np.ndarray] = None
    codebook: Optional[np.ndarray] = None
    seed: int = 0
    layer: int = 0

    @property
    def A(self) -> int:
        return self.T * self.k


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _normal_f32(shape, std: float, words) -> np.ndarray:
    out = _rng(*words).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def _expert_tensor(E, rows, cols, std, fmt, seed, layer, tid, codebook, q_block):
    """Draw E independent [rows, cols] slabs (one seed per expert) in the requested storage format."""
    if fmt == "f32":
        out = np.empty((E, rows, cols), dtype=np.float32)
    elif fmt == "bf16":
        out = np.empty((E, rows, cols), dtype=np.uint16)
    else:
        out = np.empty((E, rows, cols // 2), dtype=np.uint8)
        scales = np.empty((E, rows, cols // q_block), dtype=np.uint16)

    def one(e):
        w = _normal_f32((rows, cols), std, (seed, layer, tid, e))
        if fmt == "f32":
            out[e] = w
        elif fmt == "bf16":
            out[e] = bf16_bits(w)
        else:
            c, s = quantize_q4_rows(w, codebook, q_block)
            out[e] = c
            scales[e] = s

    if E * rows * cols >= (1 << 22):
        with _cf.ThreadPoolExecutor(_threads()) as pool:
            list(pool.map(one, range(E)))
    else:
        for e in range(E):
            one(e)
    return (out, scales) if fmt == "q4" else (out, None)


def make_custom(T, H, E, k, I, act="bf16", w="bf16", *, zipf=False, seed=0, layer=0,
                norm_topk=True, q_block=Q_BLOCK, name="custom") -> MoEInputs:
    """Draw one layer's inputs for an arbitrary shape with the standard recipe.

    x ~ N(0, 1); router, gate, up ~ N(0, 1/H); down ~ N(0, 1/I); fp32 values are
    rounded to bf16 (RNE) for bf16 storage, or encoded as 4-bit codes for q4.
    """
    assert act in ("f32", "bf16") and w in ("f32", "bf16", "q4")
    x = _normal_f32((T, H), 1.0, (seed, layer, _TENSOR_IDS["x"]))
    wr = _normal_f32((E, H), 1.0 / np.sqrt(H), (seed, layer, _TENSOR_IDS["w_router"]))
    if act == "bf16":
        x, wr = bf16_bits(x), bf16_bits(wr)
    b = zipf_router_bias(E, seed) if zipf else None
    cb = uniform_codebook16() if w == "q4" else None
    g, gs = _expert_tensor(E, I, H, 1.0 / np.sqrt(H), w, seed, layer, _TENSOR_IDS["gate"], cb, q_block)
    u, us = _expert_tensor(E, I, H, 1.0 / np.sqrt(H), w, seed, layer, _TENSOR_IDS["up"], cb, q_block)
    d, ds = _expert_tensor(E, H, I, 1.0 / np.sqrt(I), w, seed, layer, _TENSOR_IDS["down"], cb, q_block)
    return MoEInputs(name=name, T=T, H=H, E=E, k=k, I=I, act=act, w=w, norm_topk=norm_topk,
                     q_block=q_block, x=x, w_router=wr, b_router=b, w_gate=g, w_up=u, w_down=d,
                     gate_scales=gs, up_scales=us, down_scales=ds, codebook=cb, seed=seed, layer=layer)


def make_inputs(name: str, *, seed: Optional[int] = None, layer: int = 0, T: Optional[int] = None) -> MoEInputs:
    """Inputs of one named workload (one layer of it; ``layer`` selects the prefill stack member).

    ``T`` overrides the token count (same weights recipe), for reduced-size cases.
    """
    c = WORKLOADS[name]
    assert 0 <= layer < c["layers"]
    return make_custom(T if T is not None else c["T"], c["H"], c["E"], c["k"], c["I"], c["act"], c["w"],
                       zipf=c["zipf"], seed=c["seed"] if seed is None else seed, layer=layer, name=name)


def make_norm_weight(H: int, act: str = "bf16", seed: int = 0, layer: int = 0) -> np.ndarray:
    """Synthetic RMSNorm weight gamma [H]: 1 + 0.1 N(0, 1), in the activation's storage form
    (bf16 bits, or fp32).  Seeded like every other tensor; no model checkpoint exists here."""
    g = (1.0 + 0.1 * _rng(seed, layer, 901).standard_normal(H)).astype(np.float32)
    return bf16_bits(g) if act == "bf16" else g


def make_lora(E: int, H: int, I: int, rank: int = 16, seed: int = 0, layer: int = 0, alpha: float = 16.0) -> dict:
    """Synthetic fp32 LoRA adapters for the expert projections (no trained adapters exist here):
    A ~ N(0, 1/in), B ~ N(0, 0.25/rank), scale = alpha / rank.  Shapes: a_gate, a_up [E][r][H],
    b_gate, b_up [E][I][r], a_down [E][r][I], b_down [E][H][r]."""
    def draw(shape, std, tid):
        return (std * _rng(seed, layer, 950 + tid).standard_normal(shape)).astype(np.float32)
    bs = 0.5 / np.sqrt(rank)
    return dict(rank=rank, scale=alpha / rank,
                a_gate=draw((E, rank, H), 1 / np.sqrt(H), 0), b_gate=draw((E, I, rank), bs, 1),
                a_up=draw((E, rank, H), 1 / np.sqrt(H), 2), b_up=draw((E, I, rank), bs, 3),
                a_down=draw((E, rank, I), 1 / np.sqrt(I), 4), b_down=draw((E, H, rank), bs, 5))
