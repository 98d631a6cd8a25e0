"""CPU oracle of the sparse MoE block -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs may import this package.  It wraps
``moe_oracle.c`` (plain loops in double, single-threaded) through ctypes.  It
imports nothing from the CUDA package and the CUDA package imports nothing from
here; the two share only the seeded input arrays drawn by ``synth``.

Every function takes a ``synth.MoEInputs`` (storage-format arrays) and returns
float64 / int32 numpy arrays.  The step definitions and their sources are in
the header comment of ``moe_oracle.c``.

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, brute force, invariants or independent library routines
(numpy matmul, numpy stable argsort, scipy softmax) and by the hand-derived
worked examples under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

_DT = {"f32": 0, "bf16": 1, "q4": 2}


class _Lora(ctypes.Structure):
    _fields_ = [
        ("rank", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("a_gate", ctypes.c_void_p),
        ("b_gate", ctypes.c_void_p),
        ("a_up", ctypes.c_void_p),
        ("b_up", ctypes.c_void_p),
        ("a_down", ctypes.c_void_p),
        ("b_down", ctypes.c_void_p),
    ]


class _Matrix(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("q_block", ctypes.c_int32),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("data", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("codebook", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc into oracle/libmoe_oracle.so (IEEE double, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        for name in ("orc_router_logits", "orc_select_topk", "orc_permute", "orc_expert_mlp",
                     "orc_grouped_swiglu", "orc_unpermute", "orc_forward", "orc_forward_tokens",
                     "orc_forward_dense"):
            getattr(_lib, name).restype = ctypes.c_int
        _lib.orc_weight_at.restype = ctypes.c_double
        _lib.orc_weight_at.argtypes = [ctypes.POINTER(_Matrix), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        _lib.orc_rmsnorm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_double, ctypes.c_void_p]
        _lib.orc_round_bf16.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _matrix(inp, which: str, keep: list) -> _Matrix:
    data = {"gate": inp.w_gate, "up": inp.w_up, "down": inp.w_down}[which]
    rows, cols = (inp.I, inp.H) if which in ("gate", "up") else (inp.H, inp.I)
    data = np.ascontiguousarray(data)
    keep.append(data)
    m = _Matrix(_DT[inp.w], inp.q_block, rows, cols, data.ctypes.data, None, None)
    if inp.w == "q4":
        sc = np.ascontiguousarray({"gate": inp.gate_scales, "up": inp.up_scales, "down": inp.down_scales}[which])
        cb = np.ascontiguousarray(inp.codebook, dtype=np.float32)
        keep.extend([sc, cb])
        m.scales = sc.ctypes.data
        m.codebook = cb.ctypes.data
    return m


def _mats(inp):
    keep: list = []
    g, u, d = _matrix(inp, "gate", keep), _matrix(inp, "up", keep), _matrix(inp, "down", keep)
    return g, u, d, keep


def _bias(inp):
    return None if inp.b_router is None else np.ascontiguousarray(inp.b_router, dtype=np.float32)


def router_logits(inp) -> np.ndarray:
    """Step A: logits [T, E] in double."""
    out = np.empty((inp.T, inp.E), dtype=np.float64)
    x, wr, b = np.ascontiguousarray(inp.x), np.ascontiguousarray(inp.w_router), _bias(inp)
    _check(lib().orc_router_logits(inp.T, inp.H, inp.E, _DT[inp.act], _p(x), _p(wr), _p(b), _p(out)), "router")
    return out


def select_topk(logits: np.ndarray, k: int, norm_topk: bool = True):
    """Step B: (ids [T,k] int32, weights [T,k] double, tie_margin [T] double)."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    m = np.empty(T, dtype=np.float64)
    _check(lib().orc_select_topk(T, E, k, int(bool(norm_topk)), _p(logits), _p(ids), _p(w), _p(m)), "select")
    return ids, w, m


def permute(ids: np.ndarray, E: int):
    """Steps C, D: (counts [E], offsets [E+1], order [A], pos [A]) int32."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    A = ids.size
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    order = np.empty(A, dtype=np.int32)
    pos = np.empty(A, dtype=np.int32)
    _check(lib().orc_permute(A, E, _p(ids), _p(counts), _p(offsets), _p(order), _p(pos)), "permute")
    return counts, offsets, order, pos


def expert_mlp(inp, xrow: np.ndarray, e: int):
    """Steps E, F for one activation row (double [H]) through expert e: (h [I], y [H])."""
    g, u, d, keep = _mats(inp)
    xrow = np.ascontiguousarray(xrow, dtype=np.float64)
    h = np.empty(inp.I, dtype=np.float64)
    y = np.empty(inp.H, dtype=np.float64)
    _check(lib().orc_expert_mlp(inp.H, inp.I, _p(xrow), int(e), ctypes.byref(g), ctypes.byref(u),
                                ctypes.byref(d), _p(h), _p(y)), "expert_mlp")
    return h, y


def grouped_swiglu(inp, offsets: np.ndarray, order: np.ndarray):
    """Steps E, F over permuted rows: (h [A, I], y [A, H]) in double."""
    g, u, d, keep = _mats(inp)
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    order = np.ascontiguousarray(order, dtype=np.int32)
    x = np.ascontiguousarray(inp.x)
    h = np.zeros((inp.A, inp.I), dtype=np.float64)
    y = np.zeros((inp.A, inp.H), dtype=np.float64)
    _check(lib().orc_grouped_swiglu(inp.T, inp.H, inp.E, inp.k, inp.I, _DT[inp.act], _p(x), _p(offsets),
                                    _p(order), ctypes.byref(g), ctypes.byref(u), ctypes.byref(d),
                                    _p(h), _p(y)), "grouped_swiglu")
    return h, y


def unpermute(y: np.ndarray, weights: np.ndarray, pos: np.ndarray, T: int, k: int):
    """Step G: out [T, H] in double."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    weights = np.ascontiguousarray(weights, dtype=np.float64)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.float64)
    _check(lib().orc_unpermute(T, k, H, _p(y), _p(weights), _p(pos), _p(out)), "unpermute")
    return out


def forward(inp) -> dict:
    """Steps A..G over all tokens; returns every intermediate."""
    g, u, d, keep = _mats(inp)
    T, E, k, A = inp.T, inp.E, inp.k, inp.A
    r = dict(
        logits=np.empty((T, E)), ids=np.empty((T, k), np.int32), weights=np.empty((T, k)),
        tie_margin=np.empty(T), counts=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
        order=np.empty(A, np.int32), pos=np.empty(A, np.int32), h=np.empty((A, inp.I)),
        y=np.empty((A, inp.H)), out=np.empty((T, inp.H)),
    )
    x, wr, b = np.ascontiguousarray(inp.x), np.ascontiguousarray(inp.w_router), _bias(inp)
    _check(lib().orc_forward(
        T, inp.H, E, k, inp.I, int(inp.norm_topk), _DT[inp.act], _p(x), _p(wr), _p(b),
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d),
        *[_p(r[n]) for n in ("logits", "ids", "weights", "tie_margin", "counts", "offsets", "order", "pos",
                             "h", "y", "out")]), "forward")
    return r


def forward_tokens(inp, tokens: Sequence[int]) -> dict:
    """The block's output for a sample of tokens, each evaluated on its own."""
    g, u, d, keep = _mats(inp)
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n, k = toks.size, inp.k
    r = dict(tokens=toks, ids=np.empty((n, k), np.int32), weights=np.empty((n, k)), tie_margin=np.empty(n),
             out=np.empty((n, inp.H)))
    x, wr, b = np.ascontiguousarray(inp.x), np.ascontiguousarray(inp.w_router), _bias(inp)
    _check(lib().orc_forward_tokens(
        n, _p(toks), inp.H, inp.E, k, inp.I, int(inp.norm_topk), _DT[inp.act], _p(x), _p(wr), _p(b),
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d),
        _p(r["ids"]), _p(r["weights"]), _p(r["tie_margin"]), _p(r["out"])), "forward_tokens")
    return r


def forward_dense(inp) -> np.ndarray:
    """Dense brute force (all experts for every token, masked): out [T, H] in double."""
    g, u, d, keep = _mats(inp)
    out = np.empty((inp.T, inp.H), dtype=np.float64)
    x, wr, b = np.ascontiguousarray(inp.x), np.ascontiguousarray(inp.w_router), _bias(inp)
    _check(lib().orc_forward_dense(inp.T, inp.H, inp.E, inp.k, inp.I, int(inp.norm_topk), _DT[inp.act],
                                   _p(x), _p(wr), _p(b), ctypes.byref(g), ctypes.byref(u), ctypes.byref(d),
                                   _p(out)), "forward_dense")
    return out


def weight_at(inp, which: str, e: int, r: int, c: int) -> float:
    """One expert weight element as the oracle decodes it."""
    g, u, d, keep = _mats(inp)
    m = {"gate": g, "up": u, "down": d}[which]
    return lib().orc_weight_at(ctypes.byref(m), e, r, c)


def rmsnorm(hs: np.ndarray, gamma: np.ndarray, eps: float, act: str) -> np.ndarray:
    """Pre-router RMSNorm in double: hs [T, H] and gamma [H] in storage form (fp32, or bf16 bits)."""
    hs = np.ascontiguousarray(hs)
    gamma = np.ascontiguousarray(gamma)
    T, H = hs.shape
    xn = np.empty((T, H), dtype=np.float64)
    _check(lib().orc_rmsnorm(T, H, _DT[act], _p(hs), _p(gamma), float(eps), _p(xn)), "rmsnorm")
    return xn


def round_bf16(v: np.ndarray) -> np.ndarray:
    """bf16 bits of doubles, rounded to nearest even directly from double."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    bits = np.empty(v.shape, dtype=np.uint16)
    _check(lib().orc_round_bf16(v.size, _p(v), _p(bits)), "round_bf16")
    return bits


def _prenormed(inp, gamma, eps):
    import dataclasses
    xn = rmsnorm(inp.x, gamma, eps, inp.act)
    x_act = round_bf16(xn) if inp.act == "bf16" else xn.astype(np.float32)
    return xn, x_act, dataclasses.replace(inp, x=x_act)


def _widen(inp, rows):
    if inp.act == "bf16":
        return (np.ascontiguousarray(rows).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(rows, dtype=np.float64)


def forward_prenorm(inp, gamma: np.ndarray, eps: float, residual: bool = True) -> dict:
    """The block on pre-normed inputs: xn = RMSNorm(x) * gamma rounded to the activation dtype
    (the experts' and the router's input), out = MoE(xn) (+ x when residual)."""
    xn, x_act, inp2 = _prenormed(inp, gamma, eps)
    r = forward(inp2)
    if residual:
        r["out"] = r["out"] + _widen(inp, inp.x)
    r["xn"], r["xn_act"] = xn, x_act
    return r


def forward_prenorm_tokens(inp, gamma: np.ndarray, eps: float, tokens: Sequence[int], residual: bool = True) -> dict:
    """forward_prenorm for a sample of tokens."""
    xn, x_act, inp2 = _prenormed(inp, gamma, eps)
    r = forward_tokens(inp2, tokens)
    if residual:
        r["out"] = r["out"] + _widen(inp, inp.x[np.asarray(tokens)])
    r["xn"], r["xn_act"] = xn, x_act
    return r


def _lora_struct(lora: dict, keep: list) -> _Lora:
    arrs = {n: np.ascontiguousarray(lora[n], dtype=np.float32) for n in
            ("a_gate", "b_gate", "a_up", "b_up", "a_down", "b_down")}
    keep.append(arrs)
    return _Lora(int(lora["rank"]), float(lora["scale"]), *[_p(arrs[n]) for n in
                                                            ("a_gate", "b_gate", "a_up", "b_up", "a_down", "b_down")])


def forward_lora(inp, lora: dict, tokens: Optional[Sequence[int]] = None) -> dict:
    """The block with LoRA adapters on the three expert projections (fp32 adapters, all math in
    double): z = x . W^T + scale * (x . A^T) . B^T for gate, up and down.  ``lora`` holds rank,
    scale and a_gate [E][r][H], b_gate [E][I][r], a_up, b_up (same), a_down [E][r][I],
    b_down [E][H][r].  Evaluates ``tokens`` (default: all), each on its own."""
    g, u, d, keep = _mats(inp)
    L = _lora_struct(lora, keep)
    toks = np.ascontiguousarray(np.arange(inp.T, dtype=np.int32) if tokens is None
                                else np.asarray(tokens, dtype=np.int32))
    n, k = toks.size, inp.k
    r = dict(tokens=toks, ids=np.empty((n, k), np.int32), weights=np.empty((n, k)), tie_margin=np.empty(n),
             out=np.empty((n, inp.H)))
    x, wr, b = np.ascontiguousarray(inp.x), np.ascontiguousarray(inp.w_router), _bias(inp)
    _check(lib().orc_forward_tokens_lora(
        n, _p(toks), inp.H, inp.E, k, inp.I, int(inp.norm_topk), _DT[inp.act], _p(x), _p(wr), _p(b),
        ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), ctypes.byref(L),
        _p(r["ids"]), _p(r["weights"]), _p(r["tie_margin"]), _p(r["out"])), "forward_tokens_lora")
    return r
