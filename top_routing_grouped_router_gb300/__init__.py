"""GB300-native sparse Mixture-of-Experts block (Qwen3-MoE style), Python binding.

A thin ctypes binding of the C ABI in ``include/moe.h`` (``libmoe_gb300.so``,
built in-tree by ``top_routing_grouped_router_gb300.build``).  The functions
below keep the C names and only marshal arguments: torch CUDA tensors (or raw
integer device addresses) become pointers, the current torch CUDA stream becomes
the ``stream`` argument.  Every step of the block runs in the library's CUDA
kernels; there is no fallback of any kind, and every call raises if the library
is missing or returns an error.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "MOE_DT_F32", "MOE_DT_BF16", "MOE_DT_Q4", "MoEError", "MoEShape", "MoEQ4", "lib", "library_path",
    "make_shape", "moe_workspace_size", "moe_route", "moe_permute", "moe_grouped_swiglu", "moe_unpermute",
    "moe_forward", "moe_forward_launches", "moe_read_device_error", "moe_status_string", "EXPORTED_SYMBOLS",
    "moe_forward_static_scratch", "moe_forward_rmsnorm", "moe_forward_lora", "moe_graph_buckets", "moe_graphs_arena_size",
    "DecodeGraphs", "moe_lora_pack_size", "moe_lora_pack", "pack_lora", "moe_static_scratch_read_error",
    "moe_debug_set_waits",
]

MOE_DT_F32, MOE_DT_BF16, MOE_DT_Q4 = 0, 1, 2
_DT = {"f32": MOE_DT_F32, "bf16": MOE_DT_BF16, "q4": MOE_DT_Q4}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmoe_gb300.so")

EXPORTED_SYMBOLS = ("moe_workspace_size", "moe_route", "moe_permute", "moe_grouped_swiglu", "moe_unpermute",
                    "moe_forward", "moe_forward_launches", "moe_read_device_error", "moe_status_string",
                    "moe_forward_static_scratch", "moe_forward_rmsnorm", "moe_forward_lora", "moe_graph_buckets", "moe_graphs_arena_size", "moe_graphs_create",
                    "moe_graphs_bucket", "moe_graphs_run", "moe_graphs_destroy", "moe_lora_pack_size", "moe_lora_pack",
                    "moe_static_scratch_read_error", "moe_debug_set_waits")


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {moe_status_string(status)} ({status})")
        self.status = status


class MoEShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("act_dtype", ctypes.c_int32), ("w_dtype", ctypes.c_int32),
                ("norm_topk", ctypes.c_int32), ("q_block", ctypes.c_int32)]


class MoELora(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("scale", ctypes.c_float), ("a_gate", ctypes.c_void_p),
                ("b_gate", ctypes.c_void_p), ("a_up", ctypes.c_void_p), ("b_up", ctypes.c_void_p),
                ("a_down", ctypes.c_void_p), ("b_down", ctypes.c_void_p), ("packed", ctypes.c_void_p)]


class MoEQ4(ctypes.Structure):
    _fields_ = [("gate_scales", ctypes.c_void_p), ("up_scales", ctypes.c_void_p),
                ("down_scales", ctypes.c_void_p), ("codebook", ctypes.c_float * 16)]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libmoe_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"CUDA library {library_path} is missing: build it with "
                               f"`python -m top_routing_grouped_router_gb300.build`")
        L = ctypes.CDLL(library_path)
        vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
        sp = ctypes.POINTER(MoEShape)
        q4p = ctypes.POINTER(MoEQ4)
        sig = {
            "moe_workspace_size": [sp, ctypes.POINTER(ctypes.c_size_t)],
            "moe_route": [sp, vp, vp, vp, i32p, vp, vp, vp, vp, sz, vp],
            "moe_permute": [sp, i32p, i32p, i32p, i32p, i32p, vp, sz, vp],
            "moe_grouped_swiglu": [sp, vp, i32p, i32p, vp, vp, vp, q4p, vp, vp, sz, vp],
            "moe_unpermute": [sp, vp, vp, i32p, vp, vp],
            "moe_forward": [sp, vp, vp, vp, vp, vp, vp, q4p, vp, i32p, vp, vp, sz, vp],
            "moe_read_device_error": [vp, ctypes.POINTER(ctypes.c_int32), vp],
            "moe_forward_launches": [sp, ctypes.POINTER(ctypes.c_int32)],
            "moe_forward_static_scratch": [sp, vp, vp, vp, vp, vp, vp, q4p, vp, i32p, vp, vp],
            "moe_static_scratch_read_error": [ctypes.POINTER(ctypes.c_int32), vp],
            "moe_debug_set_waits": [ctypes.c_uint64, ctypes.c_int32],
            "moe_forward_rmsnorm": [sp, vp, vp, ctypes.c_float, ctypes.c_int, vp, vp, vp, vp, vp, q4p, vp, vp, i32p,
                                    vp, vp, sz, vp],
            "moe_forward_lora": [sp, vp, vp, vp, vp, vp, vp, q4p, ctypes.POINTER(MoELora), vp, i32p, vp, vp, sz, vp],
            "moe_graph_buckets": [ctypes.c_int, vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)],
            "moe_graphs_arena_size": [sp, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
            "moe_graphs_create": [sp, ctypes.c_int, vp, vp, vp, vp, vp, q4p, vp, sz, vp, ctypes.POINTER(vp)],
            "moe_graphs_bucket": [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)],
            "moe_graphs_run": [vp, ctypes.c_int, vp, vp, i32p, vp],
            "moe_graphs_destroy": [vp],
            "moe_lora_pack_size": [sp, ctypes.POINTER(ctypes.c_size_t)],
            "moe_lora_pack": [sp, ctypes.POINTER(MoELora), vp, sz, vp],
        }
        for name, argtypes in sig.items():
            f = getattr(L, name)
            f.argtypes = argtypes
            f.restype = ctypes.c_int
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def make_shape(T, H, E, k, I, act="bf16", w="bf16", norm_topk=True, q_block=64) -> MoEShape:
    return MoEShape(int(T), int(H), int(E), int(k), int(I), _DT[act] if isinstance(act, str) else int(act),
                    _DT[w] if isinstance(w, str) else int(w), int(bool(norm_topk)), int(q_block))


def _ptr(t):
    """Device address of a torch tensor, an int address, or None -> NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t):
    return t.numel() * t.element_size()


def _check(rc: int, what: str):
    if rc != 0:
        raise MoEError(rc, what)


def moe_workspace_size(shape: MoEShape) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(shape), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_route(shape, x, w_router, b_router, expert_ids, weights, tie_margin=None, logits=None, workspace=None,
              stream=None):
    _check(lib().moe_route(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(b_router), _ptr(expert_ids),
                           _ptr(weights), _ptr(tie_margin), _ptr(logits), _ptr(workspace), _nbytes(workspace),
                           _stream(stream)), "moe_route")


def moe_permute(shape, expert_ids, counts, offsets, order, pos, workspace, stream=None):
    _check(lib().moe_permute(ctypes.byref(shape), _ptr(expert_ids), _ptr(counts), _ptr(offsets), _ptr(order),
                             _ptr(pos), _ptr(workspace), _nbytes(workspace), _stream(stream)), "moe_permute")


def moe_grouped_swiglu(shape, x, offsets, order, w_gate, w_up, w_down, q4, y, workspace, stream=None):
    _check(lib().moe_grouped_swiglu(ctypes.byref(shape), _ptr(x), _ptr(offsets), _ptr(order), _ptr(w_gate),
                                    _ptr(w_up), _ptr(w_down), ctypes.byref(q4) if q4 is not None else None,
                                    _ptr(y), _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "moe_grouped_swiglu")


def moe_unpermute(shape, y, weights, pos, out, stream=None):
    _check(lib().moe_unpermute(ctypes.byref(shape), _ptr(y), _ptr(weights), _ptr(pos), _ptr(out),
                               _stream(stream)), "moe_unpermute")


def moe_forward(shape, x, w_router, b_router, w_gate, w_up, w_down, q4, out, expert_ids_out=None,
                weights_out=None, workspace=None, stream=None):
    _check(lib().moe_forward(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(b_router), _ptr(w_gate),
                             _ptr(w_up), _ptr(w_down), ctypes.byref(q4) if q4 is not None else None, _ptr(out),
                             _ptr(expert_ids_out), _ptr(weights_out), _ptr(workspace), _nbytes(workspace),
                             _stream(stream)), "moe_forward")


def moe_forward_static_scratch(shape, x, w_router, b_router, w_gate, w_up, w_down, q4, out, expert_ids_out=None,
                               weights_out=None, stream=None):
    """moe_forward with the library's fixed 32 MiB device scratch instead of a caller workspace."""
    _check(lib().moe_forward_static_scratch(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(b_router),
                                            _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                            ctypes.byref(q4) if q4 is not None else None, _ptr(out),
                                            _ptr(expert_ids_out), _ptr(weights_out), _stream(stream)),
           "moe_forward_static_scratch")


def moe_debug_set_waits(limit_ns: int = 2_000_000_000, extra_need: int = 0):
    """Failure-path test hook: the bounded device waits' limit and an unreachable extra count
    for the down tiles' h wait (see moe.h).  Call with no arguments to restore the defaults."""
    _check(lib().moe_debug_set_waits(int(limit_ns), int(extra_need)), "moe_debug_set_waits")


def moe_static_scratch_read_error(stream=None) -> int:
    """Reads and clears the device error word of the static scratch array (synchronises the stream)."""
    code = ctypes.c_int32(0)
    _check(lib().moe_static_scratch_read_error(ctypes.byref(code), _stream(stream)),
           "moe_static_scratch_read_error")
    return code.value


def moe_forward_rmsnorm(shape, hs, gamma, eps, w_router, b_router, w_gate, w_up, w_down, q4, out, add_residual=True,
                        x_norm_out=None, expert_ids_out=None, weights_out=None, workspace=None, stream=None):
    """out = hs + MoE(RMSNorm(hs) * gamma) (the residual only with add_residual)."""
    _check(lib().moe_forward_rmsnorm(ctypes.byref(shape), _ptr(hs), _ptr(gamma), float(eps), int(bool(add_residual)),
                                     _ptr(w_router), _ptr(b_router), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                     ctypes.byref(q4) if q4 is not None else None, _ptr(out), _ptr(x_norm_out),
                                     _ptr(expert_ids_out), _ptr(weights_out), _ptr(workspace), _nbytes(workspace),
                                     _stream(stream)), "moe_forward_rmsnorm")


def make_lora(rank, scale, a_gate, b_gate, a_up, b_up, a_down, b_down, packed=None) -> MoELora:
    """The moe_lora struct over device tensors (fp32, row-major; see moe.h for the shapes);
    `packed` is a buffer written by moe_lora_pack / pack_lora, or None."""
    return MoELora(int(rank), float(scale), _ptr(a_gate), _ptr(b_gate), _ptr(a_up), _ptr(b_up), _ptr(a_down),
                   _ptr(b_down), _ptr(packed))


def moe_lora_pack_size(shape: MoEShape) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_lora_pack_size(ctypes.byref(shape), ctypes.byref(n)), "moe_lora_pack_size")
    return n.value


def moe_lora_pack(shape: MoEShape, lora: MoELora, packed, stream=None):
    """Packs the adapters of `lora` into the device buffer `packed` (moe_lora_pack_size bytes)."""
    _check(lib().moe_lora_pack(ctypes.byref(shape), ctypes.byref(lora), _ptr(packed), _nbytes(packed),
                               _stream(stream)), "moe_lora_pack")


def pack_lora(shape: MoEShape, lora: MoELora, device=None, stream=None) -> MoELora:
    """A copy of `lora` that carries a freshly written pack.  The pack is a uint8 tensor on
    `device`, kept alive as the returned struct's `pack_tensor` attribute."""
    import torch
    buf = torch.empty(moe_lora_pack_size(shape), dtype=torch.uint8, device=device or "cuda")
    moe_lora_pack(shape, lora, buf, stream)
    out = MoELora(lora.rank, lora.scale, lora.a_gate, lora.b_gate, lora.a_up, lora.b_up, lora.a_down, lora.b_down,
                  _ptr(buf))
    out.pack_tensor = buf
    return out


def moe_forward_lora(shape, x, w_router, b_router, w_gate, w_up, w_down, q4, lora: MoELora, out, expert_ids_out=None,
                     weights_out=None, workspace=None, stream=None):
    """moe_forward with LoRA adapters on the expert projections."""
    _check(lib().moe_forward_lora(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(b_router), _ptr(w_gate),
                                  _ptr(w_up), _ptr(w_down), ctypes.byref(q4) if q4 is not None else None,
                                  ctypes.byref(lora), _ptr(out), _ptr(expert_ids_out), _ptr(weights_out),
                                  _ptr(workspace), _nbytes(workspace), _stream(stream)), "moe_forward_lora")


def moe_forward_launches(shape: MoEShape) -> int:
    n = ctypes.c_int32(0)
    _check(lib().moe_forward_launches(ctypes.byref(shape), ctypes.byref(n)), "moe_forward_launches")
    return n.value


def moe_read_device_error(workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().moe_read_device_error(_ptr(workspace), ctypes.byref(code), _stream(stream)),
           "moe_read_device_error")
    return code.value


def moe_graph_buckets(max_bs: int) -> list:
    """Batch-size buckets of the decode graphs for max_bs (host only)."""
    buf = (ctypes.c_int32 * 64)()
    n = ctypes.c_int32(0)
    _check(lib().moe_graph_buckets(int(max_bs), ctypes.cast(buf, ctypes.c_void_p), 64, ctypes.byref(n)),
           "moe_graph_buckets")
    return list(buf[:n.value])


def moe_graphs_arena_size(shape: MoEShape, max_bs: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_graphs_arena_size(ctypes.byref(shape), int(max_bs), ctypes.byref(n)), "moe_graphs_arena_size")
    return n.value


class DecodeGraphs:
    """Bucketed CUDA-graph decode around moe_forward (moe_graphs_* of the C ABI).

    The arena (a device uint8 tensor of moe_graphs_arena_size bytes) is allocated here and
    kept alive with the graphs; the weights are captured by address and must outlive them.
    """

    def __init__(self, shape: MoEShape, max_bs: int, w_router, b_router, w_gate, w_up, w_down, q4=None,
                 device=None, stream=None):
        import torch
        self.shape = shape
        if device is None:
            device = w_router.device if hasattr(w_router, "device") else torch.device("cuda")
        self.arena = torch.zeros(moe_graphs_arena_size(shape, max_bs), dtype=torch.uint8, device=device)
        self._keep = (w_router, b_router, w_gate, w_up, w_down, q4)
        self._stream = stream if stream is not None else torch.cuda.Stream(device=self.arena.device)
        h = ctypes.c_void_p(0)
        _check(lib().moe_graphs_create(ctypes.byref(shape), int(max_bs), _ptr(w_router), _ptr(b_router),
                                       _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                       ctypes.byref(q4) if q4 is not None else None, _ptr(self.arena),
                                       self.arena.numel(), _stream(self._stream), ctypes.byref(h)),
               "moe_graphs_create")
        self._h = h
        self.buckets = moe_graph_buckets(max_bs)

    def bucket(self, T: int) -> int:
        b = ctypes.c_int32(0)
        _check(lib().moe_graphs_bucket(self._h, int(T), ctypes.byref(b)), "moe_graphs_bucket")
        return b.value

    def run(self, T: int, x, out, expert_ids_out=None, stream=None):
        """One decode step of T tokens: x [T][H] in, out [T][H] out (device or host tensors)."""
        st = self._stream if stream is None else stream
        _check(lib().moe_graphs_run(self._h, int(T), _ptr(x), _ptr(out), _ptr(expert_ids_out), _stream(st)),
               "moe_graphs_run")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().moe_graphs_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
