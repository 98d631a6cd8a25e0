"""The C-ABI library builds, loads and exports every entry point declared in include/moe.h,
and rejects bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import top_routing_grouped_router_gb300 as moe
from top_routing_grouped_router_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert sorted(moe.EXPORTED_SYMBOLS) == names


def test_status_strings(L):
    for code in range(0, -8, -1):
        assert moe.moe_status_string(code).startswith("MOE_")


@pytest.mark.parametrize("name", ["tiny", "decode8", "decode64z", "decode48q", "prefill"])
def test_workspace_size_for_every_workload(L, name):
    import synth
    c = synth.WORKLOADS[name]
    s = moe.make_shape(c["T"], c["H"], c["E"], c["k"], c["I"], c["act"], c["w"])
    n = moe.moe_workspace_size(s)
    A = c["T"] * c["k"]
    assert n >= A * c["H"] * (4 if c["act"] == "f32" else 2)
    assert n % 256 == 0


@pytest.mark.parametrize("kw,code", [
    (dict(k=9, E=8), -2),          # k > E
    (dict(E=300, k=2), -2),        # E above 256
    (dict(H=60), -2),              # H not a multiple of 8
    (dict(I=0), -2),
    (dict(T=-1), -2),
    (dict(k=33, E=64), -2),
    (dict(act="f32", w="bf16"), -3),
    (dict(act="f32", w="q4"), -3),
    (dict(w="q4", q_block=48), -2),  # q_block does not divide H=64*...
])
def test_shape_validation(L, kw, code):
    base = dict(T=4, H=128, E=8, k=2, I=64, act="bf16", w="bf16", q_block=64)
    base.update(kw)
    s = moe.make_shape(base["T"], base["H"], base["E"], base["k"], base["I"], base["act"], base["w"],
                       q_block=base["q_block"])
    n = ctypes.c_size_t(0)
    assert L.moe_workspace_size(ctypes.byref(s), ctypes.byref(n)) == code


def test_null_and_workspace_errors_return_before_launch(L):
    s = moe.make_shape(4, 128, 8, 2, 64)
    ws_need = moe.moe_workspace_size(s)
    fake = 1 << 20  # never dereferenced: every call below fails host-side validation
    st = None
    # null shape / null pointers
    assert L.moe_route(None, fake, fake, None, fake, fake, None, None, fake, ws_need, st) == -1
    assert L.moe_route(ctypes.byref(s), None, fake, None, fake, fake, None, None, fake, ws_need, st) == -1
    assert L.moe_forward(ctypes.byref(s), fake, fake, None, None, fake, fake, None, fake, None, None, fake,
                         ws_need, st) == -1
    # workspace too small / missing
    assert L.moe_route(ctypes.byref(s), fake, fake, None, fake, fake, None, None, fake, ws_need - 1, st) == -4
    assert L.moe_permute(ctypes.byref(s), fake, fake, fake, fake, fake, None, ws_need, st) == -4
    assert L.moe_grouped_swiglu(ctypes.byref(s), fake, fake, fake, fake, fake, fake, None, fake, fake, 16, st) == -4
    # misaligned pointers
    assert L.moe_route(ctypes.byref(s), fake + 2, fake, None, fake, fake, None, None, fake, ws_need, st) == -5
    assert L.moe_unpermute(ctypes.byref(s), fake + 8, fake, fake, fake, st) == -5
    assert L.moe_forward(ctypes.byref(s), fake, fake, None, fake, fake, fake, None, fake, None, None, fake + 64,
                         ws_need, st) == -5
    # q4 without scales
    sq = moe.make_shape(4, 128, 8, 2, 64, "bf16", "q4")
    assert L.moe_grouped_swiglu(ctypes.byref(sq), fake, fake, fake, fake, fake, fake, None, fake, fake,
                                moe.moe_workspace_size(sq), st) == -1
    assert L.moe_read_device_error(None, None, st) == -1


def test_binding_raises_on_error(L):
    s = moe.make_shape(4, 128, 8, 9, 64)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_workspace_size(s)
    assert ei.value.status == -2


def test_graph_buckets_follow_the_capture_pattern():
    # [1, 2, 4, 8] + 16, 32, ... up to the first multiple of 16 covering max_bs
    assert moe.moe_graph_buckets(1) == [1]
    assert moe.moe_graph_buckets(5) == [1, 2, 4, 8]
    assert moe.moe_graph_buckets(8) == [1, 2, 4, 8]
    assert moe.moe_graph_buckets(64) == [1, 2, 4, 8, 16, 32, 48, 64]
    assert moe.moe_graph_buckets(40) == [1, 2, 4, 8, 16, 32, 48]
    with pytest.raises(moe.MoEError):
        moe.moe_graph_buckets(0)
    with pytest.raises(moe.MoEError):
        moe.moe_graph_buckets(100000)  # more buckets than the table holds


def test_graph_arena_covers_every_bucket_workspace():
    shape = moe.make_shape(1, 2048, 128, 8, 768)
    arena = moe.moe_graphs_arena_size(shape, 64)
    ws64 = moe.moe_workspace_size(moe.make_shape(64, 2048, 128, 8, 768))
    static = 2 * 64 * 2048 * 2 + 64 * 8 * 4
    assert arena >= ws64 + static
    assert arena <= ws64 + static + 4 * 256


def test_lora_pack_size_is_the_four_padded_bf16_arrays():
    # [E][64][H] + [E][32][I] + [E*I][128] + [E*H][64] bf16, each region rounded up to 256 bytes
    E, H, I = 128, 2048, 768
    shape = moe.make_shape(8, H, E, 8, I)
    al = lambda b: (b + 255) // 256 * 256
    want = al(E * 64 * H * 2) + al(E * 32 * I * 2) + al(E * I * 128 * 2) + al(E * H * 64 * 2)
    assert moe.moe_lora_pack_size(shape) == want
    odd = moe.make_shape(3, 24, 5, 2, 40)
    assert moe.moe_lora_pack_size(odd) == al(5 * 64 * 24 * 2) + al(5 * 32 * 40 * 2) + al(5 * 40 * 256) + al(5 * 24 * 128)


def test_lora_pack_rejects_bad_arguments_without_a_gpu_call(L):
    st = None
    shape = moe.make_shape(8, 128, 8, 2, 64)
    fake = ctypes.c_void_p(1 << 20)
    lo = moe.MoELora(16, 2.0, fake, fake, fake, fake, fake, fake, None)
    need = moe.moe_lora_pack_size(shape)
    # NULL pack, misaligned pack, too small, rank out of range: all refused before any launch
    assert L.moe_lora_pack(ctypes.byref(shape), ctypes.byref(lo), None, need, st) == -1
    assert L.moe_lora_pack(ctypes.byref(shape), ctypes.byref(lo), ctypes.c_void_p((1 << 20) + 16), need, st) == -5
    assert L.moe_lora_pack(ctypes.byref(shape), ctypes.byref(lo), fake, need - 1, st) == -4
    bad = moe.MoELora(17, 2.0, fake, fake, fake, fake, fake, fake, None)
    assert L.moe_lora_pack(ctypes.byref(shape), ctypes.byref(bad), fake, need, st) == -2


def test_static_scratch_rejects_misaligned_q4_scales_before_any_cuda_call(L):
    # every check of moe_forward_static_scratch runs before its first CUDA call, so on a
    # host without a GPU a misaligned 4-bit scale pointer must come back as MOE_ERR_ALIGN
    s = moe.make_shape(8, 256, 8, 2, 128, "bf16", "q4")
    fake = 1 << 20  # never dereferenced
    q4 = moe.MoEQ4(fake, fake + 8, fake, (ctypes.c_float * 16)(*[-1 + 2 * j / 15 for j in range(16)]))
    rc = L.moe_forward_static_scratch(ctypes.byref(s), fake, fake, None, fake, fake, fake, ctypes.byref(q4), fake,
                                      None, None, None)
    assert rc == -5  # MOE_ERR_ALIGN
    q4.up_scales = None
    rc = L.moe_forward_static_scratch(ctypes.byref(s), fake, fake, None, fake, fake, fake, ctypes.byref(q4), fake,
                                      None, None, None)
    assert rc == -1  # MOE_ERR_NULLPTR


def test_debug_wait_hook_validates_and_restores(L):
    assert L.moe_debug_set_waits(0, 0) == -2          # a zero limit is refused
    assert L.moe_debug_set_waits(1000, -1) == -2      # so is a negative count
    assert L.moe_debug_set_waits(2_000_000_000, 0) == 0
