"""The C-ABI library on the host: it loads, exports every declared symbol, sizes
its workspace, and rejects bad arguments before touching CUDA (no GPU needed)."""
import ctypes
import os
import re

import pytest

from communication_overlap_domino_gb300 import binding as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(b.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return b.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            names += re.findall(r"DOMINO_API\s+[\w\s\*]*?\b(domino_\w+)\s*\(", text)
    return names


def test_header_declares_entry_points():
    names = declared_functions()
    assert "domino_mlp_fwd" in names and "domino_mlp_bwd" in names and "domino_shard_sum" in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"
    bound = {name for name, _, _ in b.SIGNATURES}
    assert bound == set(declared_functions()), "binding and header disagree"


def test_status_strings(lib):
    for code, name in b.STATUS.items():
        assert lib.domino_status_string(code).decode() == name


def desc(**kw):
    base = dict(M=256, d=512, F=2048, P=2, mu=2, act="gelu", partial="f32")
    base.update(kw)
    return b.make_desc(**base)


def test_workspace_layout(lib):
    d = desc()
    M, dd, F, P, mu = 256, 512, 2048, 2, 2
    Fp = F // P
    tiles_m, tiles_n2 = (M // mu + 127) // 128, (dd + 255) // 256
    sync = 4 * (mu * P * tiles_m + mu * tiles_m * tiles_n2 * 4 + 1)
    head = (128 + sync + 255) // 256 * 256  # status, timeline, then the tile counters from byte 128
    expect = head + P * M * Fp * 2 + P * M * dd * 4
    assert b.workspace_size(d) == expect
    d16 = desc(partial="bf16")
    assert b.workspace_size(d16) == head + P * M * Fp * 2 + P * M * dd * 2
    assert b.saved_size(d) == P * M * Fp * 2 * 2
    assert b.saved_size(desc(act="swiglu")) == P * M * Fp * 3 * 2
    assert b.workspace_size(d, with_bwd=True) > b.workspace_size(d)


@pytest.mark.parametrize("kw,status", [
    (dict(P=0), 1), (dict(P=17), 1), (dict(mu=0), 1), (dict(d=0), 1), (dict(M=-1), 1),
    (dict(F=2047), 2), (dict(M=255), 2), (dict(out_slices=3), 2),
    (dict(d=516, F=2064), 3), (dict(F=2 * 1028), 3),
    (dict(mu=16, out_slices=8), 2),
])
def test_descriptor_validation(lib, kw, status):
    d = desc(**kw)
    assert b.workspace_size(d) == 0
    ws = ctypes.c_void_p(0x10000)
    arr = b._ptr_array([0x20000] * max(1, d.P))
    st = lib.domino_mlp_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, None, ws, 1 << 40, None)
    assert st == status, b.lib().domino_last_error()


def test_enum_validation(lib):
    for field, bad in (("act", 9), ("partial_dtype", 5), ("schedule", 3), ("reserve_sms", -1), ("flags", 0x80)):
        d = desc()
        setattr(d, field, bad)
        arr = b._ptr_array([0x20000] * 2)
        st = lib.domino_mlp_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, None, 0x10000, 1 << 40, None)
        assert st == 1, field


def test_null_and_alignment_and_workspace(lib):
    d = desc()
    arr = b._ptr_array([0x20000] * 2)
    assert lib.domino_mlp_fwd(None, 0x30000, arr, arr, 0x40000, None, 0x10000, 1 << 40, None) == 1
    assert lib.domino_mlp_fwd(ctypes.byref(d), None, arr, arr, 0x40000, None, 0x10000, 1 << 40, None) == 1
    bad = b._ptr_array([0x20008, 0x20000])
    assert lib.domino_mlp_fwd(ctypes.byref(d), 0x30000, bad, arr, 0x40000, None, 0x10000, 1 << 40, None) == 3
    assert lib.domino_mlp_fwd(ctypes.byref(d), 0x30004, arr, arr, 0x40000, None, 0x10000, 1 << 40, None) == 3
    assert lib.domino_mlp_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, None, 0x10010, 1 << 40, None) == 3
    small = b.workspace_size(d) - 1
    assert lib.domino_mlp_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, None, 0x10000, small, None) == 4
    assert "workspace" in lib.domino_last_error().decode()


def test_shard_sum_validation(lib):
    arr = b._ptr_array([0x20000] * 2)
    assert lib.domino_shard_sum(arr, 0, 0, 4, 8, 8, 0x40000, 8, None) == 1
    assert lib.domino_shard_sum(arr, 2, 3, 4, 8, 8, 0x40000, 8, None) == 1
    assert lib.domino_shard_sum(arr, 2, 0, 4, 12, 12, 0x40000, 12, None) == 3
    assert lib.domino_shard_sum(arr, 2, 0, 4, 8, 4, 0x40000, 8, None) == 1
    assert lib.domino_shard_sum(b._ptr_array([0x20002, 0x20000]), 2, 0, 4, 8, 8, 0x40000, 8, None) == 3
    # empty problems are a no-op that needs no device
    assert lib.domino_shard_sum(arr, 2, 0, 0, 8, 8, 0x40000, 8, None) == 0
    # 16-byte vectors of Y are counted with 32-bit indices: rows * cols / 8 must stay below 2^32
    # (rejected before any device is touched)
    assert lib.domino_shard_sum(arr, 2, 0, 1 << 29, 64, 64, 0x40000, 64, None) == 2
    assert "2^32" in lib.domino_last_error().decode()


def test_empty_batch_is_noop(lib):
    d = desc(M=0)
    arr = b._ptr_array([0x20000] * 2)
    ws = b.workspace_size(d)
    assert lib.domino_mlp_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, None, 0x10000, ws, None) == 0


def test_backward_validates(lib):
    d = desc()
    arr = b._ptr_array([0x20000] * 2)
    st = lib.domino_mlp_bwd(ctypes.byref(d), 0x30000, arr, arr, None, 0x50000, 0x60000, arr, arr, 0x10000,
                            1 << 40, None)
    assert st == 1


def test_interleaved_validates(lib):
    d = desc(schedule="fused")
    arr = b._ptr_array([0x20000] * 2)
    args = (arr, arr, 0x30000, 0x40000, None, 0x30000, 0x50000, 0x60000, 0x70000, arr, arr, 0x10000, 1 << 40, None)
    assert lib.domino_mlp_fwd_bwd_interleaved(ctypes.byref(d), *args) == 2  # FUSED: not interleavable
    d = desc(schedule="streams")
    assert b.interleaved_workspace_size(d) >= b.workspace_size(d) + b.workspace_size(d, with_bwd=True)
    bad = (arr, arr, 0x30000, None) + args[4:]
    assert lib.domino_mlp_fwd_bwd_interleaved(ctypes.byref(d), *bad) == 1
    small = args[:-2] + (b.interleaved_workspace_size(d) - 1, None)
    assert lib.domino_mlp_fwd_bwd_interleaved(ctypes.byref(d), *small) == 4


def attn_desc(**kw):
    base = dict(B=2, S=256, d=512, H=4, P=2, mu=2, partial="f32", schedule="streams")
    base.update(kw)
    return b.make_attn_desc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(P=0), 1), (dict(H=0), 1), (dict(mu=0), 1), (dict(B=-1), 1),
    (dict(S=200), 2), (dict(dh=64), 2), (dict(H=3), 2), (dict(mu=3), 2), (dict(schedule="fused", B=16, mu=16), 2),
    (dict(d=516), 3),
])
def test_attention_descriptor_validation(lib, kw, status):
    d = attn_desc(**kw)
    assert b.attn_workspace_size(d) == 0
    arr = b._ptr_array([0x20000] * max(1, d.P))
    assert lib.domino_attn_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, 0x10000, 1 << 40, None) == status


def test_attention_workspace_and_arguments(lib):
    d = attn_desc()
    M, Hp, dh = 2 * 256, 2, 128
    qkv = 2 * M * 3 * Hp * dh * 2
    o = 2 * M * Hp * dh * 2
    z = 2 * M * 512 * 4
    align = lambda x: (x + 255) // 256 * 256
    tiles_m, tiles_n = 256 // 128, 512 // 256  # one chunk of 256 rows; d = 512
    sync = 4 * (2 * tiles_m + tiles_m * tiles_n * 4 + 1)  # a fused output-projection launch's counters
    assert b.attn_workspace_size(d) == align(align(align(align(256 + sync) + qkv) + o) + z)
    arr = b._ptr_array([0x20000] * 2)
    ws = b.attn_workspace_size(d)
    assert lib.domino_attn_fwd(ctypes.byref(d), None, arr, arr, 0x40000, 0x10000, ws, None) == 1
    assert lib.domino_attn_fwd(ctypes.byref(d), 0x30008, arr, arr, 0x40000, 0x10000, ws, None) == 3
    assert lib.domino_attn_fwd(ctypes.byref(d), 0x30000, arr, arr, 0x40000, 0x10000, ws - 1, None) == 4
    assert lib.domino_attn_fwd(ctypes.byref(attn_desc(B=0, mu=1)), None, None, None, None, None, 0, None) == 0


def test_tensor_peak_validates_before_cuda(lib):
    out = b.TensorPeak()
    ref = ctypes.byref(out)
    ws = b.TENSOR_PEAK_WS_BYTES
    assert lib.domino_tensor_peak(1, 0, None, ws, 0, None, ref) == 1
    assert lib.domino_tensor_peak(1, 0, 0x40000, ws, 0, None, None) == 1
    assert lib.domino_tensor_peak(0, 0, 0x40000, ws, 0, None, ref) == 1
    assert lib.domino_tensor_peak(b.TENSOR_PEAK_MAX_MMAS + 1, 0, 0x40000, ws, 0, None, ref) == 1
    assert lib.domino_tensor_peak(1, 0, 0x40000, ws - 1, 0, None, ref) == 4
    assert lib.domino_tensor_peak(1, 0, 0x40010, ws, 0, None, ref) == 3
    assert b"mmas_per_cluster" in lib.domino_last_error() or b"256-byte" in lib.domino_last_error()


def test_partials_validates(lib):
    d = desc()
    arr = b._ptr_array([0x20000] * 2)
    z = b._ptr_array([0x50000, 0x58000])
    ws = 1 << 40
    fn = lib.domino_mlp_fwd_partials
    assert fn(None, 0x30000, arr, arr, z, None, None, 0x10000, ws, None) == 1
    assert fn(ctypes.byref(d), 0x30000, arr, arr, None, None, None, 0x10000, ws, None) == 1
    assert fn(ctypes.byref(d), 0x30000, arr, arr, b._ptr_array([0x50000, 0]), None, None, 0x10000, ws, None) == 1
    assert fn(ctypes.byref(d), 0x30000, arr, arr, b._ptr_array([0x50000, 0x58004]), None, None, 0x10000, ws,
              None) == 3
    assert fn(ctypes.byref(d), 0x30000, arr, arr, z, b._ptr_array([0x1] + [0] * 7), None, 0x10000, ws, None) == 1
    assert "event" in lib.domino_last_error().decode()
    small = b.workspace_size(d) - 1
    assert fn(ctypes.byref(d), 0x30000, arr, arr, z, None, None, 0x10000, small, None) == 4
    # an empty batch touches nothing
    e = desc(M=0)
    assert fn(ctypes.byref(e), 0, arr, arr, z, None, None, 0x10000, ws, None) == 0


def test_descriptor_rejects_outputs_beyond_32bit_vector_count(lib):
    # the shard-sum counts 16-byte vectors of Y with 32-bit indices: M * d / 8 must stay below 2^32
    d = desc(M=(1 << 28) - 1024, d=1 << 7, F=1024, mu=1)
    assert b.workspace_size(d) > 0
    d2 = desc(M=(1 << 28) + 1024, d=1 << 7, F=1024, mu=1)
    assert b.workspace_size(d2) == 0
    assert "2^32" in lib.domino_last_error().decode()
