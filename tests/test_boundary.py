"""C-ABI boundary checks that need no GPU: the library builds and loads, exports every
symbol include/gdn.h declares, and rejects contract violations before touching a device."""
import ctypes
import os
import re

import pytest

from chunked_gated_delta_05_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_\w+|kda_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    lib = _lib.load()
    names = header_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_struct_sizes_match_header_layout():
    # desc: 6 ints, pointer, int, float, 4 ints, float (x86-64 / aarch64 LP64 alignment)
    assert ctypes.sizeof(_lib.Desc) == 64
    assert ctypes.sizeof(_lib.FwdArgs) == 15 * 8
    assert ctypes.sizeof(_lib.BwdArgs) == 23 * 8


@pytest.mark.parametrize("lb", [0.0, 0.5, -5.5, float("nan")])
def test_gate_lower_bound_outside_range_rejected(lb):
    assert ws_size(desc(use_gate_in_kernel=1, lower_bound=lb), "kda_fwd_workspace_size") == 0
    assert "lower_bound" in _lib.load().gdn_last_error().decode()


def test_gate_in_kernel_is_kda_only_and_needs_parameters():
    lib = _lib.load()
    d = desc(use_gate_in_kernel=1, lower_bound=-5.0)
    a = _lib.FwdArgs()
    a.q = a.k = a.v = a.g = a.beta = 0x1000
    a.o = 0x10000000
    a.workspace, a.workspace_bytes = 0x20000000, 1 << 30
    assert lib.gdn_fwd(ctypes.byref(d), ctypes.byref(a), None) == _lib.GDN_EINVAL
    assert "KDA" in lib.gdn_last_error().decode()
    assert lib.kda_fwd(ctypes.byref(d), ctypes.byref(a), None) == _lib.GDN_EINVAL
    assert "A_log" in lib.gdn_last_error().decode()


def desc(**kw):
    d = _lib.Desc()
    d.B, d.T, d.H, d.K, d.V, d.chunk_size = 1, 128, 2, 128, 128, 64
    d.num_seqs = 1
    d.scale = 0.0
    d.use_qk_l2norm = 1
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def ws_size(d, fn="gdn_fwd_workspace_size"):
    return getattr(_lib.load(), fn)(ctypes.byref(d))


def offsets(vals):
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))


def test_valid_desc_has_workspace():
    assert ws_size(desc()) > 0


@pytest.mark.parametrize("field,value", [("K", 64), ("V", 256), ("chunk_size", 32), ("B", 0), ("T", 0),
                                         ("H", 0), ("scale", float("nan"))])
def test_invalid_desc_rejected(field, value):
    assert ws_size(desc(**{field: value})) == 0
    assert _lib.load().gdn_last_error().decode() != ""


@pytest.mark.parametrize("vals,ok", [([0, 5, 128], True), ([0, 128], True), ([1, 128], False),
                                     ([0, 64, 64, 128], False), ([0, 70, 60, 128], False),
                                     ([0, 64, 127], False)])
def test_packed_offsets_validation(vals, ok):
    arr, ptr = offsets(vals)
    d = desc(cu_seqlens=ptr, num_seqs=len(vals) - 1)
    assert (ws_size(d) > 0) == ok


def test_packed_requires_batch_one():
    arr, ptr = offsets([0, 64, 128])
    assert ws_size(desc(B=2, cu_seqlens=ptr, num_seqs=2)) == 0


def test_workspace_grows_with_chunks():
    assert ws_size(desc(T=256)) > ws_size(desc(T=128))
    arr, ptr = offsets([0, 1, 2, 128])     # three documents: 1 + 1 + 2 chunks
    assert ws_size(desc(cu_seqlens=ptr, num_seqs=3)) > ws_size(desc())


def test_fwd_rejects_null_and_small_workspace_before_device_use():
    lib = _lib.load()
    d = desc()
    a = _lib.FwdArgs()
    assert lib.gdn_fwd(ctypes.byref(d), ctypes.byref(a), None) == _lib.GDN_EINVAL
    a.q = a.k = a.v = a.g = a.beta = 0x1000
    a.o = 0x100000
    a.workspace = 0x200000
    a.workspace_bytes = 16
    assert lib.gdn_fwd(ctypes.byref(d), ctypes.byref(a), None) == _lib.GDN_EINVAL
    assert "workspace" in lib.gdn_last_error().decode()
    a.workspace_bytes = ws_size(d)
    a.o = 0x1000   # aliases q
    assert lib.gdn_fwd(ctypes.byref(d), ctypes.byref(a), None) == _lib.GDN_EINVAL
    d2 = desc(output_final_state=1)
    a.o = 0x100000
    assert lib.gdn_fwd(ctypes.byref(d2), ctypes.byref(a), None) == _lib.GDN_EINVAL


def test_strerror_names_every_code():
    lib = _lib.load()
    names = {lib.gdn_strerror(c).decode() for c in range(5)}
    assert len(names) == 5


def test_python_wrapper_rejects_bad_offsets_without_gpu():
    import torch
    from chunked_gated_delta_05_gb300 import ops
    with pytest.raises(ValueError):
        ops._offsets([0, True, 5], 5)
    with pytest.raises(ValueError):
        ops._offsets(torch.tensor([0.0, 5.0]), 5)


def plan(d):
    L, S = ctypes.c_int(), ctypes.c_int()
    rc = _lib.load().gdn_chain_plan(ctypes.byref(d), ctypes.byref(L), ctypes.byref(S))
    assert rc == _lib.GDN_OK
    return L.value, S.value


@pytest.fixture
def auto_plan():
    lib = _lib.load()
    yield lib
    assert lib.gdn_set_chain_segment(0) == _lib.GDN_OK


def test_chain_plan_covers_every_chunk(auto_plan):
    # few long chains: the segmented chain is chosen; many short ones: the plain chain
    for B, T, H in [(2, 4096, 16), (1, 8192, 16), (1, 32768, 16), (1, 8192, 32), (1, 256, 2), (64, 512, 16)]:
        nc = (T + 63) // 64
        L, S = plan(desc(B=B, T=T, H=H, num_seqs=B))
        assert 1 <= L <= nc and S == (nc + L - 1) // L, (B, T, H, L, S)
    assert plan(desc(B=1, T=8192, H=16))[1] > 1
    assert plan(desc(B=64, T=512, H=16, num_seqs=64))[1] == 1


def test_chain_plan_packed_documents(auto_plan):
    vals = [0, 100, 3000, 3100, 9000]
    arr, ptr = offsets(vals)
    L, S = plan(desc(B=1, T=9000, H=4, cu_seqlens=ptr, num_seqs=4))
    longest = (5900 + 63) // 64
    assert S == (longest + L - 1) // L


def test_chain_segment_override(auto_plan):
    lib = auto_plan
    d = desc(B=1, T=64 * 10 + 5, H=2)
    assert lib.gdn_set_chain_segment(3) == _lib.GDN_OK
    assert plan(d) == (3, 4)
    scan_ws = ws_size(d)
    assert lib.gdn_set_chain_segment(1 << 20) == _lib.GDN_OK
    assert plan(d) == (11, 1)
    plain_ws = ws_size(d)
    # three 128x128 fp32 state buffers per (segment, head) for the scan: entry states, maps,
    # offsets
    assert scan_ws - plain_ws >= 3 * 4 * 2 * 128 * 128 * 4
    assert lib.gdn_set_chain_segment(-1) == _lib.GDN_EINVAL
