"""The C ABI library loads and exports every function include/mla_dcp.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla_dcp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b((?:mla|gqa)_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("mla_decode_partial", "mla_shard_combine", "mla_workspace_size",
                 "mla_get_device_error", "mla_status_string", "mla_version"):
        assert want in names


def test_library_exports_every_declared_symbol():
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert mla.mla_version() == 200
    assert mla.mla_status_string(-5) == "block-table entry out of range"


def test_null_arguments_rejected_on_host():
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    sh = mla.mla_shape(1, 1, 16, 0, 0.07)
    kv = mla.mla_kv_pages(None, None, 0, 1, 64)
    st = L.mla_decode_partial(None, ctypes.byref(kv), None, 1, None, ctypes.byref(sh), -1, 2, 0,
                              None, None, None, 0, None)
    assert st == -1
    st = L.mla_shard_combine(None, None, 2, ctypes.byref(sh), None, None, None, None)
    assert st == -1
    bad = mla.mla_shape(0, 1, 16, 0, 0.07)
    assert L.mla_workspace_size(ctypes.byref(bad), 2, -1) == 0
    assert L.mla_get_device_error(None, None) == -1


def test_python_binding_names_match_the_abi():
    import sequence_sharded_mla_gb300 as mla
    for name in declared_functions():
        assert callable(getattr(mla, name)), name


def test_noalloc_refuses_shapes_beyond_its_scratch_before_any_cuda_call():
    """The no-allocation entry point checks its stated limits (at most 8192
    work units) with host arithmetic first, so the refusal needs no GPU and
    no buffers are ever touched."""
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    sh = mla.mla_shape(4096, 1, 64, 0, 0.07)        # 4096 requests x 8 shards = 32768 units
    kv = mla.mla_kv_pages(None, None, 0, 1, 64)
    st = L.mla_decode_partial_noalloc(None, ctypes.byref(kv), None, 1, None, ctypes.byref(sh),
                                      -1, 8, 0, None, None, None)
    assert st == -2
    assert L.mla_decode_partial_noalloc(None, ctypes.byref(kv), None, 1, None, None, -1, 8, 0,
                                        None, None, None) == -1


def test_profile_events_take_both_or_neither():
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    assert L.mla_set_profile_events(None, ctypes.c_void_p(64)) == -1
    assert L.mla_set_profile_events(ctypes.c_void_p(64), None) == -1
    assert L.mla_set_profile_events(None, None) == 0


def test_local_layouts_need_one_shard():
    """A local cache holds one shard's positions: computing every shard from
    it is an argument error, found before any CUDA call."""
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    sh = mla.mla_shape(1, 1, 16, 0, 0.07)
    kv = mla.mla_kv_pages(ctypes.c_void_p(256), None, 0, 1, 64)
    fake = ctypes.c_void_p(512)
    for layout in (2, 3):
        st = L.mla_decode_partial(fake, ctypes.byref(kv), fake, 1, fake, ctypes.byref(sh), -1, 2,
                                  layout, fake, fake, fake, 1 << 20, None)
        assert st == -1
    st = L.mla_decode_partial(fake, ctypes.byref(kv), fake, 1, fake, ctypes.byref(sh), 0, 2, 7,
                              fake, fake, fake, 1 << 20, None)
    assert st == -1


def test_index_arrays_need_only_4_byte_alignment():
    """block_table and seq_lens may be views into a larger batch (4-byte
    aligned); the query still has to be 16-byte aligned.  Without a GPU a
    call that passes the host checks stops at the first CUDA query."""
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    sh = mla.mla_shape(1, 1, 16, 0, 0.07)
    kv = mla.mla_kv_pages(ctypes.c_void_p(256), None, 0, 1, 64)
    fake, off4 = ctypes.c_void_p(512), ctypes.c_void_p(516)
    st = L.mla_decode_partial(fake, ctypes.byref(kv), off4, 1, off4, ctypes.byref(sh), -1, 2, 0,
                              fake, fake, fake, 1 << 20, None)
    assert st != -1
    st = L.mla_decode_partial(off4, ctypes.byref(kv), fake, 1, fake, ctypes.byref(sh), -1, 2, 0,
                              fake, fake, fake, 1 << 20, None)
    assert st == -1
    off2 = ctypes.c_void_p(514)
    st = L.mla_decode_partial(fake, ctypes.byref(kv), off2, 1, fake, ctypes.byref(sh), -1, 2, 0,
                              fake, fake, fake, 1 << 20, None)
    assert st == -1


def test_gqa_arguments_checked_on_host():
    """The GQA calls refuse bad arguments and unsupported shapes before any
    CUDA call: null pointers, zero sizes, head widths other than 128,
    groups that are not powers of two."""
    import sequence_sharded_mla_gb300 as mla
    L = mla.lib()
    fake = ctypes.c_void_p(512)
    kv = mla.gqa_kv_pages(fake, fake, 4, 64)
    good = mla.gqa_shape(2, 1, 16, 4, 128, 0, 0.088)
    assert L.gqa_decode_partial(None, ctypes.byref(kv), fake, 1, fake, ctypes.byref(good), -1, 2,
                                0, fake, fake, fake, 1 << 20, None) == -1
    bad = mla.gqa_shape(0, 1, 16, 4, 128, 0, 0.088)
    assert L.gqa_workspace_size(ctypes.byref(bad), 2, -1) == 0
    for shape in (mla.gqa_shape(2, 1, 16, 4, 64, 0, 0.125),    # head width 64
                  mla.gqa_shape(2, 1, 12, 4, 128, 0, 0.088),   # groups of 3
                  mla.gqa_shape(2, 1, 16, 3, 128, 0, 0.088)):  # 3 does not divide 16
        assert L.gqa_workspace_size(ctypes.byref(shape), 2, -1) == 0
    nokv = mla.gqa_kv_pages(None, fake, 4, 64)
    assert L.gqa_decode_partial(fake, ctypes.byref(nokv), fake, 1, fake, ctypes.byref(good), -1,
                                2, 0, fake, fake, fake, 1 << 20, None) == -1
    assert L.gqa_shard_combine(None, fake, 2, ctypes.byref(good), fake, None, None) == -1
