"""The C-ABI library builds, loads and exports every entry point include/kvc.h declares;
host-side argument checks reject bad calls before anything reaches a GPU.  CPU only: no
call here launches a kernel."""
import ctypes
import os
import re

import pytest

import pagedattention_kvc_store_gb300 as kvc
from pagedattention_kvc_store_gb300.kvc import PoolDesc, lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for header in os.listdir(os.path.join(ROOT, "include")):
        if header.endswith(".h"):
            text = open(os.path.join(ROOT, "include", header)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_entry_point_is_exported():
    declared = _declared_functions()
    assert "kvc_decode" in declared and "kvc_store" in declared
    L = lib()
    for name in declared:
        assert hasattr(L, name), f"{name} declared but not exported"
    assert set(kvc.EXPORTS) == set(declared)


def test_status_strings():
    L = lib()
    assert L.kvc_status_string(0) == b"KVC_OK"
    assert L.kvc_status_string(3) == b"KVC_ERR_WORKSPACE"


POOL = PoolDesc(32, 16, 2, 64)
FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: checks fail before any launch


def test_plan_is_host_only_and_consistent():
    splits, chunk, ws = kvc.kvc_decode_plan(4, 4, POOL, 100, 1)
    assert (splits, chunk, ws) == (1, 128, 0)
    splits, chunk, ws = kvc.kvc_decode_plan(8, 64, PoolDesc(2000, 64, 8, 128), 131072, 0)
    assert splits >= 1 and chunk % 64 == 0 and splits * chunk >= 131072
    assert (splits - 1) * chunk < 131072
    if splits > 1:
        rows = 8 * 64
        o_bytes = rows * splits * 128 * 4
        assert ws == -(-o_bytes // 256) * 256 + rows * splits * 4
    s2, c2, _ = kvc.kvc_decode_plan(8, 64, PoolDesc(2000, 64, 8, 128), 131072, 7)
    assert s2 <= 7 and s2 * c2 >= 131072


@pytest.mark.parametrize("pool,q_heads,code", [
    (PoolDesc(32, 16, 2, 96), 4, 2),     # head_dim 96 unsupported
    (PoolDesc(32, 8, 2, 64), 4, 2),      # page size 8 unsupported
    (PoolDesc(32, 16, 2, 64), 3, 1),     # q_heads not a multiple of kv_heads
    (PoolDesc(32, 16, 2, 64), 32, 2),    # group 16 unsupported
    (PoolDesc(0, 16, 2, 64), 4, 1),      # empty pool
])
def test_decode_rejects_bad_shapes_before_launch(pool, q_heads, code):
    st = lib().kvc_decode(FAKE, 0, FAKE, FAKE, FAKE, pool, FAKE, 8, FAKE, 4, 100, q_heads,
                          0.0, 1, None, 0, None)
    assert st == code
    assert lib().kvc_last_error()


def test_decode_requires_workspace_when_split():
    st = lib().kvc_decode(FAKE, 0, FAKE, FAKE, FAKE, POOL, FAKE, 8, FAKE, 4, 100, 4, 0.0, 2,
                          None, 0, None)
    assert st == 3


def test_decode_rejects_short_block_table_and_misalignment():
    st = lib().kvc_decode(FAKE, 0, FAKE, FAKE, FAKE, POOL, FAKE, 4, FAKE, 4, 100, 4, 0.0, 1,
                          None, 0, None)
    assert st == 1 and b"bt_stride" in lib().kvc_last_error()
    st = lib().kvc_decode(ctypes.c_void_p(0x10002), 0, FAKE, FAKE, FAKE, POOL, FAKE, 8, FAKE,
                          4, 100, 4, 0.0, 1, None, 0, None)
    assert st == 1 and b"aligned" in lib().kvc_last_error()


def test_append_and_store_argument_checks():
    st = lib().kvc_append(FAKE, 0, FAKE, FAKE, FAKE, POOL, FAKE, 8, None, FAKE, 4, 8, 2, 100,
                          4, 0.0, None)
    assert st == 1   # q_indptr required
    st = lib().kvc_store(FAKE, FAKE, POOL, FAKE, FAKE, FAKE, -1, None)
    assert st == 1
    st = lib().kvc_slot_mapping(FAKE, FAKE, 8, FAKE, None, 4, 5, 1, 16, None)
    assert st == 1   # decode form needs num_tokens == num_seqs


def test_empty_calls_are_no_ops():
    assert lib().kvc_store(FAKE, FAKE, POOL, FAKE, FAKE, FAKE, 0, None) == 0
    assert lib().kvc_decode(FAKE, 0, FAKE, FAKE, FAKE, POOL, FAKE, 8, FAKE, 0, 100, 4, 0.0, 0,
                            None, 0, None) == 0
    assert lib().kvc_merge(FAKE, 0, FAKE, FAKE, 0, 4, 64, None, None) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    t = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        kvc.kvc_store(t, t, t, t, torch.zeros(4, dtype=torch.int32))


def test_binding_refuses_pageable_decode_out():
    """The decode calls take a CUDA or a pinned host out; pageable host memory is refused."""
    import torch
    t = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    lens = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="pinned"):
        kvc.kvc_decode(t, t, t, t, torch.zeros(4, 1, dtype=torch.int32), lens, 16)
    with pytest.raises(ValueError, match="pinned"):
        kvc.kvc_merge(t, torch.zeros(4, 2, 64), torch.zeros(4, 2))


def test_error_word_setting_is_host_only():
    """kvc_set_error_word stores a pointer for the calling thread: a misaligned one is refused,
    NULL (the library's own words) is accepted, and neither touches the device."""
    L = kvc.lib()
    assert kvc.kvc.STATUS[L.kvc_set_error_word(ctypes.c_void_p(6))] == "KVC_ERR_INVALID_ARG"
    assert L.kvc_set_error_word(None) == 0
