"""C ABI checks that need no GPU: the library builds and loads, exports every function
include/dflash.h declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

from block_diffusion_drafter_kv_gb300 import binding as B
from block_diffusion_drafter_kv_gb300.build import LIB_PATH, build
from synth import QWEN3_8B, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def L():
    build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dflash_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("dflash_inject_ctx", "dflash_draft_block", "dflash_verify_greedy", "dflash_create",
              "dflash_bind_state", "dflash_workspace_size", "dflash_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dflash_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    # and the binding knows every one of them
    assert set(declared_functions()) == set(B.SIGNATURES)


def test_struct_layouts_match_header():
    assert ctypes.sizeof(B.DflashConfig) == 14 * 4
    assert ctypes.sizeof(B.DflashLayerWeights) == 9 * 8
    assert ctypes.sizeof(B.DflashWeights) == 7 * 8


def _cfg(shape=TINY, **kw):
    c = B.make_config(shape, 4, 1, 128)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value", [("hidden", 200), ("head_dim", 96), ("n_kv_heads", 3),
                                         ("intermediate", 100), ("max_block", 17), ("max_block", 0),
                                         ("n_layers", 0), ("target_hidden", 100), ("vocab", 1),
                                         ("kv_capacity", 2), ("max_batch", 0)])
def test_config_check_rejects(L, field, value):
    c = _cfg(**{field: value})
    assert L.dflash_config_check(ctypes.byref(c)) == -2
    assert L.dflash_workspace_size(ctypes.byref(c)) == 0


def test_config_check_accepts_the_workload_shapes(L):
    from synth import LLAMA31_8B
    for s, blk, bat, cap in ((TINY, 4, 1, 128), (QWEN3_8B, 16, 1, 3700), (QWEN3_8B, 16, 32, 9000),
                             (LLAMA31_8B, 16, 4, 33100)):
        c = B.make_config(s, blk, bat, cap)
        assert L.dflash_config_check(ctypes.byref(c)) == 0
        n = L.dflash_workspace_size(ctypes.byref(c))
        assert 0 < n < (2 << 30)


def test_null_arguments_fail_before_any_launch(L):
    c = _cfg()
    h = ctypes.c_void_p()
    assert L.dflash_create(None, None, ctypes.byref(h)) == -1
    assert L.dflash_create(ctypes.byref(c), None, ctypes.byref(h)) == -1
    w = B.DflashWeights()  # all null pointers
    assert L.dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == -1
    assert L.dflash_inject_ctx(None, None, 1, None, 1, None) == -1
    assert L.dflash_draft_block(None, 1, 4, None, None, None, None) == -1
    assert L.dflash_verify_greedy(None, None, None, 1, 4, None, None, None) == -1
    assert L.dflash_destroy(None) == -1
    assert L.dflash_synth_plant(None, None, None, 1, None, 1, 4, 8, 1.0, None, None) == -1


def test_status_strings(L):
    assert L.dflash_status_string(0) == b"ok"
    assert L.dflash_status_string(-3) == b"capacity exceeded"
    assert L.dflash_status_string(123) == b"unknown status"


def test_noalloc_verify_rejects_bad_arguments_before_any_launch(L):
    """The allocation-free verifier checks alignment and sizes on the host: a misaligned
    logits or token pointer, or a vocabulary beyond its stated maximum, returns
    DFLASH_E_INVAL before the scratch array is looked up or anything is launched."""
    ok16, ok4 = 1 << 20, 1 << 21   # never dereferenced: every call below fails its checks first
    f = L.dflash_verify_greedy_noalloc
    assert f(ok16 + 4, ok4, 1, 4, 1024, ok4, ok4, ok4, None) == -1      # logits not 16-byte aligned
    assert f(ok16 + 8, ok4, 1, 4, 1023, ok4, ok4, ok4, None) == -1      # whatever the vocab
    assert f(ok16, ok4 + 2, 1, 4, 1024, ok4, ok4, ok4, None) == -1      # drafted not 4-byte aligned
    assert f(ok16, ok4, 1, 4, 1024, ok4 + 1, ok4, ok4, None) == -1      # accept_len
    assert f(ok16, ok4, 1, 4, 1024, ok4, ok4 + 3, ok4, None) == -1      # committed
    assert f(ok16, ok4, 1, 4, 1024, ok4, ok4, ok4 + 2, None) == -1      # last_token
    assert f(ok16, ok4, 1, 4, (1 << 28) + 1, ok4, ok4, ok4, None) == -1  # vocab above the maximum
    assert f(ok16, ok4, 1, 4, 1, ok4, ok4, ok4, None) == -1             # vocab below 2
    assert f(ok16, ok4, 0, 4, 1024, ok4, ok4, ok4, None) == -1          # empty batch
    assert f(ok16, ok4, 65, 4, 1024, ok4, ok4, ok4, None) == -3         # beyond the array
    assert f(ok16, ok4, 1, 17, 1024, ok4, ok4, ok4, None) == -3


def test_options_and_error_read_need_a_handle(L):
    v = ctypes.c_int64(0)
    assert L.dflash_set_option(None, B.OPT_CHAIN_MAX, 4) == -1
    assert L.dflash_get_option(None, B.OPT_CHAIN_MAX, ctypes.byref(v)) == -1
    assert L.dflash_selftest_timeout(None, None) == -1
    f = ctypes.c_int32(0)
    assert L.dflash_read_device_error(None, ctypes.byref(f), 0, None) == -1


def test_wrappers_refuse_tensors_the_library_would_misread():
    """The binding checks dtype, device and contiguity before any library call: a handle
    that was never created (no library, no GPU) is enough to see each refusal."""
    import torch
    d = object.__new__(B.Drafter)   # no handle: reaching the library would raise AttributeError
    f32 = torch.zeros(2, 16, 8)
    i32 = torch.zeros(2, 16, dtype=torch.int32)
    bf = torch.zeros(5, 32, 64, dtype=torch.bfloat16)
    calls = [
        lambda: d.inject(bf, 16, torch.zeros(2, dtype=torch.int32), 2),            # CPU tensors
        lambda: d.inject(bf.float(), 16, torch.zeros(2, dtype=torch.int32), 2),    # fp32 hidden
        lambda: d.draft(2, 16, i32.to(torch.int64)),                               # int64 drafted
        lambda: d.draft(2, 16, i32, logits=f32.transpose(1, 2)),                   # non-contiguous logits
        lambda: d.verify(f32.double(), i32, 2, 16, i32[:, 0], i32),                # fp64 logits
        lambda: d.verify_sampling(f32, i32, f32[:, :, 0].half(), 1.0, 2, 16, i32[:, 0], i32),
        lambda: d.verify_hidden(bf, bf, bf.float(), i32, 2, 16, i32[:, 0], i32),
        lambda: d.linear(bf[0], bf[0], bf[0]),                                     # bf16 output
    ]
    for call in calls:
        with pytest.raises(B.DFlashError) as ei:
            call()
        assert ei.value.status == B.DFLASH_E_INVAL
