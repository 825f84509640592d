"""CPU checks of the C-ABI boundary: the library builds, loads without a GPU,
exports every function include/ft.h declares, and the Python binding exposes
the same names.  No compute call is made here."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ft.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ft_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib_path():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__
    return __graft_entry__._build_module().build()


@pytest.fixture(scope="module")
def checked_lib_path(lib_path):
    import __graft_entry__
    return __graft_entry__._build_module().build(checked=True)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ft_cache_create", "ft_cache_resize", "ft_route_classify", "ft_fetch_misses",
                     "ft_moe_forward", "ft_cache_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_checked_build_exports_the_same_symbols(lib_path, checked_lib_path):
    normal, checked = ctypes.CDLL(lib_path), ctypes.CDLL(checked_lib_path)
    missing = [n for n in declared_functions() if not hasattr(checked, n)]
    assert not missing, missing
    assert normal.ft_checked_build() == 0 and checked.ft_checked_build() == 1
    # the knob validates its arguments before anything else, in both builds
    for lib in (normal, checked):
        assert lib.ft_debug_set_key_slot(None, 0, 0) == 1  # FT_ERR_INVALID_ARG


def test_host_bank_calls_validate_before_any_cuda_call(lib_path):
    lib = ctypes.CDLL(lib_path)
    lib.ft_host_bank_alloc.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_void_p)]
    lib.ft_host_bank_free.argtypes = [ctypes.c_void_p]
    out = ctypes.c_void_p(1234)
    assert lib.ft_host_bank_alloc(0, ctypes.byref(out)) == 1   # FT_ERR_INVALID_ARG: zero bytes
    assert lib.ft_host_bank_alloc(4096, None) == 1             # FT_ERR_INVALID_ARG: null out
    assert lib.ft_host_bank_free(None) == 0                   # freeing nothing is fine


def test_binding_has_the_same_names(lib_path):
    import expert_cache_host_layer_gb300 as ft
    for n in declared_functions():
        assert hasattr(ft, n), n


def test_host_only_calls(lib_path):
    import expert_cache_host_layer_gb300 as ft
    assert ft.ft_expert_bytes(2048, 512, ft.FT_W_BF16) == 6291456
    assert ft.ft_expert_bytes(4096, 2048, ft.FT_W_FP8E4M3_B128) == 25168896
    assert ft.ft_expert_bytes(256, 128, ft.FT_W_F32) == 393216
    assert ft.ft_expert_bytes(100, 128, ft.FT_W_FP8E4M3_B128) == 0
    lib = ft.library()
    assert lib.ft_status_str(ft.FT_ERR_CAPACITY) == b"FT_ERR_CAPACITY"
    # argument validation happens before any CUDA call
    cfg = ft.ft_cache_config()
    out = ctypes.c_void_p()
    assert lib.ft_cache_create(ctypes.byref(cfg), None, 0, None, ctypes.byref(out)) == ft.FT_ERR_INVALID_ARG
    assert b"num_layers" in lib.ft_last_error()
    assert lib.ft_route_classify(None, 0, None, 0, None, None) == ft.FT_ERR_INVALID_ARG
    assert lib.ft_cache_destroy(None) == ft.FT_OK


@pytest.mark.parametrize("field,value,message", [
    ("num_experts", 0, b"num_experts"),
    ("num_experts", 2048, b"num_experts"),
    ("top_k", 0, b"top_k"),
    ("top_k", 40, b"top_k"),
    ("hidden", 102, b"unsupported hidden/inter/wdtype"),  # fp32 rows need multiples of 4
    ("max_tokens", 0, b"max_tokens"),
    ("fetch_mode", 7, b"fetch_mode"),
    ("copy_streams", 3, b"copy_streams"),
    ("fetch_warps", 5, b"fetch_warps"),
    ("bank_blobs", 0, b"bank_blobs"),
    ("host_bank_bytes", 1, b"host_bank_bytes"),
])
def test_create_rejects_bad_configs_before_any_gpu_work(lib_path, field, value, message):
    """ft_cache_create validates its arguments on the host first: each bad
    field gives FT_ERR_INVALID_ARG and a message naming it, with no GPU."""
    import expert_cache_host_layer_gb300 as ft
    lib = ft.library()
    bank = ctypes.create_string_buffer(64)  # never read: validation comes first
    cfg = ft.make_config(2, 16, 2, 256, 128, ft.FT_W_F32, ctypes.addressof(bank), 10 ** 9, 16, 1)
    setattr(cfg, field, value)
    out = ctypes.c_void_p()
    st = lib.ft_cache_create(ctypes.byref(cfg), ctypes.c_void_p(1 << 20), 12, None, ctypes.byref(out))
    assert st == ft.FT_ERR_INVALID_ARG and message in lib.ft_last_error(), (st, lib.ft_last_error())
    assert not out.value


def test_create_rejects_unaligned_pool_and_bad_slot_counts(lib_path):
    import expert_cache_host_layer_gb300 as ft
    lib = ft.library()
    bank = ctypes.create_string_buffer(64)
    cfg = ft.make_config(2, 16, 2, 256, 128, ft.FT_W_F32, ctypes.addressof(bank), 10 ** 9, 16, 1)
    out = ctypes.c_void_p()
    assert lib.ft_cache_create(ctypes.byref(cfg), ctypes.c_void_p((1 << 20) + 8), 12, None,
                               ctypes.byref(out)) == ft.FT_ERR_INVALID_ARG
    assert b"256-byte aligned" in lib.ft_last_error()
    assert lib.ft_cache_create(ctypes.byref(cfg), ctypes.c_void_p(1 << 20), 0, None,
                               ctypes.byref(out)) == ft.FT_ERR_INVALID_ARG
    assert b"num_slots" in lib.ft_last_error()
