"""The C ABI without a GPU: the library builds, loads, exports every function
include/peagle.h and include/peagle_train.h declare, its structs match the binding's layout, and host
validation rejects bad arguments before touching the device."""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("peagle.h", "peagle_train.h")]


@pytest.fixture(scope="module")
def B():
    from speculative_drafting_expand_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    binding.lib()
    return binding


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"^(?:pe_status|const char\*)\s+(pe_\w+)\(", text, re.M)))


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ("pe_create", "pe_destroy", "pe_expand_batch", "pe_draft_forward",
                 "pe_lmhead_argmax", "pe_get_device_error", "pe_status_string"):
        assert name in fns


def test_library_exports_every_declared_symbol(B):
    lib = B.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(B.EXPORTED)


def test_struct_layouts_match_the_header(B):
    src = r"""
    #include <stdio.h>
    #include <stddef.h>
    #include "peagle.h"
    int main(void) {
      printf("%zu %zu %zu %zu %zu %zu\n", sizeof(pe_model_desc), sizeof(pe_layer_weights),
             sizeof(pe_weights), sizeof(pe_expanded), offsetof(pe_expanded, T_out),
             offsetof(pe_model_desc, dtype));
      return 0;
    }
    """
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    want = [ctypes.sizeof(B.pe_model_desc), ctypes.sizeof(B.pe_layer_weights),
            ctypes.sizeof(B.pe_weights), ctypes.sizeof(B.pe_expanded),
            B.pe_expanded.T_out.offset, B.pe_model_desc.dtype.offset]
    assert got == want


def test_status_strings(B):
    assert B.status_string(0) == "ok"
    assert B.status_string(1) == "invalid argument"
    assert B.status_string(2) == "unsupported shape"
    assert B.status_string(99) == "unknown status"


def test_host_validation_rejects_bad_arguments_without_a_device(B):
    lib = B.lib()
    h = ctypes.c_void_p()
    w = B.pe_weights()
    desc = B.pe_model_desc(64, 1, 2, 1, 64, 64, 100, 192, 16, 99, 1e4, 1e-5, 0)
    # null weights
    assert lib.pe_create(ctypes.byref(desc), ctypes.byref(w), 16, 1, ctypes.byref(h)) == 1
    # bad page size / head dim are unsupported shapes
    desc.page_size = 32
    assert lib.pe_create(ctypes.byref(desc), ctypes.byref(w), 16, 1, ctypes.byref(h)) == 2
    desc.page_size, desc.head_dim = 16, 96
    assert lib.pe_create(ctypes.byref(desc), ctypes.byref(w), 16, 1, ctypes.byref(h)) == 2
    # heads not divisible by kv heads
    desc.head_dim, desc.n_heads, desc.n_kv_heads = 64, 3, 2
    assert lib.pe_create(ctypes.byref(desc), ctypes.byref(w), 16, 1, ctypes.byref(h)) == 1
    # null handles
    ex = B.pe_expanded()
    assert lib.pe_expand_batch(None, 1, 1, 1, None, None, None, None, None, None, 1, 1, None,
                               ctypes.byref(ex), None) == 1
    assert lib.pe_draft_forward(None, ctypes.byref(ex), 1, 1, None, 1, None, None, 1, None,
                                None) == 1
    assert lib.pe_lmhead_argmax(None, None, 1, None, None, None) == 1
    assert lib.pe_destroy(None) == 1
    assert lib.pe_set_kv_cache_fp8(None, None, None) == 1


def test_training_entry_points_validate_on_the_host(B):
    lib = B.lib()
    buf = ctypes.create_string_buffer(64)
    # bad sizes, leading dimension, mask type
    assert lib.pe_train_build_mask(0, 4, 0, buf, 64, None) == 1
    assert lib.pe_train_build_mask(4, 4, 0, None, 16, None) == 1
    assert lib.pe_train_build_mask(4, 4, 0, buf, 8, None) == 1      # ld < n_max K
    assert lib.pe_train_build_mask(4, 4, 1, buf, 20, None) == 1     # 40-byte rows
    assert lib.pe_train_build_mask(4, 4, 7, buf, 16, None) == 1
    # the per-sample mask is a view of the amortized one: host arithmetic only
    v = ctypes.c_void_p()
    rows, ld = ctypes.c_int64(), ctypes.c_int64()
    assert lib.pe_train_mask_view(buf, 48, 12, 4, 5, ctypes.byref(v), ctypes.byref(rows),
                                  ctypes.byref(ld)) == 0
    assert v.value == ctypes.addressof(buf) and rows.value == 20 and ld.value == 48
    assert lib.pe_train_mask_view(buf, 48, 12, 4, 13, ctypes.byref(v), ctypes.byref(rows),
                                  ctypes.byref(ld)) == 1
    # partition: boundaries must run 0 < ... < n, capacity must hold every row
    b = (ctypes.c_int32 * 3)(0, 8, 16)
    args = [buf, buf, buf, buf, buf, buf]
    bad = (ctypes.c_int32 * 3)(0, 8, 15)
    assert lib.pe_train_partition(16, 4, 0.5, buf, 2, bad, *args, 100, None) == 1
    bad = (ctypes.c_int32 * 3)(0, 8, 8)
    assert lib.pe_train_partition(8, 4, 0.5, buf, 2, bad, *args, 100, None) == 1
    assert lib.pe_train_partition(16, 4, 0.5, buf, 2, b, *args, 8 + 64 - 1, None) == 1
    assert lib.pe_train_partition(16, 4, 0.5, buf, 65, b, *args, 1000, None) == 1
    assert lib.pe_train_partition(16, 4, 0.5, None, 2, b, *args, 100, None) == 1


def test_enum_constants_match_the_binding(B):
    # every PE_* enumerator of the headers that the binding names has the
    # binding's value (read from the compiled header, not parsed)
    text = "".join(open(h).read() for h in HEADERS)
    names = sorted(set(re.findall(r"\b(PE_[A-Z0-9_]+)\s*=", text)))
    names = [n for n in names if hasattr(B, n)]
    assert "PE_TUNE_GEMM_TILE_ORDER" in names and "PE_FUSE_NORM" in names
    src = "#include <stdio.h>\n#include \"peagle.h\"\n#include \"peagle_train.h\"\nint main(void) {\n"
    src += "".join(f'  printf("%lld\\n", (long long){n});\n' for n in names) + "  return 0;\n}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "e.c")
        exe = os.path.join(d, "e")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    assert got == [int(getattr(B, n)) for n in names], list(zip(names, got))
