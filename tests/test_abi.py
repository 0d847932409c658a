"""The C-ABI library loads and exports every entry point its header declares;
host-side argument checks reject bad calls before anything is launched (CPU)."""
import ctypes
import os
import re

import pytest

import row_indexed_flash_gb300 as far

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(far.library_path):
        from row_indexed_flash_gb300 import build
        build.build()
    return far.lib()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", txt))
    return names


def test_every_declared_function_is_exported(lib):
    names = _declared()
    assert {"fa_rows_decode", "fa_rows_prefill", "fa_kv_quantize_int8", "fa_kv_page_table_to_rows"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_struct_layout_matches_header_field_order():
    txt = open(os.path.join(ROOT, "include", "fa_rows.h")).read()
    body = re.search(r"typedef struct fa_rows_args \{(.*?)\} fa_rows_args;", txt, re.S).group(1)
    fields = []
    for line in body.split(";"):
        line = line.strip()
        if not line:
            continue
        decl = line.split()[-1] if "," not in line else line
        if "," in line:
            fields += [x.strip().lstrip("*") for x in re.sub(r"^\s*\w+\s+", "", line).split(",")]
        else:
            fields.append(decl.lstrip("*"))
    assert fields == [f for f, _ in far.fa_rows_args._fields_]


def test_status_strings_and_version(lib):
    assert far.fa_status_string(0) == "FA_OK"
    assert far.fa_status_string(4) == "FA_ERR_INDEX_OOB"
    assert "sm_103a" in far.fa_version()


def _args(**kw):
    a = far.fa_rows_args()
    a.q = a.k = a.v = a.kv_rows = a.out = 4096
    a.q_dtype = a.kv_dtype = far.FA_BF16
    a.out_dtype = far.FA_F32
    a.S, a.Nq, a.Hq, a.Hkv, a.D, a.list_len, a.n_pool_rows = 1, 1, 8, 2, 128, 16, 64
    a.scale = 0.1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), far.FaRowsError),
    (dict(q_dtype=far.FA_F32), far.FaRowsError),
    (dict(kv_dtype=far.FA_F16), far.FaRowsError),        # 16-bit pool must match q
    (dict(out_dtype=far.FA_I8), far.FaRowsError),
    (dict(mask_kind=7), far.FaRowsError),
    (dict(mask_kind=far.FA_MASK_DENSE), far.FaRowsError),  # dense mask without a pointer
    (dict(kv_dtype=far.FA_I8), far.FaRowsError),           # int8 without scales
    (dict(k=4096 + 8), far.FaRowsError),                   # misaligned pool
    (dict(Nq=9, Hq=32, Hkv=8), far.FaRowsError),           # decode packs at most 32 query vectors
])
def test_bad_arguments_are_rejected_on_the_host(lib, kw, status):
    a = _args(**kw)
    st = lib.fa_rows_decode(ctypes.byref(a), None, 0, None)
    assert st in (1, 2), (st, far.fa_last_error())
    assert far.fa_last_error()


def test_null_args_and_empty_batch(lib):
    assert lib.fa_rows_decode(None, None, 0, None) == 1
    assert lib.fa_rows_decode_launches(None) == -1 and far.fa_last_error()
    bad = _args(D=100)
    assert lib.fa_rows_decode_launches(ctypes.byref(bad)) == -1
    a = _args(S=0)
    assert lib.fa_rows_prefill(ctypes.byref(a), None, 0, None) in (0, 2)


def test_kv_helpers_reject_bad_sizes(lib):
    assert lib.fa_kv_quantize_int8(4096, far.FA_BF16, 10, 2, 128, None, 4096, 4096, 100, None) == 2  # R % 64
    assert lib.fa_kv_quantize_int8(4096, far.FA_F32, 10, 2, 128, None, 4096, 4096, 128, None) == 2
    assert lib.fa_kv_dequantize_int8(4096, 4096, 100, 2, 128, 4096, None) == 2
    assert lib.fa_kv_page_table_to_rows(4096, 4, 4096, 2, 0, 4096, 256, None) == 1
    assert lib.fa_kv_append(4096, far.FA_BF16, 4, 1, 4, 4096, 4096, 8, None) == 2    # 8-byte rows
    assert lib.fa_rows_validate(None, 4096, None) == 1


def test_status_word_calls_check_their_arguments_on_the_host(lib):
    assert far.fa_status_string(6) == "FA_ERR_WAIT_EXPIRED"
    assert lib.fa_rows_status(None, 256, 4096, 0, None) == 3          # no workspace
    assert lib.fa_rows_status(4096, 128, 4096, 0, None) == 3          # shorter than the status block
    assert lib.fa_rows_status(4096, 256, None, 0, None) == 1          # no destination word
    assert lib.fa_set_wait_limit_ns(1000) == 0
    assert lib.fa_set_wait_limit_ns(0) == 0                           # back to the default


def test_every_workspace_starts_with_the_status_block(lib):
    a = _args(list_len=0)
    assert lib.fa_rows_workspace_size(ctypes.byref(a), 0) == 256      # decode of empty lists: status block only
    a = _args()
    assert lib.fa_rows_workspace_size(ctypes.byref(a), 1) == 256      # prefill: the status block
    st = lib.fa_rows_prefill(ctypes.byref(a), None, 0, None)
    assert st == 3 and "status word" in far.fa_last_error()           # refused before anything is launched
