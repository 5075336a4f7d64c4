"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point the header declares, agrees with the binding on the
parameter struct layout, and rejects bad static parameters on the host
before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_mla_decode_03_gb300 as mla
from paged_mla_decode_03_gb300 import build as mla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.load_library()


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(mla_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_entry_point_is_exported(lib):
    names = declared_functions()
    assert "mla_decode_plan" in names and "mla_decode_run" in names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", mla.library_path()], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    assert set(names) <= exported


def test_param_struct_layout_matches_c(tmp_path):
    fields = [f[0] for f in mla.MlaDecodeParams._fields_]
    src = tmp_path / "layout.c"
    prog = ['#include <stdio.h>', '#include <stddef.h>', '#include "mla_decode.h"',
            'int main(void) {', 'printf("%zu\\n", sizeof(mla_decode_params));']
    prog += [f'printf("%zu\\n", offsetof(mla_decode_params, {f}));' for f in fields]
    prog += ["return 0; }"]
    src.write_text("\n".join(prog))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    vals = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert vals[0] == ctypes.sizeof(mla.MlaDecodeParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(mla.MlaDecodeParams, f).offset == off, f


def _params(**kw):
    base = dict(batch=2, num_heads=16, max_seq_len_q=1, max_seq_len=64, page_size=32,
                max_pages_per_req=2, num_pages=8, packed=0, max_total_q=0, kv_dtype=0, mask=0,
                return_lse=1, device=0)
    base.update(kw)
    return mla.MlaDecodeParams(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_heads=96), -2),
    (dict(num_heads=8), -2),
    (dict(page_size=16), -2),
    (dict(page_size=128), -2),
    (dict(batch=-1), -1),
    (dict(max_seq_len=0), -1),
    (dict(kv_dtype=7), -1),
    (dict(mask=3), -1),
    (dict(max_pages_per_req=1), -1),   # 1 page of 32 rows < max_seq_len 64
    (dict(packed=1, max_total_q=-5), -1),
    (dict(cp_world=-1), -1),
    (dict(cp_world=4, cp_rank=4), -1),
    (dict(cp_world=4, cp_rank=-1), -1),
    (dict(cp_world=1, cp_rank=1), -1),
    (dict(sparse_top_k=-1), -1),
    (dict(sparse_top_k=(1 << 24) + 1), -1),
    (dict(sparse_top_k=64, cp_world=2, cp_rank=0), -1),  # sparse selection without DCP only
])
def test_plan_rejects_bad_static_parameters_on_host(lib, kw, status):
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    rc = lib.mla_decode_plan(ctypes.byref(_params(**kw)), ctypes.byref(handle), ctypes.byref(ws))
    assert rc == status
    assert not handle.value


def test_null_arguments_are_rejected(lib):
    assert lib.mla_decode_plan(None, None, None) == -1
    assert lib.mla_decode_run(None, None, None, None, None, None, 0, 1.0, 1.0, None, None, None,
                              0, None) == -1
    assert lib.mla_decode_run_device_scales(None, None, None, None, None, None, 0, None, None,
                                            None, None, None, 0, None) == -1
    assert lib.mla_decode_run_host(None, None, None, None, None, None, 0, 1.0, 1.0, None, None,
                                   None, 0, None, 0, None) == -1
    assert lib.mla_decode_host_staging_bytes(None, 0) == 0
    assert lib.mla_decode_run_dcp(None, None, None, None, None, None, 0, None, 1.0, 1.0, None,
                                  None, None, 0, None) == -1
    assert lib.mla_decode_run_sparse(None, None, None, None, None, None, 0, None, 1.0, 1.0, None,
                                     None, None, 0, None) == -1
    lib.mla_decode_destroy(None)
    assert lib.mla_decode_workspace_size(None) == 0


def test_status_strings_and_status_word(lib):
    assert mla.mla_decode_status_string(0) == "MLA_OK"
    assert mla.mla_decode_status_string(-3) == "MLA_ERR_WORKSPACE_TOO_SMALL"
    assert mla.mla_decode_status_string(123) == "MLA_ERR_UNKNOWN"
    assert mla.mla_decode_status_offset() == 0
