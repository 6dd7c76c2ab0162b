"""The C ABI: libsyn.so loads and exports every function include/syn.h
declares; status strings and defaults; device calls fail loudly without a GPU."""
import ctypes
import os
import re

import pytest
import torch

from chunk_scheduled_communication_gb300 import syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "syn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(syn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("syn_plan_create", "syn_plan_destroy", "syn_ag_gemm", "syn_gemm_rs", "syn_gemm_ar",
                 "syn_sync_status", "syn_plan_query", "syn_autotune", "syn_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(syn.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(syn._SIGS)


def test_status_strings_and_defaults():
    L = syn.lib()
    assert L.syn_status_string(0) == b"SYN_OK"
    assert L.syn_status_string(-4) == b"SYN_ERR_TIMEOUT"
    k = syn.make_knobs()
    assert k.backend == syn.BACKEND_TMA_COLOCATED and k.tile_n == 256 and k.debug_drop_chunk == -1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_plan_create_fails_loudly_without_gpu():
    with pytest.raises(syn.SynError) as e:
        syn.Plan("ag", 4, 0, 256, 256, 256)
    assert e.value.status == syn.ERR_CUDA


def test_null_arguments_are_rejected():
    L = syn.lib()
    assert L.syn_plan_destroy(None) == 0
    assert L.syn_sync_status(None, None) == syn.ERR_INVALID
    assert L.syn_ag_gemm(None, None, None, None, None, None) == syn.ERR_INVALID
    assert L.syn_plan_query(None, None) == syn.ERR_INVALID


def test_protocol_emulation_library_exports_its_header():
    from chunk_scheduled_communication_gb300 import proto
    src = open(os.path.join(ROOT, "include", "syn_proto.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = sorted(set(re.findall(r"\b(syn_[a-z0-9_]+)\s*\(", src)))
    assert names == ["syn_proto_emulate", "syn_proto_last_error"]
    lib = proto.lib()
    assert all(hasattr(lib, n) for n in names)


def test_attention_library_exports_its_header():
    from chunk_scheduled_communication_gb300 import attn
    src = open(os.path.join(ROOT, "include", "syn_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = sorted(set(re.findall(r"\b(syn_[a-z0-9_]+)\s*\(", src)))
    lib = ctypes.CDLL(syn.LIB_PATH)
    assert names and not [n for n in names if not hasattr(lib, n)]
    assert set(names) == set(attn.SIGS)
    L = attn.lib()
    assert L.syn_attn_plan_destroy(None) == 0
    assert L.syn_attn_sync_status(None, None) == syn.ERR_INVALID
    c = attn.make_cfg()
    assert c.d == 128 and c.split == 1 and c.debug_drop_chunk == -1


def test_headers_compile_as_plain_c(tmp_path):
    """The boundary is a C ABI: both public headers compile as C11 on their
    own (no C++ or CUDA types), and the operator calls type-check from C."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_abi.c"
    src.write_text(
        '#include "syn.h"\n#include "syn_attn.h"\n#include "syn_proto.h"\n'
        "int use(const void *const *shards, void *gathered, const void *B, void *C, void *stream) {\n"
        "    syn_layout_t L = {1024, 512, 256, 0, 0, 0};\n"
        "    syn_knobs_t kn;\n"
        "    syn_plan_t plan;\n"
        "    if (syn_knobs_default(&kn) != SYN_OK) return -1;\n"
        "    if (syn_plan_create(&plan, SYN_OP_AG_GEMM, 4, 1, &L, 0, 2, SYN_ORDER_ROW_MAJOR, &kn) != SYN_OK)\n"
        "        return (int)syn_last_error()[0];\n"
        "    syn_ag_gemm(plan, shards, gathered, B, C, stream);\n"
        "    int st = syn_sync_status(plan, stream);\n"
        "    syn_plan_destroy(plan);\n"
        "    return st;\n"
        "}\n")
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
