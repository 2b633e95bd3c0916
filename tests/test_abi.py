"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, and exports exactly the entry points include/csa2.h declares;
the product package never touches the oracle."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    return sorted(set(re.findall(r"CSA2_API\s+(?:const\s+char\s*\*|int)\s*(csa2_\w+)\s*\(", src)))


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("csa2_tail_layout", "csa2_index_score", "csa2_topk", "csa2_topk_candidates",
              "csa2_sparse_swa_attn", "csa2_status_string"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    from sparse_attention_prefill_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(lib, n), n
    lib.csa2_status_string.restype = ctypes.c_char_p
    assert lib.csa2_status_string(0) == b"ok"
    # exported dynamic symbols are exactly the declared ones
    out = os.popen("nm -D --defined-only %s" % path).read()
    exported = sorted(set(re.findall(r" T (\w+)", out)))
    assert exported == _declared()


def test_host_validation_rejects_before_launch():
    """Argument errors the host can see return a status without touching the GPU."""
    from sparse_attention_prefill_gb300 import build
    lib = ctypes.CDLL(build.build())
    # negative request count, zero window
    assert lib.csa2_tail_layout(-1, None, None, 128, None, None, None, None, None, None,
                                ctypes.c_int64(0), None, None) == 1
    assert lib.csa2_index_score(None, 32, 128, None, None, None, None, None, None, 8, 2048,
                                None, ctypes.c_int64(0), None, None) == 1


def test_product_package_does_not_use_the_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_prefill_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f), encoding="utf8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle", txt, re.M), f
                assert "csa2_oracle" not in txt, f


def test_host_validation_of_replay_and_row_calls():
    from sparse_attention_prefill_gb300 import build
    lib = ctypes.CDLL(build.build())
    i64 = ctypes.c_int64
    # negative request count; ratio outside {1, 2}
    assert lib.csa2_encoder_replay_layout(-1, None, None, 128, 2, None, None, None, None, None,
                                          None, None, i64(0), None, None) == 1
    assert lib.csa2_encoder_replay_layout(0, None, None, 128, 3, None, None, None, None, None,
                                          None, None, i64(0), None, None) == 1
    # missing row map; nothing to copy; a row size that is not a multiple of 16
    assert lib.csa2_rows_gather(None, i64(4), None, None, i64(0), None, i64(16), None,
                                None) == 1
    assert lib.csa2_rows_scatter(None, i64(0), None, None, None, i64(0), i64(16), None,
                                 None) == 0
    fake = ctypes.c_void_p(4096)
    assert lib.csa2_rows_gather(None, i64(4), fake, fake, i64(8), fake, i64(24), None,
                                None) == 2


def test_status_and_flag_values_agree():
    """The header's status codes, data-error bits and format ids, the binding's
    constants and the oracle's own copy of the error bits name the same
    values (the three are written separately)."""
    import sparse_attention_prefill_gb300 as S
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    hdr = {m.group(1): int(m.group(2))
           for m in re.finditer(r"#define CSA2_(\w+)\s+(\d+)", src)}
    for name, val in hdr.items():
        if name.startswith(("OK", "ERR_", "DERR_", "FMT_")):
            assert getattr(S, name) == val, name
    bits = [v for k, v in hdr.items() if k.startswith("DERR_")]
    assert len(bits) == len(set(bits)) and all(b & (b - 1) == 0 for b in bits)
    osrc = open(os.path.join(ROOT, "oracle", "csa2_oracle.c")).read()
    for m in re.finditer(r"OR_ERR_(\w+) = (\d+)", osrc):
        assert hdr["DERR_" + m.group(1)] == int(m.group(2)), m.group(1)


def test_binding_argtypes_match_header_prototypes():
    """Every entry point's ctypes prototype in the binding has as many
    arguments as the header declares (catches signature drift)."""
    import sparse_attention_prefill_gb300 as S
    from sparse_attention_prefill_gb300 import build
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    protos = dict(re.findall(r"CSA2_API\s+(?:const\s+char\s*\*|int)\s*(csa2_\w+)\s*\(([^;]*)\)\s*;",
                             src, re.S))
    assert set(protos) == set(_declared())
    lib = S.load(build.build())
    for name, params in protos.items():
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(getattr(lib, name).argtypes) == n, name
    assert set(S.EXPORTED) == set(protos)


def test_missing_library_fails_loudly():
    """No CPU fallback: without libcsa2.so the binding raises instead of computing."""
    import subprocess
    import sys
    code = ("import sparse_attention_prefill_gb300 as S\n"
            "try:\n"
            "    S.load('/nonexistent/libcsa2.so')\n"
            "except S.Csa2Error as e:\n"
            "    print('raised:', e)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.startswith("raised:") and "not found" in r.stdout
