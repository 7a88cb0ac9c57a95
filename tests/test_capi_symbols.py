"""The C-ABI library loads without a GPU and exports every entry point that
include/pkv.h declares (and the Python binding binds each of them)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    return sorted(set(re.findall(r"^PKV_API[^(]*?\b(pkv_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_contract():
    names = declared()
    for n in ["pkv_pool_new", "pkv_alloc_block", "pkv_unref_block", "pkv_seq_new", "pkv_seq_fork",
              "pkv_seq_truncate", "pkv_ensure_append", "pkv_ensure_append_batch", "pkv_advance",
              "pkv_advance_batch", "pkv_attn_with_paged", "pkv_attn_batch", "pkv_attn_contiguous",
              "pkv_append_layer", "pkv_sync_error"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    import paged_kv_gqa_nx_gb300 as pkv
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    missing = [n for n in declared() if n not in exported]
    assert not missing, missing
    extra = sorted(n for n in exported if n.startswith("pkv_") and n not in declared())
    assert not extra, extra
    assert sorted(pkv.exported_symbols()) == declared()


def test_binding_has_every_entry_point():
    import paged_kv_gqa_nx_gb300 as pkv
    for n in declared():
        assert callable(getattr(pkv, n)), n
