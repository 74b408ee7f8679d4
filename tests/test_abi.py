"""The C ABI library builds, loads on a machine without a GPU, and exports
every entry point include/*.h declares; the headers are valid C; the product
package never reaches the oracle.  No GPU compute call is made here."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def _declared():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_pa_gb300.build import build
    path = build()
    return ctypes.CDLL(path), path


def test_header_declares_the_operations():
    names = _declared()
    for op in ("pa_cache_write", "pa_decode_attention", "pa_copy_blocks", "pa_swap_blocks",
               "pa_decode_workspace_size", "pa_status_string", "pa_bm_create",
               "pa_bm_seq_append", "pa_bm_swap_out"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    cdll, path = lib
    for name in _declared():
        assert hasattr(cdll, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True)
    exported = set(re.findall(r"\sT\s+(pa_\w+)", out.stdout))
    assert set(_declared()) <= exported


@pytest.mark.parametrize("header", HEADERS, ids=os.path.basename)
def test_header_is_plain_c(header):
    subprocess.run(["gcc", "-fsyntax-only", "-std=c99", "-Wall", "-Werror", "-x", "c", header],
                   check=True)


def test_status_strings_and_workspace_size(lib):
    import paged_kv_cache_pa_gb300 as pa
    assert pa.status_string(0) == "PA_OK"
    assert pa.status_string(4) == "PA_ERR_WORKSPACE"
    a = pa.decode_workspace_size(256, 40, 40, 128, 2048)
    assert a == pa.decode_workspace_size(256, 40, 40, 128, 2048) > 0
    # a larger bound never needs less workspace
    assert pa.decode_workspace_size(256, 40, 40, 128, 4096) >= a
    assert pa.decode_workspace_size(-1, 40, 40, 128, 2048) == 0


def test_product_package_does_not_use_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_pa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "pa_oracle" not in src, f


def test_error_bits_match_the_header():
    """The binding's error-word bits are the header's PA_ERRBIT_* values."""
    import paged_kv_cache_pa_gb300 as pa
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    bits = {name: int(v) for name, v in re.findall(r"#define PA_ERRBIT_(\w+)\s+(\d+)u", text)}
    assert set(bits) == {"BLOCK_OOB", "SLOT_OOB", "CONTEXT_LEN", "TIMEOUT", "INTERNAL"}
    for name, v in bits.items():
        assert getattr(pa, "ERRBIT_" + name) == v, name
    assert len(set(bits.values())) == len(bits)
    assert all(v & (v - 1) == 0 for v in bits.values())   # one bit each


@pytest.mark.parametrize("S,H,Hkv,D,max_len,launches", [
    (4, 8, 8, 64, 116, 1),        # small batch: the attention kernel alone, no plan
    (128, 2, 2, 64, 255, 1),      # 256 (sequence, KV head) pairs, one partition each
    (129, 2, 2, 64, 255, 2),      # 258 pairs: plan + attention
    (32, 64, 8, 128, 256, 1),     # query groups of 8 (no shared-prefix items), 256 tokens
    (32, 64, 8, 128, 257, 3),     # two partitions: plan + attention + merge
    (4, 8, 8, 64, 300, 4),        # shared prefixes may form (G = 1): plan + both kernels + merge
    (256, 40, 40, 128, 1227, 4),  # the OPT-13B-shaped batch
    (64, 12, 2, 128, 3991, 3),    # the grouped-query batch
    (0, 8, 8, 64, 100, 0),        # invalid sizes
    (4, 12, 5, 64, 100, 0),
])
def test_kernel_launch_counts_follow_the_host_rules(lib, S, H, Hkv, D, max_len, launches):
    """pa_decode_kernel_launches (host only): which kernels a call enqueues."""
    import paged_kv_cache_pa_gb300 as pa
    assert pa.decode_kernel_launches(S, H, Hkv, D, max_len) == launches
