"""The C ABI library builds, loads and exports every declared symbol; host-side
argument checks answer without a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import _build
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pkv.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.lib()


def test_header_declares_the_path(lib):
    names = _declared()
    for want in ("pkv_slot_mapping", "pkv_kv_append", "pkv_copy_blocks", "pkv_gather_kv",
                 "pkv_paged_attention_decode", "pkv_attention_workspace_bytes", "pkv_spec_accept_greedy"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    assert set(_declared()) <= set(pkv._SIGS)


def test_error_and_status_strings(lib):
    assert lib.pkv_version() >= 100
    assert b"NULL" in lib.pkv_error_string(-1)
    assert b"workspace" in lib.pkv_error_string(-4)
    assert b"block" in lib.pkv_status_string(1)


def test_host_side_argument_checks(lib):
    f = lib.pkv_paged_attention_decode
    nullp = None
    args = dict(out=nullp, q=nullp, k=nullp, v=nullp, bt=nullp, max_blocks=4, sl=nullp, ql=nullp, num_seqs=2,
                total_q=2, max_q_len=1, max_seq_len=64, n_q=32, n_kv=8, d=128, bs=16, nb=10, scale=0.1, P=0, flags=0,
                ws=nullp, wsb=0, st=nullp, stream=nullp)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["max_blocks"], a["sl"], a["ql"], a["num_seqs"],
                 a["total_q"], a["max_q_len"], a["max_seq_len"], a["n_q"], a["n_kv"], a["d"], a["bs"], a["nb"], a["scale"], a["P"],
                 a["flags"], a["ws"], a["wsb"], a["st"], a["stream"])

    assert call(d=96) == -3                 # head_dim
    assert call(n_q=30) == -3               # n_q not a multiple of n_kv
    assert call(bs=24) == -3                # block_size not a power of two
    assert call(P=24) == -2                 # partition not a multiple of 16
    assert call(num_seqs=-1) == -2
    assert call(max_q_len=-1) == -2
    assert call(flags=8) == -2
    assert call() == -1                     # NULL pointers
    assert call(num_seqs=0) == 0            # nothing to do
    assert lib.pkv_kv_append(None, None, None, None, None, 3, 4, 16, 8, 100, None, None) == -3
    assert lib.pkv_spec_accept_greedy(None, None, 2, 0, 10, None, None, None, None) == -2
    assert lib.pkv_wait_selftest(0, None, None) == -2                  # limit out of range
    assert lib.pkv_wait_selftest(20_000_000_000, None, None) == -2
    assert lib.pkv_wait_selftest(1000, None, None) == -1               # status is required


def test_workspace_bytes_grow_with_partitions(lib):
    a = pkv.attention_workspace_bytes(256, 256, 32, 8, 128, 32768, 512)
    b = pkv.attention_workspace_bytes(256, 256, 32, 8, 128, 32768, 4096)
    assert a > b > 0
    assert a % 256 == 0
    assert pkv.attention_auto_partition(256, 256, 8, 32768) % 16 == 0
    # at most 1024 partitions per sequence in auto mode
    assert -(-2_000_000 // pkv.attention_auto_partition(1, 1, 8, 2_000_000)) <= 1024


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_23_gb300")
    for dp, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dp, fn)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, fn
                assert "pkv_oracle" not in txt, fn
