"""CPU checks of the boundary: libpa.so builds for sm_103a, loads, and
exports every function include/pa.h declares (no compute call: no GPU here);
the host step-metadata builder matches the oracle's literal one bit for bit.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_82_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ("pa_reshape_and_cache", "pa_attention", "pa_copy_blocks",
              "pa_attention_workspace_size", "pa_get_device_error",
              "pa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} not exported by libpa.so"


def _boundary_table_doc():
    """The repository document that holds the boundary table (found by the
    table's heading among the top-level Markdown files)."""
    marker = "**The boundary against the proposed header.**"
    for name in sorted(os.listdir(ROOT)):
        if name.endswith(".md"):
            text = open(os.path.join(ROOT, name)).read()
            if marker in text:
                return text, marker
    raise AssertionError("no top-level document holds the boundary table")


def test_exports_match_the_boundary_table():
    """The design notes' boundary table lists every entry point of pa.h (the
    proposed declarations mapped to the header's); nothing is missing and
    nothing extra is exported."""
    text, marker = _boundary_table_doc()
    start = text.index(marker)
    table = text[start:text.index("\n\n", text.index("| proposed |", start))]
    in_table = set()
    for line in table.splitlines()[2:]:
        cells = line.split("|")
        if len(cells) > 2 and line.startswith("|"):
            in_table |= set(re.findall(r"`(pa_[a-z_]+)", cells[2]))
    assert in_table == set(_declared())


def test_binding_names_match_the_abi():
    import paged_kv_cache_82_gb300 as pa
    for name in _declared():
        if name != "pa_status_string":
            assert callable(getattr(pa, name)), name


def test_status_strings(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(4) == b"PA_ERR_DEVICE"
    assert lib.pa_status_string(99) == b"PA_ERR_UNKNOWN"


def test_product_has_no_oracle_dependency():
    """The CUDA path and the oracle share no code: nothing in the package
    imports or links the oracle."""
    pkg = os.path.join(ROOT, "paged_kv_cache_82_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def _req_sets():
    yield workloads.config1().requests
    import random
    rnd = random.Random(3)
    for _ in range(20):
        reqs = []
        nxt = 0
        for _ in range(rnd.randint(1, 9)):
            L = rnd.randint(1, 200)
            n = rnd.randint(0, L)
            nb = -(-L // 16)
            reqs.append(workloads.Request(list(range(nxt, nxt + nb)), L - n, n))
            nxt += nb
        yield reqs


def test_step_metadata_matches_oracle_bit_exact():
    from paged_kv_cache_82_gb300.metadata import build_step_metadata
    for reqs in _req_sets():
        a = build_step_metadata(reqs)
        b = oracle.step_metadata(reqs)
        for k in ("query_start_loc", "seq_lens", "block_tables",
                  "slot_mapping"):
            assert a[k].dtype == b[k].dtype, k
            np.testing.assert_array_equal(a[k], b[k])
        assert a["max_query_len"] == b["max_query_len"]
        assert a["max_seq_len"] == b["max_seq_len"]


@pytest.mark.gpu
def test_workspace_size_grows_with_the_step_and_stays_bounded():
    """The workspace depends on host-known sizes only: it never shrinks when
    the step grows, it is the partial-slot floor plus a few bytes per request
    and per query token, and the benchmark steps fit the fixed scratch of
    pa_attention_noalloc."""
    import paged_kv_cache_82_gb300 as pa
    ws = pa.pa_attention_workspace_size
    floor = ws(1, 32, 8, 128, 1, 1, 16)
    prev = 0
    for B in (1, 2, 64, 512, 4096):
        n = ws(B, 32, 8, 128, B, 1, 4096)
        assert n >= prev and n >= floor
        # decode only: lists of O(1) bytes per (request, KV head)
        assert n - floor <= B * 8 * 64 + (1 << 16)
        prev = n
    # a longer context needs no more workspace (its pages are walked, not
    # stored); more query rows (prefill tiles) need more
    assert ws(64, 32, 8, 128, 64, 1, 131072) == ws(64, 32, 8, 128, 64, 1, 512)
    assert ws(1142, 32, 8, 128, 121, 1022, 8193) > ws(121, 32, 8, 128, 121, 1,
                                                      8193)
    from tests.test_zz_no_alloc import pa_scratch_bytes
    scratch = pa_scratch_bytes()
    for T, Hq, Hkv, B, mq, ms in ((64, 32, 8, 64, 1, 4096),        # decode
                                  (1142, 32, 8, 121, 1022, 10193),  # mixed
                                  (32, 32, 32, 32, 1, 8192),       # MHA
                                  (16, 64, 8, 16, 1, 131073)):     # FP8 long
        assert ws(T, Hq, Hkv, 128, B, mq, ms) <= scratch
    with pytest.raises(pa.PaError):
        ws(1, 7, 2, 128, 1, 1, 16)        # heads not a multiple
    with pytest.raises(pa.PaError):
        ws(1, 8, 2, 96, 1, 1, 16)         # head_dim


def test_launch_count_without_a_gpu(lib):
    n = ctypes.c_uint64(123)
    lib.pa_launch_count.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    assert lib.pa_launch_count(ctypes.byref(n)) == 0
    assert n.value == 0  # nothing launched from this thread
    lib.pa_launch_count.argtypes = [ctypes.c_void_p]
    assert lib.pa_launch_count(None) == 1  # PA_ERR_INVALID_ARG


def test_attention_flops_counts_visible_pairs():
    # two requests: 3 new tokens after 5 cached (keys 6, 7, 8 visible) and a
    # 1-token decode over 4 keys
    wl = workloads.decode_step("f", 1, seq_lens=[8, 4], q_lens=[3, 1],
                               num_q_heads=2, num_kv_heads=1, head_dim=8,
                               num_blocks=4, dtype="bf16", cache_dtype="bf16")
    assert workloads.attention_flops(wl) == (6 + 7 + 8 + 4) * 2 * 8 * 4


def test_common_prefix_blocks():
    """Leading block ids shared by every request, cut to the full blocks
    before each request's first new token."""
    from paged_kv_cache_82_gb300.metadata import common_prefix_blocks
    from workloads import Request
    a = Request([7, 3, 9, 11, 4], 70, 1)       # 4 full blocks cached
    b = Request([7, 3, 9, 12], 50, 1)          # shares 3, 3 full blocks
    c = Request([7, 3, 9, 11, 5, 6], 90, 2)    # shares 4
    assert common_prefix_blocks([a, c]) == 4
    assert common_prefix_blocks([a, b, c]) == 3
    assert common_prefix_blocks([a, Request([7, 3, 9, 11], 40, 8)]) == 2  # cut
    assert common_prefix_blocks([Request([1, 2], 20, 1), Request([2, 1], 20, 1)]) == 0
    assert common_prefix_blocks([a]) == 4
    assert common_prefix_blocks([]) == 0


def test_cascade_policy():
    """The cascade is chosen only where it measured faster: at least two
    decode requests, and a long prefix or many requests behind it."""
    from paged_kv_cache_82_gb300.metadata import (
        CASCADE_MIN_BLOCK_READS, CASCADE_MIN_BLOCKS, cascade_prefix_blocks)
    from workloads import Request

    def step(prefix, n_dec, q=1, extra=()):
        shared = list(range(prefix))
        reqs = [Request(shared + [10000 + i], prefix * 16 + 5, q)
                for i in range(n_dec)]
        return reqs + list(extra)

    assert cascade_prefix_blocks(step(600, 1), 4) == 0           # nothing shared
    assert cascade_prefix_blocks(step(600, 2), 4) == 600
    assert cascade_prefix_blocks(step(256, 2), 4) == 0
    assert cascade_prefix_blocks(step(128, 64), 4) == 128
    assert cascade_prefix_blocks(step(128, 32), 4) == 0
    assert 128 * 64 >= CASCADE_MIN_BLOCK_READS > 128 * 32
    assert 600 >= CASCADE_MIN_BLOCKS > 256
    # query rows: q_len x group <= 8 is a decode (G = 4: two tokens)
    assert cascade_prefix_blocks(step(600, 2, q=2), 4) == 600
    assert cascade_prefix_blocks(step(600, 2, q=3), 4) == 0
    # a prefill request behind the same prefix counts for the prefix, not
    # as a reader of it
    pf = Request(list(range(600)) + [20000, 20001], 600 * 16, 30)
    assert cascade_prefix_blocks(step(600, 1, extra=[pf]), 4) == 0
    assert cascade_prefix_blocks(step(600, 2, extra=[pf]), 4) == 600
    # FP8 caches: many requests behind the prefix, whatever its length;
    # 4-bit caches have no cascade path
    from paged_kv_cache_82_gb300.metadata import CASCADE_MIN_BLOCK_READS_FP8
    assert cascade_prefix_blocks(step(1024, 8), 4, "e4m3") == 0
    assert cascade_prefix_blocks(step(1024, 16), 4, "e4m3") == 1024
    assert cascade_prefix_blocks(step(128, 128), 4, "e4m3") == 128
    assert cascade_prefix_blocks(step(128, 64), 4, "e4m3") == 0
    assert 128 * 128 >= CASCADE_MIN_BLOCK_READS_FP8 > 128 * 64
    assert cascade_prefix_blocks(step(600, 64), 4, "int4") == 0
    assert cascade_prefix_blocks(step(600, 64), 4, "nvfp4") == 0
