"""The C-ABI library builds, loads and exports every entry point include/echo.h
declares; the Python binding's struct layouts match the header's; host-side
argument checks reject bad calls before anything reaches a GPU.  No GPU needed."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "echo.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return echo.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(echo_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("echo_indexer_score", "echo_select_topk", "echo_prefetch_recall", "echo_pool_alloc",
                 "echo_pool_evict", "echo_pool_init", "echo_decode_step", "echo_ema_update", "echo_append"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (echo_\w+)", out))
    assert set(declared_functions()) <= exported


def test_struct_layouts_match_the_header():
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "echo.h"
#define P(T, F) printf(#T "." #F " %zu\n", offsetof(T, F));
int main(void) {
  printf("echo_pool %zu\n", sizeof(echo_pool));
  printf("echo_workspace %zu\n", sizeof(echo_workspace));
  printf("echo_stats %zu\n", sizeof(echo_stats));
  printf("echo_stage %zu\n", sizeof(echo_stage));
  printf("echo_indexer_args %zu\n", sizeof(echo_indexer_args));
  printf("echo_step_args %zu\n", sizeof(echo_step_args));
  printf("echo_prefill_args %zu\n", sizeof(echo_prefill_args));
  printf("echo_mla_args %zu\n", sizeof(echo_mla_args));
  P(echo_pool, counters) P(echo_pool, host_kv) P(echo_pool, row_elems) P(echo_workspace, max_rows)
  P(echo_stage, cap_div)
  P(echo_stage, reserve) P(echo_stage, reserve_ctl) P(echo_stage, reserve_cap) P(echo_stage, flags)
  P(echo_prefill_args, scores) P(echo_prefill_args, s_shift) P(echo_prefill_args, k) P(echo_prefill_args, thr_bin)
  P(echo_prefill_args, stage) P(echo_prefill_args, dev_status)
  P(echo_mla_args, scale) P(echo_mla_args, workspace_bytes) P(echo_mla_args, dev_status)
  P(echo_indexer_args, scores) P(echo_indexer_args, dev_status) P(echo_step_args, k) P(echo_step_args, alpha)
  P(echo_step_args, clock) P(echo_step_args, advance_clock) P(echo_step_args, stage_events)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(prog)
        subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        lines = dict(l.rsplit(" ", 1) for l in subprocess.check_output([exe], text=True).splitlines())
    sizes = {"echo_pool": echo.c_pool, "echo_workspace": echo.c_workspace, "echo_stage": echo.c_stage,
             "echo_indexer_args": echo.c_indexer_args, "echo_step_args": echo.c_step_args,
             "echo_prefill_args": echo.c_prefill_args, "echo_mla_args": echo.c_mla_args}
    for name, cls in sizes.items():
        assert int(lines[name]) == ctypes.sizeof(cls), name
    assert int(lines["echo_stats"]) == 8 * len(echo.STAT_FIELDS)
    for key, v in lines.items():
        if "." in key:
            sname, field = key.split(".")
            assert getattr(sizes[sname], field).offset == int(v), key


def test_metadata_law_and_version(lib):
    assert lib.echo_metadata_bytes(2_000_000, 200_000) == 4 * 2_000_000 + 13 * 200_000
    assert echo.version() >> 16 == 1


def test_argument_checks_reject_before_any_launch(lib):
    P = ctypes.c_void_p
    assert lib.echo_select_topk(16, 16, 1, 1, 10, 0, 16, 16, None) == echo.ECHO_EINVAL        # k = 0
    assert b"k must be" in lib.echo_last_error_string()
    assert lib.echo_select_topk(16, 16, 1, 0, 10, 8, 16, 16, None) == echo.ECHO_EINVAL        # n_q = 0
    assert lib.echo_select_topk(16, 16, 1, 65537, 10, 8, 16, 16, None) == echo.ECHO_EINVAL    # n_q too large
    assert lib.echo_select_topk(None, 16, 1, 1, 10, 8, 16, 16, None) == echo.ECHO_EINVAL      # NULL
    a = echo.c_indexer_args(16, 16, 24, 16, 1, 1, 128, 16, None, None, None, None, None)       # misaligned k
    assert lib.echo_indexer_score(ctypes.byref(a), None) == echo.ECHO_EINVAL
    assert b"16-byte" in lib.echo_last_error_string()
    a = echo.c_indexer_args(16, 16, 32, 16, 1, 1, 128, 16, 16, None, None, None, None)         # prefetch w/o pool
    assert lib.echo_indexer_score(ctypes.byref(a), None) == echo.ECHO_EINVAL
    assert lib.echo_ema_update(16, 16, 4, ctypes.c_float(1.5), None) == echo.ECHO_EINVAL       # alpha > 1
    assert lib.echo_ema_update_strided(16, 16, 4, 0, ctypes.c_float(0.5), None) == echo.ECHO_EINVAL  # stride 0
    a = echo.c_prefill_args(16, 16, 16, 16, 1, 0, 128, 16)                                     # C = 0
    assert lib.echo_prefill_indexer_score(ctypes.byref(a), None) == echo.ECHO_EINVAL
    a = echo.c_prefill_args(16, 24, 16, 16, 1, 4, 128, 16)                                     # misaligned w
    assert lib.echo_prefill_indexer_score(ctypes.byref(a), None) == echo.ECHO_EINVAL
    a = echo.c_prefill_args(16, 16, 16, 16, 1, 4, 128, 16, 16, 0)                               # s_shift, k = 0
    assert lib.echo_prefill_indexer_score(ctypes.byref(a), None) == echo.ECHO_EINVAL
    m = echo.c_mla_args(16, 16, 10, 16, 1, 1, 0, ctypes.c_float(0.1), 16, 16, 256, 1 << 30)      # k = 0
    assert lib.echo_sparse_mla_decode(ctypes.byref(m), None) == echo.ECHO_EINVAL
    m = echo.c_mla_args(16, 16, 10, 16, 1, 1, 64, ctypes.c_float(0.1), 16, 16, 256, 16)          # small workspace
    assert lib.echo_sparse_mla_decode(ctypes.byref(m), None) == echo.ECHO_EINVAL
    assert b"workspace" in lib.echo_last_error_string()
    n = ctypes.c_size_t()
    # MLA scratch: per CTA of 128 selected rows its 128 x 512 fp16 partial output and
    # its max / sum per head (fp32)
    assert lib.echo_mla_workspace_bytes(8, 1, 2048, ctypes.byref(n)) == echo.ECHO_OK
    assert n.value == 8 * 16 * 128 * (512 * 2 + 2 * 4)
    assert lib.echo_mla_workspace_bytes(2, 1, 300, ctypes.byref(n)) == echo.ECHO_OK       # 3 CTAs each
    assert n.value == 2 * 3 * 128 * (512 * 2 + 2 * 4)
    assert lib.echo_mla_workspace_bytes(1, 1, 8193, ctypes.byref(n)) == echo.ECHO_EINVAL
    assert lib.echo_workspace_bytes(0, 10, ctypes.byref(n)) == echo.ECHO_EINVAL
    assert lib.echo_workspace_bytes(1000, 10, ctypes.byref(n)) == echo.ECHO_OK and n.value >= 4 * 1010
    pool = echo.c_pool(0, 10, 16, 16, 16, 16, 16, 16, 16, 16)                                  # n_g = 0
    assert lib.echo_pool_init(ctypes.byref(pool), None) == echo.ECHO_EINVAL
    for bad in (12, -8, 65544):                                                               # row sizes
        pool = echo.c_pool(10, 10, 16, 16, 16, 16, 16, 16, 16, 16, bad)
        assert lib.echo_pool_init(ctypes.byref(pool), None) == echo.ECHO_EINVAL
        assert b"row_elems" in lib.echo_last_error_string()
    assert lib.echo_decode_step(None, None) == echo.ECHO_EINVAL


def test_host_input_calls_reject_bad_arguments_before_any_cuda_work():
    """The host-input step and the step graph check their arguments on the host: no
    args, no host buffers, no device clock, a missing graph; destroying NULL is a no-op."""
    lib = echo.load_library()
    buf = (ctypes.c_uint8 * 64)()
    assert lib.echo_decode_step_host(None, buf, buf, None, 1) == echo.ECHO_EINVAL
    a = echo.c_step_args()
    assert lib.echo_decode_step_host(ctypes.byref(a), None, buf, None, 1) == echo.ECHO_EINVAL
    assert b"q_host" in lib.echo_last_error_string()
    h = ctypes.c_void_p(1234)
    assert lib.echo_step_graph_create(None, ctypes.byref(h)) == echo.ECHO_EINVAL and h.value is None
    assert lib.echo_step_graph_create(ctypes.byref(a), None) == echo.ECHO_EINVAL
    assert lib.echo_step_graph_create(ctypes.byref(a), ctypes.byref(h)) == echo.ECHO_EINVAL
    assert b"clock_dev" in lib.echo_last_error_string() and h.value is None
    assert lib.echo_step_graph_launch(None, None, None, None, 0) == echo.ECHO_EINVAL
    assert lib.echo_step_graph_destroy(None) == echo.ECHO_OK


def test_product_path_fails_loudly_without_the_library(tmp_path):
    code = ("import sparse_attention_kv_fp8_gb300 as e\n"
            "try:\n    e.load_library(%r)\nexcept e.EchoError as x:\n    print('raised', x)\n" % str(tmp_path / "nope.so"))
    out = subprocess.run(["python", "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "raised" in out.stdout
