"""CPU checks of the C ABI: the library builds, loads, exports every entry point the header
declares, and the binding's struct layouts match the C compiler's. No GPU calls."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds_sampler.h")


def _lib():
    from canvas_sampler_gb300 import _lib as C
    if not os.path.exists(C.LIB_PATH):
        from canvas_sampler_gb300 import build
        build.build()
    return C


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_what_the_binding_binds():
    C = _lib()
    assert _declared_functions() == sorted(C.SIGNATURES)


def test_library_exports_every_declared_symbol():
    C = _lib()
    lib = ctypes.CDLL(C.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings_without_gpu():
    C = _lib()
    lib = C.load_library()
    assert lib.ds_abi_version() == 4
    for code in range(7):
        assert lib.ds_status_string(code)
    assert lib.ds_status_string(99) == b"unknown status"


def test_create_rejects_bad_config_before_touching_the_device():
    C = _lib()
    lib = C.load_library()
    cfg = C.ds_sampler_config(max_batch=1, canvas_len=100, d_model=256, dtype=0, vocab=4096,
                              top_k=0, max_steps=48, impl=0)
    h = ctypes.c_void_p()
    assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_INVALID_ARG
    assert lib.ds_sampler_create(None, ctypes.byref(h)) == C.DS_ERR_INVALID_ARG
    assert lib.ds_sampler_destroy(None) == C.DS_OK


PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "ds_sampler.h"
#define P(T, F) printf("%s.%s %zu\n", #T, #F, offsetof(T, F));
int main(void) {
  printf("ds_sampler_config %zu\nds_step_args %zu\nds_loop_args %zu\nds_block_args %zu\n",
         sizeof(ds_sampler_config), sizeof(ds_step_args), sizeof(ds_loop_args),
         sizeof(ds_block_args));
  printf("ds_shard_partial %zu\nds_shard_row %zu\nds_shard_best %zu\nds_shard_cand %zu\n",
         sizeof(ds_shard_partial), sizeof(ds_shard_row), sizeof(ds_shard_best),
         sizeof(ds_shard_cand));
  P(ds_shard_partial, O) P(ds_shard_partial, cand)
  P(ds_sampler_config, vocab) P(ds_sampler_config, top_k) P(ds_sampler_config, lock_rule)
  P(ds_sampler_config, entropy_budget) P(ds_sampler_config, t_end)
  P(ds_step_args, seed) P(ds_step_args, H) P(ds_step_args, argmax) P(ds_step_args, prev_argmax)
  P(ds_loop_args, h_mode) P(ds_loop_args, W) P(ds_loop_args, H_buf)
  P(ds_block_args, n_blocks) P(ds_block_args, first_block) P(ds_block_args, init_canvas)
  P(ds_block_args, out_steps)
  return 0;
}
"""


def test_struct_layouts_match_c(tmp_path):
    C = _lib()
    src = tmp_path / "probe.c"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    r = subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip(f"no C compiler: {r.stderr[:200]}")
    got = dict(line.split() for line in subprocess.check_output([str(exe)], text=True).splitlines())
    assert int(got["ds_sampler_config"]) == ctypes.sizeof(C.ds_sampler_config)
    assert int(got["ds_step_args"]) == ctypes.sizeof(C.ds_step_args)
    assert int(got["ds_loop_args"]) == ctypes.sizeof(C.ds_loop_args)
    assert int(got["ds_block_args"]) == ctypes.sizeof(C.ds_block_args)
    assert int(got["ds_shard_partial"]) == ctypes.sizeof(C.ds_shard_partial)
    assert int(got["ds_shard_row"]) == C.SHARD_ROW_BYTES
    assert int(got["ds_shard_best"]) == C.SHARD_BEST_BYTES
    assert int(got["ds_shard_cand"]) == C.SHARD_CAND_BYTES
    for key, val in got.items():
        if "." in key:
            t, f = key.split(".")
            assert getattr(getattr(C, t), f).offset == int(val), key


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "canvas_sampler_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, re.M), f
    # importing the product (every module of the package) loads no oracle module
    code = ("import sys, importlib, pkgutil, canvas_sampler_gb300 as p\n"
            "for m in pkgutil.iter_modules(p.__path__):\n"
            "    if m.name != 'build':\n"
            "        importlib.import_module('canvas_sampler_gb300.' + m.name)\n"
            "bad = [n for n in sys.modules if n == 'oracle' or n.startswith('oracle.')]\n"
            "assert not bad, bad\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
