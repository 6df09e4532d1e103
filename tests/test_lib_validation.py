"""Argument checks of the C ABI that run before any CUDA call, so they are exercised here
without a GPU: the configuration checks shared by ds_sampler_create and the no-allocation step
(everything but max_batch), and the no-allocation step's refusal of the fused pass."""
import ctypes
import math

import pytest

from canvas_sampler_gb300 import _lib as C


@pytest.fixture(scope="module")
def lib():
    try:
        return C.load_library()
    except RuntimeError as e:  # not built here
        pytest.skip(str(e))


def _cfg(**kw):
    base = dict(max_batch=1, canvas_len=256, d_model=256, dtype=0, vocab=4096, top_k=0,
                max_steps=48, impl=0)
    base.update(kw)
    return C.ds_sampler_config(**base)


BAD = [dict(canvas_len=100), dict(canvas_len=2048), dict(vocab=1000), dict(vocab=1 << 25),
       dict(d_model=48), dict(dtype=7), dict(top_k=-1), dict(top_k=257), dict(max_steps=0),
       dict(max_steps=(1 << 28) + 1), dict(impl=9), dict(lock_rule=5),
       dict(entropy_budget=-0.1), dict(stop_entropy=-1.0), dict(entropy_budget=math.nan),
       dict(t_start=0.8, t_end=0.0), dict(t_start=0.8, t_end=math.nan)]


@pytest.mark.parametrize("bad", BAD, ids=[",".join(f"{k}={v}" for k, v in b.items()) for b in BAD])
def test_invalid_configs_are_refused_by_both_entry_points(lib, bad):
    cfg = _cfg(**bad)
    h = ctypes.c_void_p()
    assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_INVALID_ARG
    assert not h.value
    a = C.ds_step_args()
    a.batch = 1
    assert lib.ds_sampler_step_noalloc(ctypes.byref(cfg), ctypes.byref(a), None) == \
        C.DS_ERR_INVALID_ARG


def test_topk_pool_beyond_the_limit_is_unsupported(lib):
    cfg = _cfg(vocab=1 << 20, top_k=256)  # 128 chunks x 256 candidates > 8192
    h = ctypes.c_void_p()
    assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_UNSUPPORTED
    a = C.ds_step_args()
    a.batch = 1
    assert lib.ds_sampler_step_noalloc(ctypes.byref(cfg), ctypes.byref(a), None) == \
        C.DS_ERR_UNSUPPORTED


def test_no_alloc_step_refuses_the_fused_pass(lib):
    cfg = _cfg(impl=C.DS_IMPL_FUSED)
    a = C.ds_step_args()
    a.batch = 1
    assert lib.ds_sampler_step_noalloc(ctypes.byref(cfg), ctypes.byref(a), None) == \
        C.DS_ERR_UNSUPPORTED
