"""ctypes binding of the sampler's C ABI (include/ds_sampler.h). Argument marshalling only.

The raw entry points keep their C names (``ds_sampler_create``, ``ds_sampler_step``, ...).
Loading fails loudly when the shared library has not been built: there is no other path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int32, c_int64, c_size_t, c_uint8, c_uint32, c_uint64, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libds_sampler.so")

DS_OK = 0
DS_ERR_INVALID_ARG = 1
DS_ERR_UNSUPPORTED = 2
DS_ERR_CUDA = 3
DS_ERR_TIMEOUT = 4
DS_ERR_OOM = 5
DS_ERR_DEVICE = 6

DS_DTYPE_BF16 = 0
DS_DTYPE_FP32 = 1
DS_IMPL_AUTO = 0
DS_IMPL_TENSOR = 1
DS_IMPL_SIMT = 2
DS_IMPL_FUSED = 3
DS_H_FIXED = 0
DS_H_STANDIN = 1
DS_LOCK_THRESHOLD = 0
DS_LOCK_ENTROPY_BUDGET = 1


class ds_sampler_config(ctypes.Structure):
    _fields_ = [("max_batch", c_int32), ("canvas_len", c_int32), ("d_model", c_int32),
                ("dtype", c_int32), ("vocab", c_int64), ("top_k", c_int32),
                ("max_steps", c_int32), ("impl", c_int32), ("lock_rule", c_int32),
                ("entropy_budget", ctypes.c_float), ("stop_entropy", ctypes.c_float),
                ("t_start", ctypes.c_float), ("t_end", ctypes.c_float)]


class ds_step_args(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("reserved", c_int32), ("seed", c_uint64), ("H", c_void_p),
                ("E", c_void_p), ("temperature", c_void_p), ("tau", c_void_p), ("step", c_void_p),
                ("canvas", c_void_p), ("lock", c_void_p), ("done", c_void_p), ("s", c_void_p),
                ("sampled", c_void_p), ("conf", c_void_p), ("entropy", c_void_p),
                ("argmax", c_void_p), ("prev_argmax", c_void_p)]


class ds_loop_args(ctypes.Structure):
    _fields_ = [("step", ds_step_args), ("h_mode", c_int32), ("max_iters", c_int32),
                ("use_graph", c_int32), ("reserved", c_int32), ("W", c_void_p), ("H_buf", c_void_p)]


class ds_block_args(ctypes.Structure):
    _fields_ = [("loop", ds_loop_args), ("n_blocks", c_int32), ("first_block", c_int32),
                ("init_canvas", c_void_p), ("out_canvas", c_void_p), ("out_steps", c_void_p)]


class ds_shard_partial(ctypes.Structure):
    _fields_ = [("rows", c_void_p), ("best", c_void_p), ("O", c_void_p), ("cand", c_void_p)]


# bytes of one record of each part of a shard's partial (ds_shard_row, ds_shard_best,
# ds_shard_cand)
SHARD_ROW_BYTES = 16
SHARD_BEST_BYTES = 16
SHARD_CAND_BYTES = 8

# name -> (restype, argtypes): every function declared in include/ds_sampler.h
SIGNATURES = {
    "ds_abi_version": (c_int32, []),
    "ds_status_string": (c_char_p, [c_int32]),
    "ds_last_cuda_error": (c_char_p, []),
    "ds_sampler_create": (c_int32, [POINTER(ds_sampler_config), POINTER(c_void_p)]),
    "ds_sampler_destroy": (c_int32, [c_void_p]),
    "ds_sampler_workspace_bytes": (c_int32, [c_void_p, POINTER(c_size_t)]),
    "ds_sampler_impl": (c_int32, [c_void_p, POINTER(c_int32)]),
    "ds_sampler_step": (c_int32, [c_void_p, POINTER(ds_step_args), c_void_p]),
    "ds_sampler_step_host": (c_int32, [c_void_p, POINTER(ds_step_args), c_void_p]),
    "ds_denoise_loop": (c_int32, [c_void_p, POINTER(ds_loop_args), c_void_p]),
    "ds_block_loop": (c_int32, [c_void_p, POINTER(ds_block_args), c_void_p]),
    "ds_standin_hidden": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_int32, c_void_p]),
    "ds_sampler_device_status": (c_int32, [c_void_p, POINTER(c_int32)]),
    "ds_philox4x32_10": (c_int32, [c_void_p, c_uint64, c_void_p, c_int64, c_void_p]),
    "ds_sampler_debug_buffer": (c_int32, [c_void_p, c_int32, POINTER(c_void_p), POINTER(c_size_t)]),
    "ds_sampler_set_phase_timing": (c_int32, [c_void_p, c_int32]),
    "ds_sampler_phase_times": (c_int32, [c_void_p, POINTER(ctypes.c_float), c_int32, POINTER(c_int32)]),
    "ds_sampler_launch_count": (c_int32, [c_void_p, POINTER(c_int64)]),
    "ds_sampler_selftest_wait": (c_int32, [c_void_p, c_int64, c_void_p]),
    "ds_sampler_step_noalloc": (c_int32, [POINTER(ds_sampler_config), POINTER(ds_step_args), c_void_p]),
    "ds_sampler_noalloc_status": (c_int32, [c_void_p, POINTER(c_int32)]),
    "ds_sampler_step_shard": (c_int32, [c_void_p, POINTER(ds_step_args), c_int32, c_int64,
                                        POINTER(ds_shard_partial), c_void_p]),
    "ds_merge_shards": (c_int32, [c_void_p, POINTER(ds_step_args), c_int32,
                                  POINTER(ds_shard_partial), c_int64, c_void_p]),
}

PHASES = ["logits", "stats", "topk", "convert", "selfcond", "finalize", "lock"]

_lib = None


class DsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the built library (once). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"sampler library not built: {path} is missing "
                           "(run `python -m canvas_sampler_gb300.build`)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().ds_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != DS_OK:
        if status in (DS_ERR_CUDA, DS_ERR_OOM):
            what = f"{what} [{load_library().ds_last_cuda_error().decode()}]"
        raise DsError(status, what)


def __getattr__(name):  # expose the raw C entry points under their C names
    if name in SIGNATURES:
        return getattr(load_library(), name)
    raise AttributeError(name)
