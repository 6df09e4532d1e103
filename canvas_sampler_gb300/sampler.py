"""Python front end of the C ABI: PyTorch tensors in, pointers out. No computation here.

PyTorch only provides device memory and streams; every step of the sampler runs in the
library's CUDA kernels.
"""
from __future__ import annotations

from ctypes import byref, c_int32, c_size_t, c_void_p
from dataclasses import dataclass

import torch

from . import _lib as C

_DTYPES = {"bf16": (C.DS_DTYPE_BF16, torch.bfloat16), "fp32": (C.DS_DTYPE_FP32, torch.float32)}
_IMPLS = {"auto": C.DS_IMPL_AUTO, "tensor": C.DS_IMPL_TENSOR, "simt": C.DS_IMPL_SIMT,
          "fused": C.DS_IMPL_FUSED}
_LOCK_RULES = {"threshold": C.DS_LOCK_THRESHOLD, "entropy_budget": C.DS_LOCK_ENTROPY_BUDGET}


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class CanvasState:
    """Loop state of B canvases (device tensors, updated in place by each step)."""
    canvas: torch.Tensor  # [B, L] int32
    lock: torch.Tensor  # [B, L] uint8
    step: torch.Tensor  # [B] int32
    done: torch.Tensor  # [B] uint8
    prev_argmax: torch.Tensor | None = None  # [B, L] int32 (entropy-budget rule)

    @staticmethod
    def from_numpy(canvas, lock, step, done, device="cuda", prev_argmax=None):
        c = torch.as_tensor(canvas, dtype=torch.int32).to(device).contiguous()
        pa = (torch.full_like(c, -1) if prev_argmax is None else
              torch.as_tensor(prev_argmax, dtype=torch.int32).to(device).contiguous())
        return CanvasState(c, torch.as_tensor(lock, dtype=torch.uint8).to(device).contiguous(),
                           torch.as_tensor(step, dtype=torch.int32).to(device).contiguous(),
                           torch.as_tensor(done, dtype=torch.uint8).to(device).contiguous(), pa)

    def clone(self) -> "CanvasState":
        return CanvasState(self.canvas.clone(), self.lock.clone(), self.step.clone(),
                           self.done.clone(),
                           None if self.prev_argmax is None else self.prev_argmax.clone())


@dataclass
class StepOutputs:
    s: torch.Tensor  # [B, L, d] float32
    sampled: torch.Tensor  # [B, L] int32
    conf: torch.Tensor  # [B, L] float32
    entropy: torch.Tensor  # [B, L] float32
    argmax: torch.Tensor  # [B, L] int32

    @staticmethod
    def empty(B, L, d, device="cuda", pin=False):
        kw = dict(device=device) if not pin else dict(pin_memory=True)
        return StepOutputs(torch.zeros(B, L, d, dtype=torch.float32, **kw),
                           torch.zeros(B, L, dtype=torch.int32, **kw),
                           torch.zeros(B, L, dtype=torch.float32, **kw),
                           torch.zeros(B, L, dtype=torch.float32, **kw),
                           torch.zeros(B, L, dtype=torch.int32, **kw))


@dataclass
class ShardPartial:
    """Partial records of n vocabulary shards, stacked in token order (device tensors):
    rows [n, R, 4] (m, l, entropy, argmax bits), best [n, R, 4] (score, token bits, ln p, 0),
    O [n, R, d] and, with top-k, cand [n, R, k, 2] (y, token bits); R = B L. See
    ds_sampler_step_shard / ds_merge_shards in include/ds_sampler.h."""
    rows: torch.Tensor
    best: torch.Tensor
    O: torch.Tensor
    cand: torch.Tensor | None = None

    @staticmethod
    def empty(n, B, L, d, top_k=0, device="cuda"):
        R = B * L
        return ShardPartial(torch.zeros(n, R, 4, dtype=torch.float32, device=device),
                            torch.zeros(n, R, 4, dtype=torch.float32, device=device),
                            torch.zeros(n, R, d, dtype=torch.float32, device=device),
                            torch.zeros(n, R, top_k, 2, dtype=torch.float32, device=device)
                            if top_k else None)

    @staticmethod
    def stack(parts: list["ShardPartial"]) -> "ShardPartial":
        return ShardPartial(torch.cat([p.rows for p in parts]), torch.cat([p.best for p in parts]),
                            torch.cat([p.O for p in parts]),
                            None if parts[0].cand is None else torch.cat([p.cand for p in parts]))

    def tensors(self) -> list[torch.Tensor]:
        return [t for t in (self.rows, self.best, self.O, self.cand) if t is not None]

    def c_struct(self):
        return C.ds_shard_partial(_ptr(self.rows), _ptr(self.best), _ptr(self.O), _ptr(self.cand))


class Sampler:
    """One sampler (workspace + graphs) on one CUDA device."""

    def __init__(self, vocab: int, d_model: int, *, canvas_len: int = 256, max_batch: int = 1,
                 dtype: str = "bf16", top_k: int = 0, max_steps: int = 48, impl: str = "auto",
                 lock_rule: str = "threshold", entropy_budget: float = 0.1,
                 stop_entropy: float = 0.005, t_schedule: tuple | None = None):
        self.lib = C.load_library()
        if not torch.cuda.is_available():
            raise RuntimeError("the canvas sampler needs a CUDA device")
        self.vocab, self.d, self.L, self.max_batch = int(vocab), int(d_model), int(canvas_len), int(max_batch)
        self.dtype_name = dtype
        self.dtype_code, self.torch_dtype = _DTYPES[dtype]
        self.top_k, self.max_steps = int(top_k), int(max_steps)
        self.lock_rule = lock_rule
        t0, t1 = (0.0, 0.0) if t_schedule is None else (float(t_schedule[0]), float(t_schedule[1]))
        cfg = C.ds_sampler_config(max_batch=self.max_batch, canvas_len=self.L, d_model=self.d,
                                  dtype=self.dtype_code, vocab=self.vocab, top_k=self.top_k,
                                  max_steps=self.max_steps, impl=_IMPLS[impl],
                                  lock_rule=_LOCK_RULES[lock_rule],
                                  entropy_budget=float(entropy_budget),
                                  stop_entropy=float(stop_entropy), t_start=t0, t_end=t1)
        self._cfg = cfg
        handle = c_void_p()
        C.check(self.lib.ds_sampler_create(byref(cfg), byref(handle)), "ds_sampler_create")
        self.handle = handle

    # ---------------------------------------------------------------- properties
    @property
    def impl(self) -> str:
        v = c_int32()
        C.check(self.lib.ds_sampler_impl(self.handle, byref(v)), "ds_sampler_impl")
        return {C.DS_IMPL_TENSOR: "tensor", C.DS_IMPL_SIMT: "simt", C.DS_IMPL_FUSED: "fused"}[v.value]

    @property
    def workspace_bytes(self) -> int:
        v = c_size_t()
        C.check(self.lib.ds_sampler_workspace_bytes(self.handle, byref(v)), "workspace_bytes")
        return v.value

    # ---------------------------------------------------------------- marshalling
    def _step_args(self, H, E, temperature, tau, state: CanvasState, out: StepOutputs, seed: int):
        B = state.canvas.shape[0]
        a = C.ds_step_args()
        a.batch = B
        a.seed = int(seed) & 0xFFFFFFFFFFFFFFFF
        a.H, a.E = _ptr(H), _ptr(E)
        a.temperature, a.tau = _ptr(temperature), _ptr(tau)
        a.step, a.canvas, a.lock, a.done = (_ptr(state.step), _ptr(state.canvas), _ptr(state.lock),
                                            _ptr(state.done))
        a.s, a.sampled, a.conf, a.entropy, a.argmax = (_ptr(out.s), _ptr(out.sampled), _ptr(out.conf),
                                                       _ptr(out.entropy), _ptr(out.argmax))
        a.prev_argmax = _ptr(state.prev_argmax)
        return a

    def _check_tensors(self, H, E, state, out, device_side=True):
        for name, t, dt in (("E", E, self.torch_dtype), ("canvas", state.canvas, torch.int32),
                            ("lock", state.lock, torch.uint8), ("step", state.step, torch.int32),
                            ("done", state.done, torch.uint8), ("s", out.s, torch.float32),
                            ("sampled", out.sampled, torch.int32), ("conf", out.conf, torch.float32),
                            ("entropy", out.entropy, torch.float32),
                            ("argmax", out.argmax, torch.int32)):
            if t.dtype != dt or not t.is_contiguous():
                raise ValueError(f"{name}: expected contiguous {dt}, got {t.dtype}")
        if H is not None and (H.dtype != self.torch_dtype or not H.is_contiguous()):
            raise ValueError(f"H: expected contiguous {self.torch_dtype}")
        if not E.is_cuda:
            raise ValueError("E must be on the device")
        if device_side and not state.canvas.is_cuda:
            raise ValueError("state must be on the device")

    # ---------------------------------------------------------------- entry points
    def step(self, H, E, temperature, tau, state: CanvasState, seed: int,
             out: StepOutputs | None = None, stream=None) -> StepOutputs:
        """Enqueue one step (ds_sampler_step); returns the output tensors."""
        B = state.canvas.shape[0]
        if out is None:
            out = StepOutputs.empty(B, self.L, self.d, device=E.device)
        self._check_tensors(H, E, state, out)
        a = self._step_args(H, E, temperature, tau, state, out, seed)
        C.check(self.lib.ds_sampler_step(self.handle, byref(a), _stream_handle(stream)),
                "ds_sampler_step")
        return out

    def step_host(self, H, E, temperature, tau, state: CanvasState, seed: int,
                  out: StepOutputs, stream=None) -> StepOutputs:
        """ds_sampler_step_host: per-step buffers in (pinned) host memory, E on the device."""
        self._check_tensors(H, E, state, out, device_side=False)
        a = self._step_args(H, E, temperature, tau, state, out, seed)
        C.check(self.lib.ds_sampler_step_host(self.handle, byref(a), _stream_handle(stream)),
                "ds_sampler_step_host")
        return out

    def loop(self, E, temperature, tau, state: CanvasState, seed: int, out: StepOutputs, *,
             H=None, W=None, H_buf=None, max_iters: int | None = None, use_graph: bool = True,
             stream=None) -> StepOutputs:
        """ds_denoise_loop. Fixed H (H given) or the stand-in (W and H_buf given); in stand-in
        mode out.s must hold the previous self-conditioning vector (zeros at the start)."""
        standin = W is not None
        self._check_tensors(H if not standin else H_buf, E, state, out)
        la = C.ds_loop_args()
        la.step = self._step_args(H if not standin else H_buf, E, temperature, tau, state, out, seed)
        la.h_mode = C.DS_H_STANDIN if standin else C.DS_H_FIXED
        la.max_iters = self.max_steps if max_iters is None else int(max_iters)
        la.use_graph = 1 if use_graph else 0
        la.W = _ptr(W)
        la.H_buf = _ptr(H_buf)
        self._keep = (E, temperature, tau, state, out, H, W, H_buf)  # graphs hold these pointers
        C.check(self.lib.ds_denoise_loop(self.handle, byref(la), _stream_handle(stream)),
                "ds_denoise_loop")
        return out

    def block_loop(self, E, temperature, tau, state: CanvasState, seed: int, out: StepOutputs,
                   init_canvas, out_canvas, out_steps, *, first_block: int = 0, H=None, W=None,
                   H_buf=None, max_iters: int | None = None, use_graph: bool = True,
                   stream=None):
        """ds_block_loop: generate init_canvas.shape[0] blocks one after another (each from its
        initial canvas with fresh state), committing each finished canvas to out_canvas
        [n_blocks, B, L] and its step counts to out_steps [n_blocks, B]. state and out are the
        working buffers (their contents on entry are replaced)."""
        standin = W is not None
        self._check_tensors(H if not standin else H_buf, E, state, out)
        n_blocks = int(init_canvas.shape[0])
        B, L = state.canvas.shape
        for t, shape in ((init_canvas, (n_blocks, B, L)), (out_canvas, (n_blocks, B, L)),
                         (out_steps, (n_blocks, B))):
            if tuple(t.shape) != shape or t.dtype != torch.int32 or not t.is_cuda:
                raise ValueError(f"block buffers must be int32 CUDA tensors of shape {shape}")
        ba = C.ds_block_args()
        ba.loop.step = self._step_args(H if not standin else H_buf, E, temperature, tau, state, out,
                                       seed)
        ba.loop.h_mode = C.DS_H_STANDIN if standin else C.DS_H_FIXED
        ba.loop.max_iters = self.max_steps if max_iters is None else int(max_iters)
        ba.loop.use_graph = 1 if use_graph else 0
        ba.loop.W = _ptr(W)
        ba.loop.H_buf = _ptr(H_buf)
        ba.n_blocks = n_blocks
        ba.first_block = int(first_block)
        ba.init_canvas = _ptr(init_canvas)
        ba.out_canvas = _ptr(out_canvas)
        ba.out_steps = _ptr(out_steps)
        # graphs hold these pointers
        self._keep = (E, temperature, tau, state, out, H, W, H_buf, init_canvas, out_canvas,
                      out_steps)
        C.check(self.lib.ds_block_loop(self.handle, byref(ba), _stream_handle(stream)),
                "ds_block_loop")
        return out_canvas, out_steps

    def step_shard(self, H, E_shard, temperature, tau, state: CanvasState, seed: int,
                   token_offset: int, vocab_total: int, out: ShardPartial | None = None,
                   stream=None) -> ShardPartial:
        """The partial record of one vocabulary shard (E_shard = rows token_offset ..
        token_offset + vocab of the full table); state is read (step, done), not updated."""
        B = state.canvas.shape[0]
        out = ShardPartial.empty(1, B, self.L, self.d, self.top_k) if out is None else out
        dummy = StepOutputs.empty(B, self.L, self.d) if not hasattr(self, "_shard_dummy") or \
            self._shard_dummy.s.shape[0] != B else self._shard_dummy
        self._shard_dummy = dummy
        a = self._step_args(H, E_shard, temperature, tau, state, dummy, seed)
        part = out.c_struct()
        C.check(self.lib.ds_sampler_step_shard(self.handle, byref(a), int(token_offset),
                                               int(vocab_total), byref(part),
                                               _stream_handle(stream)), "ds_sampler_step_shard")
        return out

    def merge_shards(self, parts: ShardPartial, temperature, tau, state: CanvasState, seed: int,
                     vocab_total: int, out: StepOutputs | None = None, stream=None,
                     E=None) -> StepOutputs:
        """Merge n shards' records (token order) into the step's outputs and update state."""
        B = state.canvas.shape[0]
        out = StepOutputs.empty(B, self.L, self.d) if out is None else out
        n = parts.rows.shape[0]
        a = self._step_args(None, None, temperature, tau, state, out, seed)  # merge reads no H, E
        part = parts.c_struct()
        C.check(self.lib.ds_merge_shards(self.handle, byref(a), int(n), byref(part),
                                         int(vocab_total), _stream_handle(stream)),
                "ds_merge_shards")
        return out

    def standin_hidden(self, W, s_prev, E, canvas, done, H_out, stream=None):
        B = canvas.shape[0]
        C.check(self.lib.ds_standin_hidden(self.handle, _ptr(W), _ptr(s_prev), _ptr(E), _ptr(canvas),
                                           _ptr(done), _ptr(H_out), B, _stream_handle(stream)),
                "ds_standin_hidden")
        return H_out

    def set_phase_timing(self, enable: bool, coarse: bool = False) -> None:
        """Per-phase CUDA-event timing of each step (coarse: only the ends of the logits,
        up-to-self-conditioning, self-conditioning and final phases are marked)."""
        level = 0 if not enable else (2 if coarse else 1)
        C.check(self.lib.ds_sampler_set_phase_timing(self.handle, level), "set_phase_timing")

    def phase_times(self) -> tuple[dict, int]:
        """Accumulated milliseconds per phase since timing was enabled, and the step count."""
        import ctypes
        ms = (ctypes.c_float * len(C.PHASES))()
        steps = c_int32()
        C.check(self.lib.ds_sampler_phase_times(self.handle, ms, len(C.PHASES), byref(steps)),
                "phase_times")
        return dict(zip(C.PHASES, [float(x) for x in ms])), steps.value

    @property
    def launch_count(self) -> int:
        import ctypes
        v = ctypes.c_int64()
        C.check(self.lib.ds_sampler_launch_count(self.handle, byref(v)), "launch_count")
        return v.value

    def device_status(self) -> int:
        v = c_int32()
        C.check(self.lib.ds_sampler_device_status(self.handle, byref(v)), "device_status")
        return v.value

    def debug_buffer(self, which: int):
        p, n = c_void_p(), c_size_t()
        C.check(self.lib.ds_sampler_debug_buffer(self.handle, which, byref(p), byref(n)),
                "debug_buffer")
        return p.value, n.value

    def debug_tensor(self, which: int) -> torch.Tensor:
        """Device copy (uint8) of an internal buffer of the last step (0: y, 1: row stats,
        2/3: bf16 hi/lo of exp(y - m))."""
        ptr, nbytes = self.debug_buffer(which)

        class _View:
            __cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                        "data": (ptr, False), "version": 3}

        return torch.as_tensor(_View(), device="cuda").clone()

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.ds_sampler_destroy(self.handle)
            self.handle = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def philox4x32_10(ctr: torch.Tensor, seed: int, stream=None) -> torch.Tensor:
    """Philox4x32-10 blocks of uint32 counters ctr [n, 4] (device, int32 storage)."""
    lib = C.load_library()
    out = torch.empty_like(ctr)
    C.check(lib.ds_philox4x32_10(_ptr(ctr), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out), ctr.shape[0],
                                 _stream_handle(stream)), "ds_philox4x32_10")
    return out
