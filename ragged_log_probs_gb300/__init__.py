"""Ragged batched log-probabilities on GB300: thin Python binding of the C ABI.

Argument marshalling only. Every step of the path (output offsets, the streaming
max / sum-exp / top-k reduction, the split-row merge, the target gather) runs in
the CUDA kernels of ``liblp_ragged.so``; there is no CPU or library fallback, and
importing this package fails loudly when the library has not been built.

Integer tensors may be ``torch.int32`` or ``torch.uint32`` (same bits); echo flags
``torch.uint8`` or ``torch.bool``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build
from .results import LogProbabilities, assemble  # noqa: F401  (host-side result assembly)

__all__ = [
    "LpError", "lib_path", "load", "workspace_size", "new_workspace", "plan", "compute", "row_kernel",
    "compute_ex", "step", "read_status", "ragged_log_probs", "tuple_bytes", "shard_partials", "shard_merge",
    "gather_shard_tuples", "ragged_log_probs_vocab_parallel", "out_per_token", "STATUS_NAMES", "LogProbabilities", "assemble",
]

LP_MAX_LEVELS = 6
PAD_TOKEN = 0xFFFFFFFF
STATUS_NAMES = {
    0: "LP_OK", 1: "LP_ERR_NULL", 2: "LP_ERR_LEVELS", 3: "LP_ERR_SHAPE", 4: "LP_ERR_OFFSETS",
    5: "LP_ERR_TOKEN_RANGE", 6: "LP_ERR_WORKSPACE", 7: "LP_ERR_CUDA", 8: "LP_ERR_TEMPERATURE",
}
EXPORTS = ("lp_ragged_workspace_size", "lp_ragged_plan", "lp_ragged_compute", "lp_ragged_compute_ex",
           "lp_ragged_step", "lp_ragged_tuple_bytes", "lp_ragged_shard_partials", "lp_ragged_shard_merge",
           "lp_ragged_read_status", "lp_ragged_strerror")


class LpError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({_strerror(code)})")


_LIB: Optional[ctypes.CDLL] = None


def lib_path() -> str:
    return _build.lib_path()


def load() -> ctypes.CDLL:
    """Load ``liblp_ragged.so`` (built by ``__graft_entry__.build()``); raise if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run __graft_entry__.build() (nvcc, sm_103a) first")
    lib = ctypes.CDLL(path)
    u32, vp, sz = ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t
    lib.lp_ragged_workspace_size.argtypes = [u32, u32, u32, u32]
    lib.lp_ragged_workspace_size.restype = sz
    lib.lp_ragged_plan.argtypes = [vp, vp, u32, u32, vp, vp, vp, sz, vp]
    lib.lp_ragged_plan.restype = ctypes.c_int
    lib.lp_ragged_compute.argtypes = [vp, u32, u32, vp, u32, vp, vp, vp, vp, u32, vp, vp, vp, sz, vp]
    lib.lp_ragged_compute.restype = ctypes.c_int
    lib.lp_ragged_compute_ex.argtypes = [vp, u32, u32, vp, vp, u32, u32, vp, vp, vp, vp, vp, u32, vp, vp, vp, sz, vp]
    lib.lp_ragged_compute_ex.restype = ctypes.c_int
    lib.lp_ragged_step.argtypes = [vp, u32, u32, vp, vp, u32, u32, vp, vp, vp, vp, u32, vp, vp, vp, vp, u32, vp, sz,
                                   vp]
    lib.lp_ragged_step.restype = ctypes.c_int
    lib.lp_ragged_tuple_bytes.argtypes = [u32]
    lib.lp_ragged_tuple_bytes.restype = u32
    lib.lp_ragged_shard_partials.argtypes = [vp, u32, u32, u32, vp, vp, u32, u32, vp, vp, vp, vp, vp, u32, vp, u32,
                                             vp, sz, vp]
    lib.lp_ragged_shard_partials.restype = ctypes.c_int
    lib.lp_ragged_shard_merge.argtypes = [vp, u32, u32, u32, vp, u32, vp, u32, vp, vp, vp, sz, vp]
    lib.lp_ragged_shard_merge.restype = ctypes.c_int
    lib.lp_ragged_read_status.argtypes = [vp, vp, vp]
    lib.lp_ragged_read_status.restype = ctypes.c_int
    lib.lp_ragged_row_kernel.argtypes = [u32, u32, u32, u32, vp]
    lib.lp_ragged_row_kernel.restype = ctypes.c_int
    lib.lp_ragged_strerror.argtypes = [ctypes.c_int]
    lib.lp_ragged_strerror.restype = ctypes.c_char_p
    _LIB = lib
    return lib


def _strerror(code: int) -> str:
    try:
        return load().lp_ragged_strerror(code).decode()
    except Exception:  # pragma: no cover
        return "?"


def out_per_token(levels: int) -> int:
    return 2 ** levels if levels > 0 else 1


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _on_current_device(t: torch.Tensor, name: str) -> None:
    # The library launches on the current device: another GPU's pointer would reach the kernel.
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{cur}")


def _dev_u32(t: torch.Tensor, name: str, n: Optional[int] = None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    _on_current_device(t, name)
    if t.dtype not in (torch.int32, torch.uint32):
        raise TypeError(f"{name} must be int32/uint32, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.numel() < n:
        raise ValueError(f"{name} needs {n} elements, has {t.numel()}")
    return t.data_ptr()


def _dev_u8(t: torch.Tensor, name: str, n: int) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    _on_current_device(t, name)
    if t.dtype not in (torch.uint8, torch.bool, torch.int8):
        raise TypeError(f"{name} must be uint8/bool, got {t.dtype}")
    if not t.is_contiguous() or t.numel() < n:
        raise ValueError(f"{name} must be contiguous with {n} elements")
    return t.data_ptr()


def _dev_f32(t: torch.Tensor, name: str, n: Optional[int] = None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    _on_current_device(t, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.numel() < n:
        raise ValueError(f"{name} needs {n} elements, has {t.numel()}")
    return t.data_ptr()


def _ws(workspace: torch.Tensor) -> int:
    """Device pointer of a workspace tensor (the kernels write it: a host tensor is refused)."""
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor (see new_workspace)")
    _on_current_device(workspace, "workspace")
    return workspace.data_ptr()


def workspace_size(B: int, T: int, V: int, levels: int) -> int:
    """Bytes of scratch for one call on the current device."""
    return int(load().lp_ragged_workspace_size(B, T, V, levels))


def new_workspace(B: int, T: int, V: int, levels: int, device=None) -> torch.Tensor:
    """Allocate a workspace tensor (uint8) on ``device`` (torch allocates; the library never does)."""
    device = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(device):
        n = workspace_size(B, T, V, levels)
        if n == 0:
            raise LpError(2 if levels > LP_MAX_LEVELS else 7, "lp_ragged_workspace_size")
        return torch.zeros(n, dtype=torch.uint8, device=device)


def plan(logit_row_offsets: torch.Tensor, echo: torch.Tensor, T: int, workspace: torch.Tensor,
         output_row_offsets: Optional[torch.Tensor] = None, host_out: Optional[torch.Tensor] = None,
         stream=None) -> torch.Tensor:
    """Enqueue ``lp_ragged_plan``; returns ``output_row_offsets`` (device, B+1).

    ``host_out`` (optional, 2 x int32 on the host, pinned for an async copy) receives
    ``{R, status bits}`` once the stream has reached this point."""
    lib = load()
    B = logit_row_offsets.numel() - 1
    if output_row_offsets is None:
        output_row_offsets = torch.empty(B + 1, dtype=logit_row_offsets.dtype, device=logit_row_offsets.device)
    hp = None
    if host_out is not None:
        if host_out.is_cuda or host_out.numel() < 2 or host_out.element_size() != 4 or not host_out.is_contiguous():
            raise ValueError("host_out must be a contiguous 2-word host tensor")
        hp = host_out.data_ptr()
    rc = lib.lp_ragged_plan(_dev_u32(logit_row_offsets, "logit_row_offsets", B + 1), _dev_u8(echo, "echo", B),
                            B, T, _dev_u32(output_row_offsets, "output_row_offsets", B + 1), hp,
                            _ws(workspace), workspace.numel() * workspace.element_size(),
                            _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_plan")
    return output_row_offsets


def compute(logits: torch.Tensor, logit_row_offsets: torch.Tensor, tokens: torch.Tensor,
            sampled_tokens: torch.Tensor, output_row_offsets: torch.Tensor, echo: torch.Tensor, levels: int,
            out_logprobs: torch.Tensor, out_tokens: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Enqueue ``lp_ragged_compute`` (outputs must hold R x W entries, R = output_row_offsets[B])."""
    lib = load()
    if logits.dim() != 2 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise TypeError("logits must be a 2-D float32 CUDA tensor")
    if logits.stride(1) != 1 or logits.stride(0) != logits.shape[1]:
        raise ValueError("logits must be row-major contiguous")
    T, V = logits.shape
    B = logit_row_offsets.numel() - 1
    if out_logprobs.dtype != torch.float32 or not out_logprobs.is_cuda or not out_logprobs.is_contiguous():
        raise TypeError("out_logprobs must be a contiguous float32 CUDA tensor")
    rc = lib.lp_ragged_compute(
        logits.data_ptr(), T, V, _dev_u32(logit_row_offsets, "logit_row_offsets", B + 1), B,
        _dev_u32(tokens, "tokens", T), _dev_u32(sampled_tokens, "sampled_tokens", B),
        _dev_u32(output_row_offsets, "output_row_offsets", B + 1), _dev_u8(echo, "echo", B), levels,
        out_logprobs.data_ptr(), _dev_u32(out_tokens, "out_tokens"),
        _ws(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_compute")


def compute_ex(logits: torch.Tensor, logit_row_offsets: torch.Tensor, tokens: torch.Tensor,
               sampled_tokens: torch.Tensor, output_row_offsets: torch.Tensor, echo: torch.Tensor, levels: int,
               out_logprobs: torch.Tensor, out_tokens: torch.Tensor, workspace: torch.Tensor,
               input_row_offsets: Optional[torch.Tensor] = None, temperatures: Optional[torch.Tensor] = None,
               stream=None) -> None:
    """Enqueue ``lp_ragged_compute_ex``: VARIABLE logits (``input_row_offsets`` gives the
    positions, ``logit_row_offsets`` the rows present in ``logits``, each batch's last
    positions) and/or per-batch ``temperatures`` (float32 [B])."""
    lib = load()
    if logits.dim() != 2 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise TypeError("logits must be a 2-D float32 CUDA tensor")
    if logits.stride(1) != 1 or logits.stride(0) != logits.shape[1]:
        raise ValueError("logits must be row-major contiguous")
    T_logits, V = logits.shape
    B = logit_row_offsets.numel() - 1
    T = tokens.numel()
    ioff = 0
    if input_row_offsets is not None:
        ioff = _dev_u32(input_row_offsets, "input_row_offsets", B + 1)
    elif T != T_logits:
        raise ValueError("without input_row_offsets every position needs a logits row (tokens and logits rows)")
    tp = 0
    if temperatures is not None:
        if temperatures.dtype != torch.float32 or not temperatures.is_cuda or not temperatures.is_contiguous() \
                or temperatures.numel() < B:
            raise TypeError("temperatures must be a contiguous float32 CUDA tensor with B entries")
        tp = temperatures.data_ptr()
    if out_logprobs.dtype != torch.float32 or not out_logprobs.is_cuda or not out_logprobs.is_contiguous():
        raise TypeError("out_logprobs must be a contiguous float32 CUDA tensor")
    rc = lib.lp_ragged_compute_ex(
        logits.data_ptr(), T_logits, V, _dev_u32(logit_row_offsets, "logit_row_offsets", B + 1), ioff, T, B,
        _dev_u32(tokens, "tokens", T), _dev_u32(sampled_tokens, "sampled_tokens", B),
        _dev_u32(output_row_offsets, "output_row_offsets", B + 1), _dev_u8(echo, "echo", B), tp, levels,
        out_logprobs.data_ptr(), _dev_u32(out_tokens, "out_tokens"),
        _ws(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_compute_ex")


def step(logits: torch.Tensor, logit_row_offsets: torch.Tensor, tokens: torch.Tensor, sampled_tokens: torch.Tensor,
         echo: torch.Tensor, levels: int, output_row_offsets: torch.Tensor, out_logprobs: torch.Tensor,
         out_tokens: torch.Tensor, workspace: torch.Tensor, input_row_offsets: Optional[torch.Tensor] = None,
         temperatures: Optional[torch.Tensor] = None, host_out: Optional[torch.Tensor] = None, stream=None) -> None:
    """Enqueue ``lp_ragged_step``: plan and reduction in one call, the reduction streaming
    while the plan runs. ``out_logprobs`` / ``out_tokens`` are [rows, W] with rows >= R
    (R <= T); ``host_out`` (pinned int32 [2]) receives {R, status of plan and reduction}."""
    lib = load()
    if logits.dim() != 2 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise TypeError("logits must be a 2-D float32 CUDA tensor")
    if logits.stride(1) != 1 or logits.stride(0) != logits.shape[1]:
        raise ValueError("logits must be row-major contiguous")
    T_logits, V = logits.shape
    B = logit_row_offsets.numel() - 1
    T = tokens.numel()
    ioff = 0
    if input_row_offsets is not None:
        ioff = _dev_u32(input_row_offsets, "input_row_offsets", B + 1)
    elif T != T_logits:
        raise ValueError("without input_row_offsets every position needs a logits row (tokens and logits rows)")
    tp = 0
    if temperatures is not None:
        if temperatures.dtype != torch.float32 or not temperatures.is_cuda or not temperatures.is_contiguous() \
                or temperatures.numel() < B:
            raise TypeError("temperatures must be a contiguous float32 CUDA tensor with B entries")
        tp = temperatures.data_ptr()
    W = out_per_token(levels)
    if out_logprobs.dtype != torch.float32 or not out_logprobs.is_cuda or not out_logprobs.is_contiguous() \
            or out_logprobs.dim() != 2 or out_logprobs.shape[1] != W:
        raise TypeError(f"out_logprobs must be a contiguous float32 CUDA tensor [rows, {W}]")
    rows = out_logprobs.shape[0]
    if out_tokens.shape != out_logprobs.shape:
        raise ValueError("out_tokens must have the shape of out_logprobs")
    hp = 0
    if host_out is not None:
        if host_out.dtype != torch.int32 or host_out.numel() < 2 or host_out.is_cuda or not host_out.is_pinned():
            raise TypeError("host_out must be a pinned int32 CPU tensor with 2 elements")
        hp = host_out.data_ptr()
    rc = lib.lp_ragged_step(
        logits.data_ptr(), T_logits, V, _dev_u32(logit_row_offsets, "logit_row_offsets", B + 1), ioff, T, B,
        _dev_u32(tokens, "tokens", T), _dev_u32(sampled_tokens, "sampled_tokens", B), _dev_u8(echo, "echo", B), tp,
        levels, _dev_u32(output_row_offsets, "output_row_offsets", B + 1), hp, out_logprobs.data_ptr(),
        _dev_u32(out_tokens, "out_tokens"), rows, _ws(workspace),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_step")


def tuple_bytes(levels: int) -> int:
    """Bytes of one row tuple of the vocab-parallel form (a multiple of 16)."""
    n = int(load().lp_ragged_tuple_bytes(levels))
    if n == 0:
        raise LpError(2, "lp_ragged_tuple_bytes")
    return n


def shard_partials(logits: torch.Tensor, vocab_base: int, logit_row_offsets: torch.Tensor, tokens: torch.Tensor,
                   sampled_tokens: torch.Tensor, output_row_offsets: torch.Tensor, echo: torch.Tensor, levels: int,
                   tuples: torch.Tensor, rows_capacity: int, workspace: torch.Tensor,
                   input_row_offsets: Optional[torch.Tensor] = None, temperatures: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Enqueue ``lp_ragged_shard_partials``: this rank's vocab columns
    ``[vocab_base, vocab_base + logits.shape[1])`` -> one row tuple per output row in
    ``tuples`` (uint8 CUDA tensor of at least ``rows_capacity * tuple_bytes(levels)``)."""
    lib = load()
    if logits.dim() != 2 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise TypeError("logits must be a 2-D float32 CUDA tensor")
    if logits.stride(1) != 1 or logits.stride(0) != logits.shape[1]:
        raise ValueError("logits must be row-major contiguous")
    T_logits, V_shard = logits.shape
    B = logit_row_offsets.numel() - 1
    T = tokens.numel()
    if input_row_offsets is None and T != T_logits:
        raise ValueError("without input_row_offsets every position needs a logits row")
    if not tuples.is_cuda or not tuples.is_contiguous() or \
            tuples.numel() * tuples.element_size() < rows_capacity * tuple_bytes(levels):
        raise ValueError("tuples must be a contiguous CUDA buffer of rows_capacity * tuple_bytes(levels) bytes")
    ioff = 0 if input_row_offsets is None else _dev_u32(input_row_offsets, "input_row_offsets", B + 1)
    tp = 0 if temperatures is None else _dev_f32(temperatures, "temperatures", B)
    rc = lib.lp_ragged_shard_partials(
        logits.data_ptr(), T_logits, V_shard, vocab_base, _dev_u32(logit_row_offsets, "logit_row_offsets", B + 1),
        ioff, T, B, _dev_u32(tokens, "tokens", T), _dev_u32(sampled_tokens, "sampled_tokens", B),
        _dev_u32(output_row_offsets, "output_row_offsets", B + 1), _dev_u8(echo, "echo", B), tp, levels,
        tuples.data_ptr(), rows_capacity, _ws(workspace), workspace.numel() * workspace.element_size(),
        _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_shard_partials")


def shard_merge(tuples: torch.Tensor, P: int, rows_capacity: int, V: int, output_row_offsets: torch.Tensor,
                levels: int, out_logprobs: torch.Tensor, out_tokens: torch.Tensor, workspace: torch.Tensor,
                temperatures: Optional[torch.Tensor] = None, stream=None) -> None:
    """Enqueue ``lp_ragged_shard_merge`` over ``tuples`` = [P][rows_capacity][stride] bytes."""
    lib = load()
    B = output_row_offsets.numel() - 1
    if not tuples.is_cuda or not tuples.is_contiguous() or \
            tuples.numel() * tuples.element_size() < P * rows_capacity * tuple_bytes(levels):
        raise ValueError("tuples must hold P * rows_capacity row tuples")
    tp = 0 if temperatures is None else _dev_f32(temperatures, "temperatures", B)
    rc = lib.lp_ragged_shard_merge(tuples.data_ptr(), P, rows_capacity, V,
                                   _dev_u32(output_row_offsets, "output_row_offsets", B + 1), B, tp, levels,
                                   _dev_f32(out_logprobs, "out_logprobs"), _dev_u32(out_tokens, "out_tokens"),
                                   _ws(workspace), workspace.numel() * workspace.element_size(),
                                   _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_shard_merge")


def gather_shard_tuples(local: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange step of the vocab-parallel form: every rank's tuple buffer (same
    size on all ranks), concatenated in rank order = shard order, on every rank."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(local.shape), dtype=local.dtype, device=local.device)
    if local.is_cuda:
        dist.all_gather_into_tensor(out, local.contiguous(), group=group)
    else:  # gloo has no all_gather_into_tensor
        dist.all_gather(list(out.unbind(0)), local.contiguous(), group=group)
    return out


def ragged_log_probs_vocab_parallel(logits_shard: torch.Tensor, vocab_base: int, vocab_size: int,
                                    logit_row_offsets: torch.Tensor, tokens: torch.Tensor,
                                    sampled_tokens: torch.Tensor, echo: torch.Tensor, levels: int, group=None,
                                    input_row_offsets: Optional[torch.Tensor] = None,
                                    temperatures: Optional[torch.Tensor] = None, check: bool = True):
    """One rank of the vocab-parallel form: plan -> shard partials -> all-gather of the
    tuples (torch.distributed) -> merge. Ranks hold contiguous column ranges in rank
    order covering [0, vocab_size). Returns the same triple as ``ragged_log_probs``."""
    T_logits, V_shard = logits_shard.shape
    B = logit_row_offsets.numel() - 1
    T = tokens.numel() if input_row_offsets is not None else T_logits
    pos_off = input_row_offsets if input_row_offsets is not None else logit_row_offsets
    dev = logits_shard.device
    workspace = new_workspace(B, T, V_shard, levels, dev)
    host = torch.zeros(2, dtype=torch.int32).pin_memory()
    out_off = plan(pos_off, echo, T, workspace, host_out=host)
    torch.cuda.current_stream().synchronize()
    R, status = int(host[0]), int(host[1]) & 0xFFFFFFFF
    if status:
        raise LpError(_first_bit(status), "lp_ragged_plan (device)")
    stride = tuple_bytes(levels)
    local = torch.empty(max(R, 1) * stride, dtype=torch.uint8, device=dev)
    shard_partials(logits_shard, vocab_base, logit_row_offsets, tokens, sampled_tokens, out_off, echo, levels, local,
                   max(R, 1), workspace, input_row_offsets=input_row_offsets, temperatures=temperatures)
    gathered = gather_shard_tuples(local, group)
    W = out_per_token(levels)
    out_lp = torch.empty((R, W), dtype=torch.float32, device=dev)
    out_tok = torch.empty((R, W), dtype=torch.int32, device=dev)
    shard_merge(gathered, gathered.shape[0], max(R, 1), vocab_size, out_off, levels, out_lp, out_tok, workspace,
                temperatures=temperatures)
    if check:
        status = read_status(workspace)
        if status:
            raise LpError(_first_bit(status), "vocab-parallel ragged log-probabilities (device)")
    return out_off, out_lp, out_tok


def row_kernel(T_logits: int, T: int, V: int, levels: int) -> str:
    """The row kernel the library launches for this shape on the current device:
    ``"queue"`` (row queue) or ``"warp"`` (warp-owned ranges)."""
    kind = ctypes.c_int(-1)
    rc = load().lp_ragged_row_kernel(T_logits, T, V, levels, ctypes.addressof(kind))
    if rc:
        raise LpError(rc, "lp_ragged_row_kernel")
    return "queue" if kind.value == 1 else "warp"


def read_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronously read the device status bits (bit c set <=> error code c seen)."""
    lib = load()
    wp = _ws(workspace)
    host = torch.zeros(1, dtype=torch.int32).pin_memory()
    rc = lib.lp_ragged_read_status(wp, host.data_ptr(), _stream_handle(stream))
    if rc:
        raise LpError(rc, "lp_ragged_read_status")
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    return int(host.item()) & 0xFFFFFFFF


def ragged_log_probs(logits: torch.Tensor, logit_row_offsets: torch.Tensor, tokens: torch.Tensor,
                     sampled_tokens: torch.Tensor, echo: torch.Tensor, levels: int,
                     workspace: Optional[torch.Tensor] = None, stream=None, check: bool = True,
                     input_row_offsets: Optional[torch.Tensor] = None,
                     temperatures: Optional[torch.Tensor] = None):
    """plan -> size outputs (one host sync for R) -> compute.

    With ``input_row_offsets`` (VARIABLE logits) and/or ``temperatures`` the compute
    step is ``lp_ragged_compute_ex``.
    Returns ``(output_row_offsets [B+1], logprobs f32 [R, W], token_ids int32-storage-of-uint32 [R, W])``."""
    T_logits, V = logits.shape
    B = logit_row_offsets.numel() - 1
    extended = input_row_offsets is not None or temperatures is not None
    T = tokens.numel() if input_row_offsets is not None else T_logits
    pos_off = input_row_offsets if input_row_offsets is not None else logit_row_offsets
    if workspace is None:
        workspace = new_workspace(B, T, V, levels, logits.device)
    host = torch.zeros(2, dtype=torch.int32).pin_memory()
    out_off = plan(pos_off, echo, T, workspace, host_out=host, stream=stream)
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    R, status = int(host[0]), int(host[1]) & 0xFFFFFFFF
    if status:
        raise LpError(_first_bit(status), "lp_ragged_plan (device)")
    W = out_per_token(levels)
    out_lp = torch.empty((R, W), dtype=torch.float32, device=logits.device)
    out_tok = torch.empty((R, W), dtype=torch.int32, device=logits.device)
    if extended:
        compute_ex(logits, logit_row_offsets, tokens, sampled_tokens, out_off, echo, levels, out_lp, out_tok,
                   workspace, input_row_offsets=input_row_offsets, temperatures=temperatures, stream=stream)
    else:
        compute(logits, logit_row_offsets, tokens, sampled_tokens, out_off, echo, levels, out_lp, out_tok,
                workspace, stream=stream)
    if check:
        status = read_status(workspace, stream)
        if status:
            raise LpError(_first_bit(status), "lp_ragged_compute (device)")
    return out_off, out_lp, out_tok


def _first_bit(bits: int) -> int:
    for c in range(1, 32):
        if bits & (1 << c):
            return c
    return 0
