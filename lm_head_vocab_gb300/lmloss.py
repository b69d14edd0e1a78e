"""PyTorch-facing wrapper of the lmloss C ABI.

Tensors only supply device pointers and the current CUDA stream; every step
of the loss runs in the library's kernels.  The library must be built and a
CUDA device present: there is no CPU path.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Union

import ctypes

import torch

from . import _lib
from ._lib import LMLossError

_DT = {torch.bfloat16: _lib.LMLOSS_BF16, torch.float32: _lib.LMLOSS_FP32}
_RED = {"sum": _lib.LMLOSS_REDUCE_SUM, "token_mean": _lib.LMLOSS_REDUCE_TOKEN_MEAN}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, numel: Optional[int], device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {t.numel()}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, logits on {device}")


@dataclass
class Outputs:
    loss: torch.Tensor                      # [5] float32: total, ce, z, kl, gspo
    grad: Optional[torch.Tensor] = None
    logp: Optional[torch.Tensor] = None
    lse: Optional[torch.Tensor] = None
    kl: Optional[torch.Tensor] = None
    count: Optional[torch.Tensor] = None    # [2] int64: active rows, non-empty segments
    seg_count: Optional[torch.Tensor] = None
    seg_ratio: Optional[torch.Tensor] = None
    seg_flag: Optional[torch.Tensor] = None
    seg_loss: Optional[torch.Tensor] = None
    entropy: Optional[torch.Tensor] = None


class LMLoss:
    """One library handle (workspace for up to max_T rows / max_segments segments)."""

    def __init__(self, device: Union[int, torch.device, None] = None, max_T: int = 1 << 17,
                 max_segments: int = 1 << 14):
        if not torch.cuda.is_available():
            raise RuntimeError("lmloss needs a CUDA device")
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index or 0) \
            if not isinstance(device, int) else torch.device("cuda", device)
        self.device = dev
        self.max_T = int(max_T)
        self.max_segments = int(max_segments)
        self.handle = _lib.lmloss_create(dev.index, self.max_T, self.max_segments)

    def close(self):
        if getattr(self, "handle", None) is not None:
            _lib.lmloss_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------- tuning
    def set_launch_config(self, cluster: int = 0, threads: int = 0, nbuf: int = 0):
        st = _lib.lmloss_set_launch_config(self.handle, cluster, threads, nbuf)
        if st != _lib.LMLOSS_OK:
            raise LMLossError(st, "lmloss_set_launch_config")

    def set_timing(self, enable: bool):
        _lib.lmloss_set_timing(self.handle, enable)

    def kernel_time(self):
        """(summed main-kernel ms, calls) recorded since set_timing(True)."""
        return _lib.lmloss_get_timing(self.handle)

    def call_info(self) -> dict:
        return _lib.lmloss_get_call_info(self.handle)

    def device_error(self) -> int:
        return _lib.lmloss_get_device_error(self.handle)

    # --------------------------------------------------------------- call
    def build_args(self, logits: torch.Tensor, targets: torch.Tensor, loss_mask=None, *,
                   ce_weight: float = 1.0, z_alpha: float = 0.0, teacher_logits=None,
                   kl_weight: float = 0.0, temperature: float = 1.0, segment_ids=None,
                   num_segments: Optional[int] = None, advantages=None, old_logprobs=None,
                   clip_eps_low: float = 0.0, clip_eps_high: float = 0.0, token_advantages=None,
                   reduction: str = "token_mean", denominator: float = 1.0,
                   grad: Union[None, str, torch.Tensor] = "new", V: Optional[int] = None,
                   want=("logp", "lse")):
        """Allocate outputs and fill the C argument struct.  Returns (args, Outputs, keepalive)."""
        if logits.dim() != 2 or logits.stride(1) != 1:
            raise ValueError("logits must be [T, V] with unit column stride")
        if logits.dtype not in _DT:
            raise TypeError("logits must be bfloat16 or float32")
        dev = logits.device
        T = logits.shape[0]
        V = logits.shape[1] if V is None else int(V)
        ld = logits.stride(0) if T > 1 else max(logits.shape[1], V)
        _need(targets, "targets", torch.int64, T, dev)
        if loss_mask is not None:
            _need(loss_mask, "loss_mask", torch.uint8, T, dev)
        if teacher_logits is not None:
            if teacher_logits.dtype != logits.dtype or teacher_logits.shape != logits.shape \
                    or teacher_logits.stride() != logits.stride():
                raise ValueError("teacher_logits must match logits in dtype, shape and strides")
        out = Outputs(loss=torch.empty(5, dtype=torch.float32, device=dev))
        if isinstance(grad, torch.Tensor):
            if grad.dtype != logits.dtype or grad.shape != logits.shape or grad.stride() != logits.stride():
                raise ValueError("grad must match logits in dtype, shape and strides")
            out.grad = grad
        elif grad == "inplace":
            out.grad = logits
        elif grad == "new":
            out.grad = torch.empty_strided(logits.shape, logits.stride(), dtype=logits.dtype, device=dev)
        elif grad is not None:
            raise ValueError("grad must be None, 'new', 'inplace' or a tensor")
        S = 0
        if segment_ids is not None:
            _need(segment_ids, "segment_ids", torch.int32, T, dev)
            S = int(num_segments) if num_segments is not None else int(advantages.numel())
            _need(advantages, "advantages", torch.float32, S, dev)
            _need(old_logprobs, "old_logprobs", torch.float32, T, dev)
        if token_advantages is not None:
            _need(token_advantages, "token_advantages", torch.float32, T, dev)
            _need(old_logprobs, "old_logprobs", torch.float32, T, dev)
        f32 = dict(dtype=torch.float32, device=dev)
        if "entropy" in want:
            out.entropy = torch.empty(T, **f32)
        if "logp" in want:
            out.logp = torch.empty(T, **f32)
        if "lse" in want:
            out.lse = torch.empty(T, **f32)
        if "kl" in want and teacher_logits is not None:
            out.kl = torch.empty(T, **f32)
        if "count" in want:
            out.count = torch.empty(2, dtype=torch.int64, device=dev)
        if segment_ids is not None and "seg" in want:
            out.seg_count = torch.empty(S, dtype=torch.int32, device=dev)
            out.seg_ratio = torch.empty(S, **f32)
            out.seg_flag = torch.empty(S, dtype=torch.uint8, device=dev)
            out.seg_loss = torch.empty(S, **f32)

        a = _lib.lmloss_args()
        a.logits = _ptr(logits)
        a.T, a.V, a.ld = T, V, ld
        a.dtype = _DT[logits.dtype]
        a.reduction = _RED[reduction]
        a.targets = _ptr(targets)
        a.loss_mask = _ptr(loss_mask)
        a.ce_weight = float(ce_weight)
        a.z_alpha = float(z_alpha)
        a.teacher_logits = _ptr(teacher_logits)
        a.kl_weight = float(kl_weight)
        a.temperature = float(temperature)
        a.segment_ids = _ptr(segment_ids)
        a.num_segments = S
        a.advantages = _ptr(advantages)
        a.old_logprobs = _ptr(old_logprobs)
        a.clip_eps_low = float(clip_eps_low)
        a.clip_eps_high = float(clip_eps_high)
        a.denominator = float(denominator)
        a.grad_out = _ptr(out.grad)
        a.loss_out = _ptr(out.loss)
        a.logp_out = _ptr(out.logp)
        a.lse_out = _ptr(out.lse)
        a.kl_out = _ptr(out.kl)
        a.count_out = _ptr(out.count)
        a.seg_count_out = _ptr(out.seg_count)
        a.seg_ratio_out = _ptr(out.seg_ratio)
        a.seg_flag_out = _ptr(out.seg_flag)
        a.seg_loss_out = _ptr(out.seg_loss)
        a.token_advantages = _ptr(token_advantages)
        a.entropy_out = _ptr(out.entropy)
        keep = (logits, targets, loss_mask, teacher_logits, segment_ids, advantages, old_logprobs,
                token_advantages)
        return a, out, keep

    def call(self, args: "_lib.lmloss_args", stream: Optional[torch.cuda.Stream] = None):
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = _lib.lmloss_forward_backward(self.handle, args, s.cuda_stream)
        if st != _lib.LMLOSS_OK:
            raise LMLossError(st, "lmloss_forward_backward")

    def forward_backward(self, logits: torch.Tensor, targets: torch.Tensor, loss_mask=None,
                         stream: Optional[torch.cuda.Stream] = None, **kw) -> Outputs:
        args, out, _keep = self.build_args(logits, targets, loss_mask, **kw)
        self.call(args, stream)
        return out

    def call_host(self, args: "_lib.lmloss_args", host_logits: torch.Tensor, host_teacher=None,
                  chunk_rows: int = 0, stream: Optional[torch.cuda.Stream] = None):
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        st = _lib.lmloss_forward_backward_host(self.handle, args, _ptr(host_logits), _ptr(host_teacher),
                                               int(chunk_rows), s.cuda_stream)
        if st != _lib.LMLOSS_OK:
            raise LMLossError(st, "lmloss_forward_backward_host")

    def forward_backward_host(self, host_logits: torch.Tensor, logits: torch.Tensor, targets: torch.Tensor,
                              loss_mask=None, *, host_teacher=None, chunk_rows: int = 0,
                              stream: Optional[torch.cuda.Stream] = None, **kw) -> Outputs:
        """forward_backward with the logits (and the teacher's) taken from host
        tensors: the library copies them into `logits` (and `teacher_logits`) in
        row chunks and runs each chunk's kernel as soon as it has landed.  The
        host tensors must match the device ones in dtype, shape and strides, and
        should be pinned."""
        for hst, d, name in ((host_logits, logits, "host_logits"), (host_teacher, kw.get("teacher_logits"), "host_teacher")):
            if (hst is None) != (d is None):
                raise ValueError(f"{name} and its device tensor go together")
            if hst is not None and (hst.device.type != "cpu" or hst.dtype != d.dtype or hst.shape != d.shape
                                    or hst.stride() != d.stride()):
                raise ValueError(f"{name} must be a host tensor matching its device tensor")
        args, out, _keep = self.build_args(logits, targets, loss_mask, **kw)
        self.call_host(args, host_logits, host_teacher, chunk_rows, stream)
        return out

    # ------------------------------------------- vocabulary-split rows
    def _stream(self, stream):
        return (torch.cuda.current_stream(self.device) if stream is None else stream).cuda_stream

    def shard_stats(self, logits: torch.Tensor, targets: torch.Tensor, loss_mask=None, *, v0: int,
                    V_total: int, stream=None) -> torch.Tensor:
        """Per-row partial statistics [T, 4] of one vocabulary shard (columns
        [v0, v0 + logits.shape[1]) of V_total); targets are global column numbers."""
        a, _out, keep = self.build_args(logits, targets, loss_mask, grad=None, want=())
        part = torch.empty((logits.shape[0], 4), dtype=torch.float32, device=logits.device)
        st = _lib.load().lmloss_shard_stats(self.handle, a, int(v0), int(V_total), _ptr(part),
                                            self._stream(stream))
        if st != _lib.LMLOSS_OK:
            raise LMLossError(st, "lmloss_shard_stats")
        return part

    def shard_merge(self, parts, targets: torch.Tensor, loss_mask=None, *, V_total: int, ce_weight: float = 1.0,
                    z_alpha: float = 0.0, reduction: str = "token_mean", denominator: float = 1.0,
                    want=("logp", "lse", "count"), stream=None) -> Outputs:
        """Merge the shards' partials (a list of [T, 4] tensors, in shard order) into
        the rows' NLL and lse and the losses; the statistics stay in the handle for
        shard_grad."""
        T = targets.shape[0]
        dev = targets.device
        _need(targets, "targets", torch.int64, T, dev)
        if loss_mask is not None:
            _need(loss_mask, "loss_mask", torch.uint8, T, dev)
        for k, q in enumerate(parts):
            _need(q, f"parts[{k}]", torch.float32, 4 * T, dev)
        f32 = dict(dtype=torch.float32, device=dev)
        out = Outputs(loss=torch.empty(5, **f32))
        out.logp = torch.empty(T, **f32) if "logp" in want else None
        out.lse = torch.empty(T, **f32) if "lse" in want else None
        out.count = torch.empty(2, dtype=torch.int64, device=dev) if "count" in want else None
        a = _lib.lmloss_args()
        a.T, a.V, a.ld = T, int(V_total), int(V_total)
        a.dtype = _lib.LMLOSS_FP32
        a.reduction = _RED[reduction]
        a.targets = _ptr(targets)
        a.loss_mask = _ptr(loss_mask)
        a.ce_weight = float(ce_weight)
        a.z_alpha = float(z_alpha)
        a.temperature = 1.0
        a.denominator = float(denominator)
        a.loss_out = _ptr(out.loss)
        a.logp_out = _ptr(out.logp)
        a.lse_out = _ptr(out.lse)
        a.count_out = _ptr(out.count)
        ptrs = (ctypes.c_void_p * len(parts))(*[_ptr(q) for q in parts])
        st = _lib.load().lmloss_shard_merge(self.handle, a, ptrs, len(parts), self._stream(stream))
        if st != _lib.LMLOSS_OK:
            raise LMLossError(st, "lmloss_shard_merge")
        return out

    def shard_grad(self, logits: torch.Tensor, targets: torch.Tensor, loss_mask=None, *, v0: int, V_total: int,
                   ce_weight: float = 1.0, z_alpha: float = 0.0, reduction: str = "token_mean",
                   denominator: float = 1.0, grad: Union[str, torch.Tensor] = "new", stream=None) -> torch.Tensor:
        """Gradient of one vocabulary shard from the statistics of the last shard_merge."""
        a, out, keep = self.build_args(logits, targets, loss_mask, ce_weight=ce_weight, z_alpha=z_alpha,
                                       reduction=reduction, denominator=denominator, grad=grad, want=())
        st = _lib.load().lmloss_shard_grad(self.handle, a, int(v0), int(V_total), self._stream(stream))
        if st != _lib.LMLOSS_OK:
            raise LMLossError(st, "lmloss_shard_grad")
        return out.grad


def lmloss_forward_backward(logits, targets, loss_mask=None, **kw) -> Outputs:
    """One-shot convenience: creates a handle sized for this call."""
    seg = kw.get("segment_ids")
    S = 0 if seg is None else int(kw.get("num_segments") or kw["advantages"].numel())
    h = LMLoss(logits.device, max_T=max(1, logits.shape[0]), max_segments=max(1, S))
    try:
        out = h.forward_backward(logits, targets, loss_mask, **kw)
        torch.cuda.current_stream(logits.device).synchronize()
        return out
    finally:
        h.close()
