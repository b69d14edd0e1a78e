"""Fused LM-head loss: plain fp64 CPU oracle (Python half).

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg import this module.  The product path never does,
and nothing here is shared with the CUDA library.

Row-level arithmetic (logsumexp, softplus, softmax, KL, the per-row gradient)
lives in ``oracle.c``; this file does the O(T) bookkeeping in plain Python /
numpy fp64: the active-token mask, the GSPO segment seam, the reduction scales
and the final sums.

Sources (page title, then section):
  torchtitan PR 5661 "fix softmax collapse with improved CE perf", commit
      message, "Numerics (TP > 1 only)": ignored labels give a finite loss and
      gradient that the label mask then zeroes.
  xtuner PR 1963 "[FSDP][Loss] Switch gradient reduction to SUM", description:
      under SUM reduction each shard's loss is its local component, the sum over
      its tokens divided by the *global* token count; z-loss diff: the z term is
      scaled by z_loss_alpha / batch_size.
  Fast-LLM PR 552 "Fuse GSPO into the monolithic compiled loss (#507)",
      "Why it needed special handling": GSPO aggregates per segment with an
      index_add over a per-batch num_segments, then clips, between forward and
      backward.

Readings where the pages are silent (each listed in the design notes):
  * ignore_index is -100; a row is active iff target != -100 and (no mask or
    mask != 0).
  * "batch_size" in the z-loss scale is the same denominator as the CE term.
  * TOKEN_MEAN with no active token gives scale 0 (loss 0, gradient 0).
  * GSPO under TOKEN_MEAN is averaged over the non-empty segments; under SUM it
    is divided by the caller's denominator like every other term.
  * A GSPO segment's gradient flows iff s_i*A_i <= clamp(s_i)*A_i (ties flow).
  * Tokens with a negative segment id belong to no segment.
  * GRPO (named on the Fast-LLM page as a combinable loss that shares the
    softmax, without a formula) is read as the token-level version of the same
    clipped surrogate: rho_r = exp(logp_r - old_logp_r),
    L_r = -min(rho_r A_r, clamp(rho_r, 1-eps_lo, 1+eps_hi) A_r), its gradient
    flowing iff rho_r A_r <= clamp(rho_r) A_r, reduced like the token terms.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

IGNORE_INDEX = -100
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

BF16 = 0
FP32 = 1
REDUCE_SUM = 0
REDUCE_TOKEN_MEAN = 1


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (fp64, no FMA contraction, OpenMP over rows)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        d = ctypes.c_double
        lib.orc_forward.argtypes = [ctypes.c_int, i64, i64, i64, p, p, d, p, p, p, p, p, p, ctypes.c_int]
        lib.orc_forward.restype = ctypes.c_int
        lib.orc_grad.argtypes = [ctypes.c_int, i64, i64, i64, p, p, d, p, p, d, d, d, d, p, p, p, ctypes.c_int]
        lib.orc_grad.restype = ctypes.c_int
        lib.orc_entropy.argtypes = [ctypes.c_int, i64, i64, i64, p, p, p, ctypes.c_int]
        lib.orc_entropy.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Problem:
    """One call's inputs, all host numpy arrays.

    logits / teacher: [T, ld] uint16 (bf16 bit patterns) or float32; the first V
    columns of each row are the logits.
    """
    logits: np.ndarray
    V: int
    targets: np.ndarray                      # int64 [T]
    loss_mask: Optional[np.ndarray] = None   # uint8 [T] or None
    ce_weight: float = 1.0
    z_alpha: float = 0.0
    teacher: Optional[np.ndarray] = None
    kl_weight: float = 0.0
    temperature: float = 1.0
    segment_ids: Optional[np.ndarray] = None  # int32 [T]
    num_segments: int = 0
    advantages: Optional[np.ndarray] = None   # float32 [S]
    old_logprobs: Optional[np.ndarray] = None  # float32 [T]
    token_advantages: Optional[np.ndarray] = None  # float32 [T]: GRPO (per-token) advantages
    clip_eps_low: float = 0.0
    clip_eps_high: float = 0.0
    reduction: int = REDUCE_TOKEN_MEAN
    denominator: float = 1.0

    def __post_init__(self):
        # the C oracle reads the buffers by these element types: anything else
        # would be reinterpreted, not converted
        if self.logits.dtype not in (np.uint16, np.float32) or self.logits.ndim != 2:
            raise TypeError("logits must be a 2-D uint16 (bf16 bits) or float32 array")
        if self.teacher is not None and (self.teacher.dtype != self.logits.dtype
                                         or self.teacher.shape != self.logits.shape):
            raise TypeError("teacher must match logits in dtype and shape")

    @property
    def T(self) -> int:
        return int(self.logits.shape[0])

    @property
    def ld(self) -> int:
        return int(self.logits.shape[1])

    @property
    def dtype(self) -> int:
        return BF16 if self.logits.dtype == np.uint16 else FP32


def active_mask(targets: np.ndarray, loss_mask: Optional[np.ndarray]) -> np.ndarray:
    """Row r takes part iff targets[r] != -100 and (no mask or mask[r] != 0)."""
    act = targets != IGNORE_INDEX
    if loss_mask is not None:
        act = act & (loss_mask != 0)
    return act.astype(np.uint8)


def row_forward(P: Problem, active: np.ndarray, nthreads: int = 0):
    """Per-row nll, lse, lse_nt, kl (fp64 [T] each); zeros on inactive rows."""
    lib = _load()
    T = P.T
    logits = np.ascontiguousarray(P.logits)
    teacher = None if P.teacher is None else np.ascontiguousarray(P.teacher)
    if teacher is not None and teacher.dtype != logits.dtype:
        raise ValueError("teacher and logits must share a dtype")
    targets = np.ascontiguousarray(P.targets, dtype=np.int64)
    act = np.ascontiguousarray(active, dtype=np.uint8)
    bad = (act != 0) & ((targets < 0) | (targets >= P.V))
    if bad.any():
        raise ValueError("active row with a target outside [0, V)")
    out = [np.zeros(T, dtype=np.float64) for _ in range(4)]
    rc = lib.orc_forward(P.dtype, T, P.V, P.ld, _ptr(logits), _ptr(teacher), float(P.temperature),
                         _ptr(targets), _ptr(act), *[_ptr(o) for o in out], int(nthreads))
    if rc != 0:
        raise MemoryError("oracle: out of host memory")
    return tuple(out)


def entropy(P: Problem, active: Optional[np.ndarray] = None, nthreads: int = 0) -> np.ndarray:
    """Per-row entropy of softmax(z) (fp64 [T]); 0 on inactive rows."""
    lib = _load()
    act = active_mask(P.targets, P.loss_mask) if active is None else active
    logits = np.ascontiguousarray(P.logits)
    out = np.zeros(P.T, dtype=np.float64)
    rc = lib.orc_entropy(P.dtype, P.T, P.V, P.ld, _ptr(logits), _ptr(np.ascontiguousarray(act, dtype=np.uint8)),
                         _ptr(out), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle: out of host memory")
    return out


@dataclass
class Seam:
    """GSPO per-segment results (all [S])."""
    n: np.ndarray          # int64 active-token count
    D: np.ndarray          # fp64 sum of (logp_t - old_logp)
    ratio: np.ndarray      # s_i = exp(D_i / n_i)            (0 for empty segments)
    clipped: np.ndarray    # clamp(s_i, 1-eps_lo, 1+eps_hi)
    loss: np.ndarray       # L_i = -min(s_i A_i, clamp(s_i) A_i)  (0 for empty)
    flag: np.ndarray       # uint8, 1 iff the gradient flows through s_i
    nonempty: int


def gspo_seam(logp: np.ndarray, old_logprobs: np.ndarray, segment_ids: np.ndarray,
              active: np.ndarray, advantages: np.ndarray, num_segments: int,
              eps_low: float, eps_high: float) -> Seam:
    """Segment index-add then clipping, as a plain loop over tokens then segments."""
    S = int(num_segments)
    n = np.zeros(S, dtype=np.int64)
    D = np.zeros(S, dtype=np.float64)
    seg = segment_ids.astype(np.int64)
    for r in range(len(seg)):
        g = int(seg[r])
        if not active[r] or g < 0:
            continue
        if g >= S:
            raise ValueError("segment id outside [0, num_segments)")
        n[g] += 1
        D[g] += float(logp[r]) - float(old_logprobs[r])
    ratio = np.zeros(S)
    clipped = np.zeros(S)
    loss = np.zeros(S)
    flag = np.zeros(S, dtype=np.uint8)
    lo, hi = 1.0 - float(eps_low), 1.0 + float(eps_high)
    for i in range(S):
        if n[i] == 0:
            continue
        A = float(advantages[i])
        s = math.exp(D[i] / n[i])
        c = min(max(s, lo), hi)
        ratio[i] = s
        clipped[i] = c
        loss[i] = -min(s * A, c * A)
        flag[i] = 1 if s * A <= c * A else 0
    return Seam(n, D, ratio, clipped, loss, flag, int((n > 0).sum()))


@dataclass
class Result:
    active: np.ndarray
    n_active: int
    s_tok: float
    s_seg: float
    nll: np.ndarray
    lse: np.ndarray
    lse_nt: np.ndarray
    kl: np.ndarray
    logp: np.ndarray
    ce: float        # s_tok * sum nll
    z: float         # s_tok * sum alpha * lse^2
    kl_loss: float   # s_tok * sum kl
    gspo: float      # policy term: s_seg * sum L_i (GSPO) or s_tok * sum L_r (GRPO)
    total: float     # ce_weight*ce + z + kl_weight*kl + gspo
    seam: Optional[Seam] = None
    coef: Optional[np.ndarray] = None   # per-row GSPO coefficient c_r
    extra: dict = field(default_factory=dict)


def forward(P: Problem, nthreads: int = 0) -> Result:
    """Losses and per-row scalars for a whole problem."""
    act = active_mask(P.targets, P.loss_mask)
    nll, lse, lse_nt, kl = row_forward(P, act, nthreads)
    n_active = int(act.sum())
    if P.reduction == REDUCE_TOKEN_MEAN:
        s_tok = 1.0 / n_active if n_active > 0 else 0.0
    else:
        s_tok = 1.0 / float(P.denominator)
    logp = -nll
    ce = s_tok * float(np.sum(nll))
    z = s_tok * float(np.sum(P.z_alpha * lse * lse))
    kl_loss = s_tok * float(np.sum(kl))
    seam = None
    coef = None
    gspo = 0.0
    s_seg = 0.0
    if P.segment_ids is not None:
        seam = gspo_seam(logp, P.old_logprobs, P.segment_ids, act, P.advantages,
                         P.num_segments, P.clip_eps_low, P.clip_eps_high)
        if P.reduction == REDUCE_TOKEN_MEAN:
            s_seg = 1.0 / seam.nonempty if seam.nonempty > 0 else 0.0
        else:
            s_seg = 1.0 / float(P.denominator)
        gspo = s_seg * float(np.sum(seam.loss))
        # d L_i / d logp_t(r) for a flowing segment is -A_i s_i / n_i, and
        # d logp_t / d z_j = [j==t] - p_j, so the row gradient is c_r (p - onehot).
        coef = np.zeros(P.T)
        for r in range(P.T):
            g = int(P.segment_ids[r])
            if act[r] and g >= 0 and seam.flag[g]:
                A = float(P.advantages[g])
                coef[r] = s_seg * A * seam.ratio[g] / seam.n[g]
    if P.token_advantages is not None:
        if P.segment_ids is not None:
            raise ValueError("GRPO and GSPO are exclusive")
        lo, hi = 1.0 - float(P.clip_eps_low), 1.0 + float(P.clip_eps_high)
        coef = np.zeros(P.T)
        pol = np.zeros(P.T)
        for r in range(P.T):
            if not act[r]:
                continue
            A = float(P.token_advantages[r])
            rho = math.exp(float(logp[r]) - float(P.old_logprobs[r]))
            c = min(max(rho, lo), hi)
            pol[r] = -min(rho * A, c * A)
            if rho * A <= c * A:
                coef[r] = s_tok * A * rho      # d L_r / d z = A rho (p - onehot)
        gspo = s_tok * float(np.sum(pol))
        s_seg = s_tok
    total = P.ce_weight * ce + z + P.kl_weight * kl_loss + gspo
    return Result(act, n_active, s_tok, s_seg, nll, lse, lse_nt, kl, logp,
                  ce, z, kl_loss, gspo, total, seam, coef)


def grad_rows(P: Problem, R: Result, rows: Optional[np.ndarray] = None, nthreads: int = 0,
              with_scale: bool = False):
    """fp64 gradient [len(rows), V] of the total loss for the given rows (default all).
    with_scale: also return, per element, the sum of the magnitudes of the terms
    that make up the gradient (a rounding error in one term is judged against it)."""
    lib = _load()
    if rows is None:
        rows = np.arange(P.T)
    rows = np.asarray(rows, dtype=np.int64)
    sub = np.ascontiguousarray(P.logits[rows])
    tsub = None if P.teacher is None else np.ascontiguousarray(P.teacher[rows])
    targets = np.ascontiguousarray(P.targets[rows], dtype=np.int64)
    act = np.ascontiguousarray(R.active[rows], dtype=np.uint8)
    coef = None if R.coef is None else np.ascontiguousarray(R.coef[rows])
    g = np.zeros((len(rows), P.V), dtype=np.float64)
    gs = np.zeros_like(g) if with_scale else None
    rc = lib.orc_grad(P.dtype, len(rows), P.V, sub.shape[1], _ptr(sub), _ptr(tsub), float(P.temperature),
                      _ptr(targets), _ptr(act), float(R.s_tok), float(P.ce_weight), float(P.z_alpha),
                      float(P.kl_weight), _ptr(coef), _ptr(g), _ptr(gs), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle: out of host memory")
    return (g, gs) if with_scale else g


def forward_backward(P: Problem, nthreads: int = 0, with_scale: bool = False):
    """(Result, fp64 gradient [T, V]) for a small problem; with_scale adds the
    per-element term magnitudes as a third item."""
    R = forward(P, nthreads)
    if with_scale:
        g, gs = grad_rows(P, R, None, nthreads, with_scale=True)
        return R, g, gs
    return R, grad_rows(P, R, None, nthreads)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
