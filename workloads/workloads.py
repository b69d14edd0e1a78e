"""Seeded synthetic workloads for the fused LM-head loss.

No loss arithmetic lives here: these functions draw logits, targets, masks,
planted margins and packed segments.  The same host arrays feed the CUDA path
(copied to the device) and the oracle, so both see identical bits.

Recipes (seed 0, counter-based Philox4x32-10, Box-Muller normals, bf16 by
round-to-nearest-even):

  ce_fp32_small    fp32, T=64, V=1024, logits N(0, 2^2), targets uniform; exactly
                   round(0.1 T) = 6 rows set to ignore_index -100 by a seeded
                   permutation; 8 of the other rows planted with
                   z_t = max_{j!=t} z_j + margin, margin alternating 20, 30;
                   token-mean.
  ce_z_bf16        bf16, T=8192, V=32000, logits N(0, 3^2); round(0.05 T) = 410
                   rows set to -100; z-loss alpha = 1e-4; gradient in place;
                   SUM reduction with denominator = number of active rows.
  confident_bf16   bf16, T=16384, V=128256, logits N(0, 2^2); round(0.3 T) = 4915
                   rows planted with margin U[15, 40] (added to the bf16 max, then
                   rounded to bf16); CE only; gradient in place; token-mean.
  gspo_z_bf16      bf16, T=32768 = 8 packed rows x 4096, V=151936, logits
                   N(0, 2.5^2); per packed row K ~ U{1..64} segments cut at K-1
                   distinct points drawn from 1..4095; global segment ids;
                   advantages N(0, 1) per segment; old log-prob noise N(0, 0.05^2)
                   per token (added to the oracle's log-prob by the caller);
                   clip [1 - 3e-4, 1 + 4e-4]; z-loss 1e-4; ce_weight 0; no mask;
                   token-mean.
  ce_z_kl_bf16     bf16, T=65536, V=262144, student N(0, 3^2); teacher =
                   bf16(student + N(0, 1^2)); temperature 1, KL weight 0.5,
                   z-loss 1e-4, ce_weight 1; round(0.05 T) rows with loss_mask 0;
                   gradient in place; token-mean.

Any workload can be shrunk (``.with_shape``) for fast parity cases: the recipe
is kept, only T, V (and the packed-row length for GSPO) change.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgen.so")
_lib = None

IGNORE_INDEX = -100

# Philox streams: one per kind of draw.
S_LOGITS, S_TEACHER, S_TARGETS, S_MASK, S_PLANT, S_MARGIN, S_SEGK, S_ADV, S_OLDLP = range(1, 10)
S_SEGCUT = 100   # + packed row index


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u32, i64, d, p, i = ctypes.c_uint32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.gen_normal_rows.argtypes = [u32, u32, u32, i64, i64, i64, i64, d, d, i, p, i]
        lib.gen_add_normal_rows.argtypes = [u32, u32, u32, i64, i64, i64, i64, d, i, p, p, i]
        lib.gen_normal_1d.argtypes = [u32, u32, u32, i64, i64, d, d, p]
        lib.gen_uniform_1d.argtypes = [u32, u32, u32, i64, i64, d, d, p]
        lib.gen_randint_1d.argtypes = [u32, u32, u32, i64, i64, i64, p]
        lib.gen_permutation.argtypes = [u32, u32, u32, i64, p]
        lib.gen_plant_rows.argtypes = [i, i64, i64, i64, p, p, p, i]
        lib.gen_philox_kat.argtypes = [p, p, p]
        for f in ("gen_normal_rows", "gen_add_normal_rows", "gen_normal_1d", "gen_uniform_1d",
                  "gen_randint_1d", "gen_permutation", "gen_plant_rows", "gen_philox_kat"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def philox_kat(ctr, key):
    lib = _load()
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    lib.gen_philox_kat(_p(c), _p(k), _p(o))
    return o


def normal_1d(seed, cfg, stream, n, mean=0.0, sigma=1.0, i0=0):
    out = np.empty(n, dtype=np.float64)
    _load().gen_normal_1d(seed, cfg, stream, i0, n, mean, sigma, _p(out))
    return out


def uniform_1d(seed, cfg, stream, n, lo, hi, i0=0):
    out = np.empty(n, dtype=np.float64)
    _load().gen_uniform_1d(seed, cfg, stream, i0, n, lo, hi, _p(out))
    return out


def randint_1d(seed, cfg, stream, n, rng, i0=0):
    out = np.empty(n, dtype=np.int64)
    _load().gen_randint_1d(seed, cfg, stream, i0, n, rng, _p(out))
    return out


def permutation(seed, cfg, stream, n):
    out = np.empty(n, dtype=np.int64)
    _load().gen_permutation(seed, cfg, stream, n, _p(out))
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: int
    T: int
    V: int
    dtype: str                       # "bf16" | "fp32"
    sigma: float
    seed: int = 0
    mask_count: int = 0              # rows masked
    mask_via: str = "ignore"         # "ignore" (target -100) | "loss_mask"
    plant_count: int = 0
    plant_margins: tuple = ()        # cycled fixed margins, or () with plant_range
    plant_range: Optional[tuple] = None
    z_alpha: float = 0.0
    ce_weight: float = 1.0
    kl_weight: float = 0.0
    teacher_sigma: Optional[float] = None
    temperature: float = 1.0
    reduction: str = "token_mean"    # "token_mean" | "sum_active"
    in_place: bool = False
    packed_len: int = 0              # GSPO: tokens per packed row (0 = no GSPO)
    max_seg_per_row: int = 64
    clip_eps_low: float = 0.0
    clip_eps_high: float = 0.0
    old_logp_sigma: float = 0.05
    ld: int = 0                      # row stride in elements (0 = V)

    # ---------------------------------------------------------------- shape
    @property
    def row_stride(self) -> int:
        return self.ld if self.ld else self.V

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def np_dtype(self):
        return np.uint16 if self.dtype == "bf16" else np.float32

    @property
    def gen_dtype(self) -> int:
        return 0 if self.dtype == "bf16" else 1

    @property
    def has_gspo(self) -> bool:
        return self.packed_len > 0

    def with_shape(self, T: int, V: int, ld: int = 0, packed_len: Optional[int] = None) -> "Workload":
        """Same recipe at another size; counts scale with T."""
        scale = T / self.T
        kw = dict(T=T, V=V, ld=ld,
                  mask_count=int(round(self.mask_count * scale)),
                  plant_count=min(T, int(round(self.plant_count * scale))) if self.plant_count else 0)
        if self.has_gspo:
            kw["packed_len"] = packed_len if packed_len else max(2, min(self.packed_len, T))
            kw["max_seg_per_row"] = max(1, min(self.max_seg_per_row, kw["packed_len"] // 2))
        return replace(self, **kw)

    # ------------------------------------------------------------- O(T) parts
    def targets(self) -> np.ndarray:
        t = randint_1d(self.seed, self.cfg, S_TARGETS, self.T, self.V)
        if self.mask_via == "ignore" and self.mask_count:
            t[self.masked_rows()] = IGNORE_INDEX
        return t

    def masked_rows(self) -> np.ndarray:
        if not self.mask_count:
            return np.zeros(0, dtype=np.int64)
        return np.sort(permutation(self.seed, self.cfg, S_MASK, self.T)[: self.mask_count])

    def loss_mask(self) -> Optional[np.ndarray]:
        if self.mask_via != "loss_mask":
            return None
        m = np.ones(self.T, dtype=np.uint8)
        m[self.masked_rows()] = 0
        return m

    def margins(self) -> np.ndarray:
        """Per-row planted margin, NaN where nothing is planted."""
        out = np.full(self.T, np.nan)
        if not self.plant_count:
            return out
        masked = set(self.masked_rows().tolist())
        order = [r for r in permutation(self.seed, self.cfg, S_PLANT, self.T).tolist() if r not in masked]
        chosen = order[: self.plant_count]
        if self.plant_margins:
            for k, r in enumerate(chosen):
                out[r] = self.plant_margins[k % len(self.plant_margins)]
        else:
            lo, hi = self.plant_range
            u = uniform_1d(self.seed, self.cfg, S_MARGIN, self.T, lo, hi)
            for r in chosen:
                out[r] = u[r]
        return out

    def n_active(self) -> int:
        t = self.targets()
        act = t != IGNORE_INDEX
        m = self.loss_mask()
        if m is not None:
            act &= m != 0
        return int(act.sum())

    def denominator(self) -> float:
        return float(self.n_active()) if self.reduction == "sum_active" else 1.0

    # --------------------------------------------------------------- rows
    def logits_rows(self, r0: int, n: int, targets: Optional[np.ndarray] = None,
                    margins: Optional[np.ndarray] = None, nthreads: int = 0) -> np.ndarray:
        """Rows [r0, r0+n) of the student logits, [n, ld], padding columns 0."""
        lib = _load()
        ld = self.row_stride
        out = np.zeros((n, ld), dtype=self.np_dtype)
        lib.gen_normal_rows(self.seed, self.cfg, S_LOGITS, r0, n, self.V, ld, 0.0, self.sigma,
                            self.gen_dtype, _p(out), nthreads)
        if self.plant_count:
            t = (self.targets() if targets is None else targets)[r0:r0 + n]
            mg = (self.margins() if margins is None else margins)[r0:r0 + n]
            t = np.ascontiguousarray(t, dtype=np.int64)
            mg = np.ascontiguousarray(mg, dtype=np.float64)
            lib.gen_plant_rows(self.gen_dtype, n, self.V, ld, _p(out), _p(t), _p(mg), nthreads)
        return out

    def teacher_rows(self, r0: int, n: int, student: np.ndarray, nthreads: int = 0) -> Optional[np.ndarray]:
        """Rows of teacher = round(student + N(0, teacher_sigma^2))."""
        if self.teacher_sigma is None:
            return None
        out = np.zeros_like(student)
        _load().gen_add_normal_rows(self.seed, self.cfg, S_TEACHER, r0, n, self.V, self.row_stride,
                                    self.teacher_sigma, self.gen_dtype, _p(student), _p(out), nthreads)
        return out

    # --------------------------------------------------------------- GSPO
    def segments(self):
        """(segment_ids int32 [T], num_segments, advantages float32 [S])."""
        if not self.has_gspo:
            return None, 0, None
        L = self.packed_len
        n_packed = self.T // L
        seg = np.full(self.T, -1, dtype=np.int32)
        k_per_row = randint_1d(self.seed, self.cfg, S_SEGK, n_packed, self.max_seg_per_row) + 1
        nxt = 0
        for p in range(n_packed):
            K = int(min(k_per_row[p], L))
            cuts = np.sort(permutation(self.seed, self.cfg, S_SEGCUT + p, L - 1)[: K - 1] + 1)
            bounds = [0] + cuts.tolist() + [L]
            for s in range(K):
                seg[p * L + bounds[s]: p * L + bounds[s + 1]] = nxt
                nxt += 1
        adv = normal_1d(self.seed, self.cfg, S_ADV, nxt).astype(np.float32)
        return seg, nxt, adv

    def old_logp_noise(self) -> np.ndarray:
        return normal_1d(self.seed, self.cfg, S_OLDLP, self.T, 0.0, self.old_logp_sigma)

    # ---------------------------------------------------------------- bytes
    def algorithmic_bytes(self) -> int:
        """Bytes an ideal pass over this workload must move: every active row's
        logits read once (twice for GSPO, whose seam sits between the reads) and
        its teacher row once; every row's gradient written once (an inactive
        row's is zeros, and its logits are never read); plus the per-row side
        inputs."""
        e = self.elem_bytes
        n_act = self.n_active()
        row = self.V * e
        reads = (2 if self.has_gspo else 1) * n_act * row
        if self.teacher_sigma is not None:
            reads += n_act * row
        writes = self.T * row
        side = 8 * self.T
        if self.mask_via == "loss_mask":
            side += self.T
        if self.has_gspo:
            side += 4 * self.T + 4 * self.T + 4 * self.segments()[1]
        return reads + writes + side


WORKLOADS = {
    "ce_fp32_small": Workload(
        name="ce_fp32_small", cfg=1, T=64, V=1024, dtype="fp32", sigma=2.0,
        mask_count=6, mask_via="ignore", plant_count=8, plant_margins=(20.0, 30.0),
        reduction="token_mean"),
    "ce_z_bf16": Workload(
        name="ce_z_bf16", cfg=2, T=8192, V=32000, dtype="bf16", sigma=3.0,
        mask_count=410, mask_via="ignore", z_alpha=1e-4, reduction="sum_active", in_place=True),
    "confident_bf16": Workload(
        name="confident_bf16", cfg=3, T=16384, V=128256, dtype="bf16", sigma=2.0,
        plant_count=4915, plant_range=(15.0, 40.0), reduction="token_mean", in_place=True),
    "gspo_z_bf16": Workload(
        name="gspo_z_bf16", cfg=4, T=32768, V=151936, dtype="bf16", sigma=2.5,
        packed_len=4096, max_seg_per_row=64, clip_eps_low=3e-4, clip_eps_high=4e-4,
        z_alpha=1e-4, ce_weight=0.0, reduction="token_mean"),
    "ce_z_kl_bf16": Workload(
        name="ce_z_kl_bf16", cfg=5, T=65536, V=262144, dtype="bf16", sigma=3.0,
        teacher_sigma=1.0, temperature=1.0, kl_weight=0.5, z_alpha=1e-4, ce_weight=1.0,
        mask_count=3277, mask_via="loss_mask", reduction="token_mean", in_place=True),
}

ORDER = ["ce_fp32_small", "ce_z_bf16", "confident_bf16", "gspo_z_bf16", "ce_z_kl_bf16"]


def get(name: str) -> Workload:
    return WORKLOADS[name]


def mask_count_for(T: int, frac: float) -> int:
    return int(math.floor(frac * T + 0.5))
