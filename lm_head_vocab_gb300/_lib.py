"""ctypes binding of the lmloss C ABI (include/lmloss.h): same names, argument
marshalling only.  The CUDA library must have been built (``build()``); nothing
here computes any part of the loss, and there is no CPU fallback."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_BUILD = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(_BUILD, "liblmloss.so")
HEADER = os.path.join(_ROOT, "include", "lmloss.h")
# (source, extra flags, object): the host code with the small kernels, and the
# staged-row kernel's eight (dtype, teacher, temperature, entropy) instantiation
# sets, one object each so that they compile in parallel
UNITS = [("lmloss.cu", [], "lmloss.o")] + [
    ("fused_inst.cu", [f"-DLMLOSS_FUSED_VARIANT={k}"], f"fused_{k}.o") for k in range(8)]
DEPENDS = ["lmloss.cu", "fused_inst.cu", "fused_entry.cuh", "kernels.cuh", "aux_kernels.cuh", "ptx.cuh"]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC"]

LMLOSS_OK = 0
LMLOSS_ERR_INVALID_ARG = 1
LMLOSS_ERR_UNSUPPORTED = 2
LMLOSS_ERR_CUDA = 3
LMLOSS_ERR_BAD_TARGET = 4
LMLOSS_ERR_BAD_SEGMENT = 5
LMLOSS_ERR_RANGE = 6
LMLOSS_ERR_TIMEOUT = 7
LMLOSS_BF16 = 0
LMLOSS_FP32 = 1
LMLOSS_REDUCE_SUM = 0
LMLOSS_REDUCE_TOKEN_MEAN = 1
LMLOSS_IGNORE_INDEX = -100


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a into the package's _build folder:
    every translation unit at once, then one link."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(os.path.join(_CSRC, f)) for f in DEPENDS)
    newest = max(newest, os.path.getmtime(HEADER))
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    work = os.path.join(_BUILD, f"tmp{os.getpid()}")
    os.makedirs(work, exist_ok=True)
    objs, procs = [], []
    try:
        for src, extra, obj in UNITS:
            o = os.path.join(work, obj)
            objs.append(o)
            cmd = [_nvcc(), *NVCC_FLAGS, *extra, "-c", "-o", o, os.path.join(_CSRC, src)]
            procs.append((cmd, subprocess.Popen(cmd)))
        failed = [cmd for cmd, pr in procs if pr.wait() != 0]
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = os.path.join(work, "liblmloss.so")
        subprocess.run([_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs],
                       check=True)
        os.replace(tmp, LIB_PATH)
    finally:
        for _, pr in procs:
            if pr.poll() is None:
                pr.kill()
                pr.wait()
        shutil.rmtree(work, ignore_errors=True)
    return LIB_PATH


class lmloss_args(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("T", ctypes.c_int64),
        ("V", ctypes.c_int64),
        ("ld", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("reduction", ctypes.c_int32),
        ("targets", ctypes.c_void_p),
        ("loss_mask", ctypes.c_void_p),
        ("ce_weight", ctypes.c_float),
        ("z_alpha", ctypes.c_float),
        ("teacher_logits", ctypes.c_void_p),
        ("kl_weight", ctypes.c_float),
        ("temperature", ctypes.c_float),
        ("segment_ids", ctypes.c_void_p),
        ("num_segments", ctypes.c_int32),
        ("advantages", ctypes.c_void_p),
        ("old_logprobs", ctypes.c_void_p),
        ("clip_eps_low", ctypes.c_float),
        ("clip_eps_high", ctypes.c_float),
        ("denominator", ctypes.c_double),
        ("grad_out", ctypes.c_void_p),
        ("loss_out", ctypes.c_void_p),
        ("logp_out", ctypes.c_void_p),
        ("lse_out", ctypes.c_void_p),
        ("kl_out", ctypes.c_void_p),
        ("count_out", ctypes.c_void_p),
        ("seg_count_out", ctypes.c_void_p),
        ("seg_ratio_out", ctypes.c_void_p),
        ("seg_flag_out", ctypes.c_void_p),
        ("seg_loss_out", ctypes.c_void_p),
        ("token_advantages", ctypes.c_void_p),
        ("entropy_out", ctypes.c_void_p),
    ]


class lmloss_call_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("launches", "path", "cluster", "threads", "nbuf", "grid", "smem_bytes", "reserved")]


_lib: Optional[ctypes.CDLL] = None


def load() -> ctypes.CDLL:
    """Load the built library.  Raises if it was never built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"lmloss CUDA library not built ({LIB_PATH} missing); run build() first")
    lib = ctypes.CDLL(LIB_PATH)
    h = ctypes.c_void_p
    st = ctypes.c_int
    sig = {
        "lmloss_create": ([ctypes.POINTER(h), ctypes.c_int, ctypes.c_int64, ctypes.c_int32], st),
        "lmloss_destroy": ([h], st),
        "lmloss_check_args": ([ctypes.POINTER(lmloss_args)], st),
        "lmloss_forward_backward": ([h, ctypes.POINTER(lmloss_args), ctypes.c_void_p], st),
        "lmloss_get_device_error": ([h], st),
        "lmloss_status_string": ([st], ctypes.c_char_p),
        "lmloss_set_launch_config": ([h, ctypes.c_int, ctypes.c_int, ctypes.c_int], st),
        "lmloss_forward_backward_host": ([h, ctypes.POINTER(lmloss_args), ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_void_p], st),
        "lmloss_set_timing": ([h, ctypes.c_int], st),
        "lmloss_get_timing": ([h, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32)], st),
        "lmloss_get_call_info": ([h, ctypes.POINTER(lmloss_call_info)], st),
        "lmloss_selftest_bounded_wait": ([h, ctypes.c_longlong], st),
        "lmloss_shard_stats": ([h, ctypes.POINTER(lmloss_args), ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_void_p], st),
        "lmloss_shard_merge": ([h, ctypes.POINTER(lmloss_args), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                                ctypes.c_void_p], st),
        "lmloss_shard_grad": ([h, ctypes.POINTER(lmloss_args), ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def exported_names():
    """Function names declared in include/lmloss.h."""
    import re
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:lmloss_status|const char\*)\s+(lmloss_\w+)\s*\(", txt, re.M)))


class LMLossError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = lmloss_status_string(status)
        super().__init__(f"{where}: {msg} (status {status})" if where else f"{msg} (status {status})")


# ---- same-name wrappers over the C entry points -----------------------------
def lmloss_status_string(status: int) -> str:
    return load().lmloss_status_string(int(status)).decode()


def lmloss_create(device: int, max_T: int, max_segments: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    st = load().lmloss_create(ctypes.byref(h), int(device), int(max_T), int(max_segments))
    if st != LMLOSS_OK:
        raise LMLossError(st, "lmloss_create")
    return h


def lmloss_destroy(handle) -> int:
    return load().lmloss_destroy(handle)


def lmloss_check_args(args: lmloss_args) -> int:
    return load().lmloss_check_args(ctypes.byref(args))


def lmloss_forward_backward(handle, args: lmloss_args, stream: int) -> int:
    return load().lmloss_forward_backward(handle, ctypes.byref(args), ctypes.c_void_p(stream))


def lmloss_get_device_error(handle) -> int:
    return load().lmloss_get_device_error(handle)


def lmloss_forward_backward_host(handle, args, host_logits, host_teacher, chunk_rows: int, stream) -> int:
    return load().lmloss_forward_backward_host(handle, ctypes.byref(args), host_logits, host_teacher, chunk_rows,
                                               ctypes.c_void_p(stream))


def lmloss_set_launch_config(handle, cluster: int = 0, threads: int = 0, nbuf: int = 0) -> int:
    return load().lmloss_set_launch_config(handle, cluster, threads, nbuf)


def lmloss_set_timing(handle, enable: bool) -> int:
    return load().lmloss_set_timing(handle, 1 if enable else 0)


def lmloss_get_timing(handle):
    """(summed main-kernel milliseconds, calls recorded) since timing was enabled."""
    ms = ctypes.c_float()
    n = ctypes.c_int32()
    st = load().lmloss_get_timing(handle, ctypes.byref(ms), ctypes.byref(n))
    if st != LMLOSS_OK:
        raise LMLossError(st, "lmloss_get_timing")
    return float(ms.value), int(n.value)


def lmloss_selftest_bounded_wait(handle, limit_cycles: int) -> int:
    return load().lmloss_selftest_bounded_wait(handle, int(limit_cycles))


def lmloss_get_call_info(handle) -> dict:
    info = lmloss_call_info()
    st = load().lmloss_get_call_info(handle, ctypes.byref(info))
    if st != LMLOSS_OK:
        raise LMLossError(st, "lmloss_get_call_info")
    return {n: getattr(info, n) for n, _ in lmloss_call_info._fields_}


def lmloss_forward_backward_noalloc(args: lmloss_args, stream: int) -> int:
    """Allocation-free variant of lmloss_forward_backward on the current device.

    For callers that may not allocate device memory once running (an
    inference-engine plugin whose enqueue step must not allocate, or a service
    that plans all device memory at start-up).  The workspace is a fixed array
    inside the library; a call with more than LMLOSS_NOALLOC_MAX_T rows or
    LMLOSS_NOALLOC_MAX_SEGMENTS segments returns LMLOSS_ERR_INVALID_ARG.  The
    first call on a device does a one-time look-up (make it before any stream
    capture); calls that overlap on the GPU share the array and race.
    """
    fn = load().lmloss_forward_backward_noalloc
    fn.argtypes = [ctypes.POINTER(lmloss_args), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(args), ctypes.c_void_p(stream))
