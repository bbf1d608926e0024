"""Build and load the in-tree CUDA library libidxtopk.so (sm_103a).

build() compiles the translation units under csrc/ in parallel with nvcc and
links one shared library next to this file (git-ignored).  load() opens it
with ctypes and declares the C ABI of include/idxtopk.h.  There is no fallback:
if the library cannot be built or loaded, load() raises.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
CSRC = os.path.join(_HERE, "csrc")
INCLUDE = os.path.join(_ROOT, "include")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_HERE, "libidxtopk.so")
# the range-checked variant (-DIDX_DEBUG_BOUNDS): every indexed scratch and
# output access of the kernels is checked; an index outside its buffer fails
# the call with IDX_ERR_INTERNAL instead of touching memory (a software stand-in
# for a memory checker, run by the GPU tests on small cases)
DEBUG_BUILD_DIR = os.path.join(_HERE, "_build_dbg")
DEBUG_LIB_PATH = os.path.join(_HERE, "libidxtopk_dbg.so")
SOURCES = ["host.cu", "plan.cu", "score.cu", "finish.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I" + INCLUDE, "-I" + CSRC] + ARCH

_lock = threading.Lock()
_lib = None


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: cannot build the sm_103a library")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "idxtopk.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a and link libidxtopk.so (no-op when fresh);
    debug_bounds=True builds the range-checked libidxtopk_dbg.so instead."""
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug_bounds else BUILD_DIR
    flags = NVCC_FLAGS + (["-DIDX_DEBUG_BOUNDS"] if debug_bounds else [])
    if (not force and os.path.exists(lib_path)
            and os.path.getmtime(lib_path) >= _deps_mtime()):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared"] + ARCH + objs + ["-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


class IdxTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


# descriptors are passed as addresses (the binding packs them into one buffer per call)
_DESC_PTR = ctypes.c_void_p

EXPORTS = {
    "idx_topk_fp4_prefill": (ctypes.c_int, [_DESC_PTR] * 9 +
                             [ctypes.c_int32, _DESC_PTR, _DESC_PTR,
                              ctypes.c_void_p]),
    "idx_topk_fp4_prefill_paged": (ctypes.c_int, [_DESC_PTR] * 8 +
                                   [ctypes.c_int32, _DESC_PTR,
                                    _DESC_PTR, ctypes.c_void_p]),
    "idx_topk_fp4_prefill_async": (ctypes.c_int, [_DESC_PTR] * 9 +
                                   [ctypes.c_int32, _DESC_PTR,
                                    _DESC_PTR, ctypes.c_void_p, ctypes.c_uint64,
                                    ctypes.c_void_p, ctypes.c_void_p]),
    "idx_topk_fp4_prefill_host": (ctypes.c_int, [_DESC_PTR] * 9 +
                                  [ctypes.c_int32, _DESC_PTR,
                                   _DESC_PTR, ctypes.c_int32, ctypes.c_void_p]),
    "idx_topk_fp4_prefill_noalloc": (ctypes.c_int, [_DESC_PTR] * 9 +
                                     [ctypes.c_int32, _DESC_PTR,
                                      _DESC_PTR, ctypes.c_void_p]),
    "idx_topk_fp4_prefill_mma_scales": (ctypes.c_int, [_DESC_PTR] * 9 +
                                        [ctypes.c_int32, _DESC_PTR,
                                         _DESC_PTR, ctypes.c_void_p]),
    "idx_topk_fp4_prefill_shard": (ctypes.c_int, [_DESC_PTR] * 9 +
                                   [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    _DESC_PTR, _DESC_PTR,
                                    ctypes.c_void_p]),
    "idx_topk_merge_shards": (ctypes.c_int, [_DESC_PTR] * 6 +
                              [ctypes.c_int32, _DESC_PTR,
                               _DESC_PTR, ctypes.c_void_p]),
    "idx_tiled_topk_fp4_prefill": (ctypes.c_int, [_DESC_PTR] * 9 +
                                   [ctypes.c_int32, ctypes.c_int32, _DESC_PTR,
                                    _DESC_PTR, ctypes.c_void_p]),
    "idx_dense_topk_fp4_prefill": (ctypes.c_int, [_DESC_PTR] * 9 +
                                   [ctypes.c_int32] + [_DESC_PTR] * 3 +
                                   [ctypes.c_void_p]),
    "idx_fp4_debug_scores": (ctypes.c_int, [_DESC_PTR] * 11 + [ctypes.c_void_p]),
    "idx_topk_select_scores": (ctypes.c_int, [_DESC_PTR] * 3 +
                               [ctypes.c_int32, _DESC_PTR, ctypes.c_void_p]),
    "idx_topk_supported_k": (ctypes.c_int, [ctypes.POINTER(ctypes.POINTER(ctypes.c_int32)),
                                            ctypes.POINTER(ctypes.c_int32)]),
    "idx_topk_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "idx_topk_fp4_scratch_bytes": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                  ctypes.POINTER(ctypes.c_uint64)]),
    "idx_topk_scratch_high_water": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_uint64)]),
    "idx_debug_bounded_wait": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]),
    "idx_topk_set_timing": (ctypes.c_int, [ctypes.c_int32]),
    "idx_topk_last_timings": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float)]),
}


def load(path: str = None):
    """Build if needed, then open the library and declare its C ABI."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib = ctypes.CDLL(path or build())
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib
