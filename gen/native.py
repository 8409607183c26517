"""ctypes bindings of the generator's host twin and device filler."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
HOST_SO = os.path.join(BUILD, "libgenhost.so")
DEV_SO = os.path.join(BUILD, "libgendev.so")
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(device: bool = True) -> None:
    """Compile the host twin (gcc) and, if `device`, the device filler (nvcc)."""
    os.makedirs(BUILD, exist_ok=True)
    procs = [subprocess.Popen(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-o", HOST_SO, os.path.join(HERE, "gen_host.c")])]
    if device:
        procs.append(subprocess.Popen([_nvcc(), "-O3", "-std=c++17", "-shared",
                                       "-Xcompiler", "-fPIC", *NVCC_ARCH, "-lineinfo",
                                       "-o", DEV_SO, os.path.join(HERE, "gen_dev.cu")]))
    for p in procs:
        if p.wait() != 0:
            raise RuntimeError("generator build failed")


_host = None
_dev = None


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_SO):
            build(device=False)
        lib = ctypes.CDLL(HOST_SO)
        vp, i64, i32, u64, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_uint64, ctypes.c_float)
        lib.gen_host_logits.argtypes = [u64, vp, vp, i64, i32, i32, vp, i32, f32, vp]
        lib.gen_host_logit_rows.argtypes = [u64, vp, vp, vp, vp, i64, i32, i32, vp, i32, f32, vp]
        lib.gen_host_hidden.argtypes = [u64, i64, i64, i32, vp]
        lib.gen_host_wgate.argtypes = [u64, i32, i32, i32, f32, vp]
        for f in (lib.gen_host_logits, lib.gen_host_logit_rows, lib.gen_host_hidden,
                  lib.gen_host_wgate):
            f.restype = None
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_SO):
            raise RuntimeError("device generator not built: run gen.build()")
        lib = ctypes.CDLL(DEV_SO)
        vp, i64, i32, u64, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_uint64, ctypes.c_float)
        lib.gen_dev_logits.argtypes = [u64, vp, vp, i64, i32, i32, vp, i32, f32, vp, vp]
        lib.gen_dev_hidden.argtypes = [u64, i64, i32, vp, vp]
        lib.gen_dev_wgate.argtypes = [u64, i32, i32, i32, f32, vp, vp]
        for f in (lib.gen_dev_logits, lib.gen_dev_hidden, lib.gen_dev_wgate):
            f.restype = ctypes.c_int
        _dev = lib
    return _dev


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ------------------------------------------------------------------ host twin
def host_logits(wl, tok_key, tok_dom) -> np.ndarray:
    """Logits [L][T][E] float32 of the given tokens of workload `wl`."""
    tok_key, tok_dom = _c(tok_key, np.int64), _c(tok_dom, np.int32)
    T = tok_key.shape[0]
    out = np.empty((wl.L, T, wl.E), dtype=np.float32)
    bm = _c(wl.bias_mask, np.uint8)
    _host_lib().gen_host_logits(wl.seed, _p(tok_key), _p(tok_dom), T, wl.L, wl.E,
                                _p(bm), wl.ndom, wl.bias, _p(out))
    return out


def host_logit_rows(wl, tok_key, tok_dom, layers, toks) -> np.ndarray:
    """Rows (layers[n], toks[n]) of the logits, [n][E] float32."""
    tok_key, tok_dom = _c(tok_key, np.int64), _c(tok_dom, np.int32)
    layers, toks = _c(layers, np.int32), _c(toks, np.int64)
    out = np.empty((layers.shape[0], wl.E), dtype=np.float32)
    bm = _c(wl.bias_mask, np.uint8)
    _host_lib().gen_host_logit_rows(wl.seed, _p(tok_key), _p(tok_dom), _p(layers), _p(toks),
                                    layers.shape[0], wl.L, wl.E, _p(bm), wl.ndom, wl.bias,
                                    _p(out))
    return out


def host_hidden(seed: int, t0: int, nt: int, H: int) -> np.ndarray:
    """Rows [t0, t0+nt) of the hidden states as bf16 bit patterns (uint16)."""
    out = np.empty((nt, H), dtype=np.uint16)
    _host_lib().gen_host_hidden(seed, t0, nt, H, _p(out))
    return out


def host_wgate(seed: int, L: int, H: int, E: int, scale: float) -> np.ndarray:
    out = np.empty((L, H, E), dtype=np.uint16)
    _host_lib().gen_host_wgate(seed, L, H, E, scale, _p(out))
    return out


# ------------------------------------------------------------- device filler
def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with cudaError {rc}")


def dev_logits(wl, tok_key_dev, tok_dom_dev, out_dev, bias_mask_dev, stream=0) -> None:
    """Fill a [L][T][E] float32 device tensor (torch) with the workload's logits."""
    T = tok_key_dev.shape[0]
    _check(_dev_lib().gen_dev_logits(wl.seed, tok_key_dev.data_ptr(), tok_dom_dev.data_ptr(),
                                     T, wl.L, wl.E, bias_mask_dev.data_ptr(), wl.ndom,
                                     wl.bias, out_dev.data_ptr(), stream), "gen_dev_logits")


def dev_hidden(seed: int, T: int, H: int, out_dev, stream=0) -> None:
    _check(_dev_lib().gen_dev_hidden(seed, T, H, out_dev.data_ptr(), stream), "gen_dev_hidden")


def dev_wgate(seed: int, L: int, H: int, E: int, scale: float, out_dev, stream=0) -> None:
    _check(_dev_lib().gen_dev_wgate(seed, L, H, E, scale, out_dev.data_ptr(), stream),
           "gen_dev_wgate")
