"""fp64 CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline leg
of the benchmark may import this package; the product path never does.  It
shares no code with the CUDA library: the arithmetic lives in sv_oracle.c
(plain fp64 loops, the definition written out), loaded here through ctypes.

Parity status: every function below is pinned by tests/test_oracle_pins.py
(worked example and NumPy-operator vectors of the Speculative Decoding overview
page, losslessness chi-square, the expected-tokens closed form, brute force at
tiny V, textbook softmax and argmax), and tests/test_oracle_mutants.py shows
that planted mistakes fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

# per-request flag bits (mirror the SVO_* defines in sv_oracle.c)
INVALID_NONFINITE = 1
INVALID_TOKEN = 2
INVALID_TEMP = 4
INVALID_ANY = INVALID_NONFINITE | INVALID_TOKEN | INVALID_TEMP
NEAR_ACCEPT = 16
NEAR_SAMPLE = 32
DEGENERATE = 64
NEAR_ANY = NEAR_ACCEPT | NEAR_SAMPLE | DEGENERATE

NEAR_EPS = 1e-6


def compile_oracle(out_path: str | None = None, mutant: int = 0) -> str:
    """Compile sv_oracle.c with gcc into a shared library; returns its path.
    -ffp-contract=off keeps fp64 rounding identical on x86 and Arm."""
    if out_path is None:
        out_path = os.path.join(_BUILD, "libsvoracle.so" if mutant == 0
                                else f"libsvoracle_m{mutant}.so")
    os.makedirs(os.path.dirname(os.path.abspath(out_path)), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           f"-DSVO_MUTANT={int(mutant)}", _SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


_LIBS: dict[str, ctypes.CDLL] = {}


def load(path: str | None = None) -> ctypes.CDLL:
    if path is None:
        path = os.path.join(_BUILD, "libsvoracle.so")
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            compile_oracle(path)
    if path not in _LIBS:
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.svo_verify.argtypes = [I, P, P, P, P, P, P, I, I, I, P, P, P, P, P, P, P,
                                   ctypes.c_double, I]
        lib.svo_verify.restype = I
        lib.svo_greedy.argtypes = [I, P, P, I, I, I, P, P, P, P, I]
        lib.svo_greedy.restype = I
        lib.svo_mutant_id.restype = I
        _LIBS[path] = lib
    return _LIBS[path]


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(nthreads):
    return nthreads if nthreads else (os.cpu_count() or 1)


def verify(Lt, Ld, x, u_acc, u_res, temp, dtype: int, near_eps: float = NEAR_EPS,
           nthreads: int | None = None, lib: ctypes.CDLL | None = None) -> dict:
    """Sampling-path oracle.  Arrays as in synth.Inputs (C-contiguous).
    Returns tokens [B][gamma+1], n [B], pt/pd [B][gamma], Z [B], flags [B] and
    dist [B][2] (distance of u_acc to the nearest decided ratio, and of
    u_resample to the emitted token's nearer CDF edge)."""
    lib = lib or load()
    Lt = np.ascontiguousarray(Lt)
    B, R, V = Lt.shape
    g = R - 1
    Ld = np.ascontiguousarray(Ld) if g > 0 else np.zeros((B, 0, V), Lt.dtype)
    x = np.ascontiguousarray(x, dtype=np.int32).reshape(B, g)
    u_acc = np.ascontiguousarray(u_acc, dtype=np.float32).reshape(B, g)
    u_res = np.ascontiguousarray(u_res, dtype=np.float32).reshape(B, R)
    temp = np.ascontiguousarray(temp, dtype=np.float32).reshape(B)
    out = dict(tokens=np.empty((B, R), np.int32), n=np.empty(B, np.int32),
               pt=np.empty((B, g), np.float64), pd=np.empty((B, g), np.float64),
               Z=np.empty(B, np.float64), dist=np.empty((B, 2), np.float64),
               flags=np.zeros(B, np.int32))
    rc = lib.svo_verify(int(dtype), _ptr(Lt), _ptr(Ld), _ptr(x), _ptr(u_acc), _ptr(u_res),
                        _ptr(temp), B, g, V, _ptr(out["tokens"]), _ptr(out["n"]),
                        _ptr(out["pt"]), _ptr(out["pd"]), _ptr(out["Z"]), _ptr(out["dist"]),
                        _ptr(out["flags"]),
                        float(near_eps), _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"svo_verify failed with {rc}")
    return out


def greedy(Lt, x, dtype: int, nthreads: int | None = None,
           lib: ctypes.CDLL | None = None) -> dict:
    """Greedy-path oracle.  Returns tokens [B][gamma+1], n [B],
    argmax [B][gamma+1], flags [B]."""
    lib = lib or load()
    Lt = np.ascontiguousarray(Lt)
    B, R, V = Lt.shape
    g = R - 1
    x = np.ascontiguousarray(x, dtype=np.int32).reshape(B, g)
    out = dict(tokens=np.empty((B, R), np.int32), n=np.empty(B, np.int32),
               argmax=np.full((B, R), -1, np.int32), flags=np.zeros(B, np.int32))
    rc = lib.svo_greedy(int(dtype), _ptr(Lt), _ptr(x), B, g, V, _ptr(out["tokens"]),
                        _ptr(out["n"]), _ptr(out["argmax"]), _ptr(out["flags"]),
                        _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"svo_greedy failed with {rc}")
    return out
