"""fp64 CPU oracle for the speculative-decoding verification step and the
steps around it (draft-row sampling, KV commit on a sink + ring cache, the
draft KV window's block table) and of token-tree verification.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline leg
of the benchmark may import this package; the product path never does.  It
shares no code with the CUDA library: the arithmetic lives in sv_oracle.c and
kv_oracle.c (plain loops, the definitions written out), loaded here through
ctypes.

Parity status: every function below is pinned by tests/test_oracle_pins.py
(worked example and NumPy-operator vectors of the Speculative Decoding overview
page, losslessness chi-square, the expected-tokens closed form, brute force at
tiny V, textbook softmax and argmax; for the draft side a u-grid brute force,
the ln p closed form and losslessness of draft sampling followed by
verification; for the KV steps the slot formula's permutation property, the
cache content against a plain sink + sliding-window model, and the draft
window page's unit-test example with the clone's gather invariant; for token
trees the reduction of a chain to the pinned chain rule, the single-node
inverse CDF, multi-draft losslessness and the never-re-accepted rejected
token), and
tests/test_oracle_mutants.py shows that planted mistakes fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "sv_oracle.c"), os.path.join(_HERE, "kv_oracle.c")]
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
KV_INVALID = 1  # kv_oracle.c: a request the KV steps reject


def compile_oracle(out_path: str | None = None, mutant: int = 0) -> str:
    """Compile sv_oracle.c and kv_oracle.c with gcc into one shared library;
    returns its path.
    -ffp-contract=off keeps fp64 rounding identical on x86 and Arm."""
    if out_path is None:
        out_path = os.path.join(_BUILD, "libsvoracle.so" if mutant == 0
                                else f"libsvoracle_m{mutant}.so")
    os.makedirs(os.path.dirname(os.path.abspath(out_path)), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           f"-DSVO_MUTANT={int(mutant)}", *_SRCS, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


_LIBS: dict[str, ctypes.CDLL] = {}


def load(path: str | None = None) -> ctypes.CDLL:
    if path is None:
        path = os.path.join(_BUILD, "libsvoracle.so")
        if not os.path.exists(path) or os.path.getmtime(path) < max(
                os.path.getmtime(f) for f in _SRCS):
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
        lib.svo_draft_sample.argtypes = [I, P, P, P, I, I, I, P, P, P, P, P, ctypes.c_double, I]
        lib.svo_draft_sample.restype = I
        lib.svo_tree_verify.argtypes = [I, P, P, P, P, P, P, P, I, I, I, P, P, P, P,
                                        ctypes.c_double, I]
        lib.svo_tree_verify.restype = I
        lib.kvo_slot_of.argtypes = [ctypes.c_int64, I, I]
        lib.kvo_slot_of.restype = ctypes.c_int64
        lib.kvo_commit.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
        lib.kvo_commit.restype = I
        lib.kvo_valid_slots.argtypes = [P, I, I, I, P, P]
        lib.kvo_valid_slots.restype = I
        lib.kvo_window_block_table.argtypes = [P, P, I, I, I, I, I, I, P, P, P, P, P]
        lib.kvo_window_block_table.restype = I
        lib.kvo_window_cols.argtypes = [I, I]
        lib.kvo_window_cols.restype = I
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


def draft_sample(L, u, temp, dtype: int, near_eps: float = NEAR_EPS,
                 nthreads: int | None = None, lib: ctypes.CDLL | None = None) -> dict:
    """Draft-row sampling oracle.  L [B][n][V] (float32, or uint16 bf16 bits),
    u [B][n], temp [B].  Returns tokens, m, S, dist, flags, each [B][n]."""
    lib = lib or load()
    L = np.ascontiguousarray(L)
    B, n, V = L.shape
    u = np.ascontiguousarray(u, dtype=np.float32).reshape(B, n)
    temp = np.ascontiguousarray(temp, dtype=np.float32).reshape(B)
    out = dict(tokens=np.empty((B, n), np.int32), m=np.empty((B, n), np.float64),
               S=np.empty((B, n), np.float64), dist=np.empty((B, n), np.float64),
               flags=np.zeros((B, n), np.int32))
    rc = lib.svo_draft_sample(int(dtype), _ptr(L), _ptr(u), _ptr(temp), B, n, V,
                              _ptr(out["tokens"]), _ptr(out["m"]), _ptr(out["S"]),
                              _ptr(out["dist"]), _ptr(out["flags"]), float(near_eps),
                              _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"svo_draft_sample failed with {rc}")
    return out


TREE_MAX_N = 256  # sv_oracle.c: nodes per token tree


def tree_verify(Lt, Ld, parent, tokens, u_acc, u_res, temp, dtype: int,
                near_eps: float = NEAR_EPS, nthreads: int | None = None,
                lib: ctypes.CDLL | None = None) -> dict:
    """Token-tree verification oracle (readings T1-T3 of sv_oracle.c).
    Lt, Ld [B][N][V] (float32, or uint16 bf16 bits); parent, tokens [B][N]
    int32; u_acc, u_res [B][N]; temp [B].  Returns tokens [B][N], n [B],
    nodes [B][N] and flags [B]."""
    lib = lib or load()
    Lt, Ld = np.ascontiguousarray(Lt), np.ascontiguousarray(Ld)
    B, N, V = Lt.shape
    assert Ld.shape == Lt.shape and Ld.dtype == Lt.dtype
    arr = [np.ascontiguousarray(a, dtype=t).reshape(B, N) for a, t in
           ((parent, np.int32), (tokens, np.int32), (u_acc, np.float32), (u_res, np.float32))]
    temp = np.ascontiguousarray(temp, dtype=np.float32).reshape(B)
    out = dict(tokens=np.empty((B, N), np.int32), n=np.empty(B, np.int32),
               nodes=np.empty((B, N), np.int32), flags=np.zeros(B, np.int32))
    rc = lib.svo_tree_verify(int(dtype), _ptr(Lt), _ptr(Ld), *(_ptr(a) for a in arr), _ptr(temp),
                             B, N, V, _ptr(out["tokens"]), _ptr(out["n"]), _ptr(out["nodes"]),
                             _ptr(out["flags"]), float(near_eps), _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"svo_tree_verify failed with {rc}")
    return out


def kv_slot(pos: int, sink: int, window: int, lib: ctypes.CDLL | None = None) -> int:
    """Slot(pos) of the sink + ring cache."""
    return int((lib or load()).kvo_slot_of(int(pos), int(sink), int(window)))


def kv_commit(k_pool, v_pool, k_new, v_new, num_accepted, pos, sink: int, window: int,
              lib: ctypes.CDLL | None = None) -> dict:
    """KV commit oracle, in place on copies: pools [B][LH][sink+window][row]
    and staged entries [B][LH][R][row] of any fixed-size element type (the
    copy is bytewise).  Returns the new pools, pos and flags."""
    lib = lib or load()
    kp = np.array(k_pool, copy=True, order="C")
    vp = np.array(v_pool, copy=True, order="C")
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    B, LH, C = kp.shape[:3]
    R = kn.shape[2]
    row_bytes = kp[0, 0, 0].nbytes if kp.size else 0
    assert C == sink + window and kn.shape[:2] == (B, LH) and vn.shape == kn.shape
    na = np.ascontiguousarray(num_accepted, dtype=np.int32).reshape(B)
    p = np.array(pos, dtype=np.int32, copy=True).reshape(B)
    flags = np.zeros(B, np.int32)
    rc = lib.kvo_commit(_ptr(kp), _ptr(vp), _ptr(kn), _ptr(vn), _ptr(na), _ptr(p), B, LH, R,
                        row_bytes, sink, window, _ptr(flags))
    if rc != 0:
        raise RuntimeError(f"kvo_commit failed with {rc}")
    return dict(k_pool=kp, v_pool=vp, pos=p, flags=flags)


def kv_valid_slots(pos, sink: int, window: int, lib: ctypes.CDLL | None = None) -> dict:
    """Valid physical slots of every request in logical order: slots
    [B][sink+window] (-1 padded) and len [B]."""
    lib = lib or load()
    p = np.ascontiguousarray(pos, dtype=np.int32).reshape(-1)
    B = p.shape[0]
    out = dict(slots=np.empty((B, sink + window), np.int32), len=np.empty(B, np.int32))
    rc = lib.kvo_valid_slots(_ptr(p), B, sink, window, _ptr(out["slots"]), _ptr(out["len"]))
    if rc != 0:
        raise RuntimeError(f"kvo_valid_slots failed with {rc}")
    return out


def window_block_table(seq_lens, table, W: int, blk: int, K: int,
                       lib: ctypes.CDLL | None = None) -> dict:
    """Draft KV window oracle: windowed seq_lens [B], the block-table clone
    [B][max(W // blk + 1, ceil((W + blk - 1) / blk))], start_block [B],
    needed [B], flags [B]."""
    lib = lib or load()
    s = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(-1)
    t = np.ascontiguousarray(table, dtype=np.int32)
    B, full_cols = t.shape
    mc = int(lib.kvo_window_cols(W, blk))
    out = dict(seq=np.empty(B, np.int32), table=np.empty((B, mc), np.int32),
               start_block=np.empty(B, np.int32), needed=np.empty(B, np.int32),
               flags=np.zeros(B, np.int32))
    rc = lib.kvo_window_block_table(_ptr(s), _ptr(t), B, full_cols, W, blk, K, mc,
                                    _ptr(out["seq"]), _ptr(out["table"]),
                                    _ptr(out["start_block"]), _ptr(out["needed"]),
                                    _ptr(out["flags"]))
    if rc != 0:
        raise RuntimeError(f"kvo_window_block_table failed with {rc}")
    return out
