"""Seeded synthetic inputs for the verification step.

This module only draws random numbers and rounds them to the stored dtype;
it holds none of the verification arithmetic (no acceptance test, no
residual, no inverse CDF).  Both the CUDA path and the CPU oracle consume
exactly the arrays it returns, so the stored (rounded) values are the inputs
of both sides.

Workloads follow the shapes the pages work with: LLM vocabularies of 32000,
50257, 128256 and 151936 entries, gamma = 3..7 draft positions.  The five
named workloads:

  c1  B=1,    gamma=4, V=32000,  fp32  target N(0,2^2), draft = target + N(0,0.5^2), T=1
  c2  B=64,   gamma=5, V=32000,  bf16  greedy: target N(0,3^2), draft = target + N(0,1),
                                       draft tokens = draft argmax
  c3  B=32,   gamma=7, V=128256, bf16  Zipf-shaped rows, draft correlated rho=0.9, T=0.8
  c4  B=256,  gamma=4, V=151936, bf16  target N(0,2.5^2); draft = log of a w-mixture of the
                                       target softmax and an independent one,
                                       w = 0.3 / 0.6 / 0.9 per third of the batch, T=1
  c5  B=1024, gamma=3, V=50257,  fp32  target N(0,2^2), draft = target + N(0,0.7^2),
                                       per-request T ~ U(0.5, 1.5)

Every random stream is a Philox generator keyed by (seed, input set, stream
tag, request, position), so rows can be drawn in parallel and any row can be
regenerated alone.  Draft tokens are drawn from the stored draft logits at the
request's temperature with the Gumbel-max trick (a sampling device of the
draft side, not part of verification).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

F32, BF16 = 0, 1
DTYPE_CODE = {"f32": F32, "bf16": BF16}
ELEM_BYTES = {F32: 4, BF16: 2}

CONFIGS = {
    1: dict(name="c1_B1_g4_V32000_f32", B=1, gamma=4, V=32000, dtype="f32",
            kind="normal", sigma_t=2.0, sigma_noise=0.5, temp=1.0),
    2: dict(name="c2_greedy_B64_g5_V32000_bf16", B=64, gamma=5, V=32000, dtype="bf16",
            kind="greedy", sigma_t=3.0, sigma_noise=1.0, temp=0.0),
    3: dict(name="c3_zipf_B32_g7_V128256_bf16", B=32, gamma=7, V=128256, dtype="bf16",
            kind="zipf", zipf_s=1.1, zipf_noise=0.3, rho=0.9, temp=0.8),
    4: dict(name="c4_mix_B256_g4_V151936_bf16", B=256, gamma=4, V=151936, dtype="bf16",
            kind="mix", sigma=2.5, weights=(0.3, 0.6, 0.9), temp=1.0),
    5: dict(name="c5_B1024_g3_V50257_f32", B=1024, gamma=3, V=50257, dtype="f32",
            kind="normal", sigma_t=2.0, sigma_noise=0.7, temp=("uniform", 0.5, 1.5)),
}
BASE_SEED = 20260

_TAG_TARGET, _TAG_DRAFT, _TAG_AUX, _TAG_TOKEN, _TAG_UNIFORM, _TAG_TEMP = range(6)
_TAG_DRAFT_UNIFORM, _TAG_KV = 6, 7


@dataclasses.dataclass
class Inputs:
    """One batch of verification inputs, host-resident.

    Lt  [B][gamma+1][V]  target logits (float32, or uint16 holding bf16 bits)
    Ld  [B][gamma][V]    draft logits, same dtype
    x   [B][gamma]       int32 draft tokens
    u_acc [B][gamma]     float32 uniforms in [0, 1) for the accept tests
    u_res [B][gamma+1]   float32 uniforms in [0, 1) for the resample / bonus
    temp  [B]            float32 temperature (0 for the greedy workload)
    """
    Lt: np.ndarray
    Ld: np.ndarray
    x: np.ndarray
    u_acc: np.ndarray
    u_res: np.ndarray
    temp: np.ndarray
    dtype: int
    B: int
    gamma: int
    V: int
    name: str = "custom"

    @property
    def logit_bytes(self) -> int:
        return (self.Lt.size + self.Ld.size) * ELEM_BYTES[self.dtype]


def rng_for(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, *tags])))


def round_to_dtype(a64: np.ndarray, dtype: int) -> np.ndarray:
    """fp64 -> stored dtype.  bf16 is rounded to nearest-even from the fp32
    value and returned as its raw 16-bit pattern."""
    f32 = np.asarray(a64, dtype=np.float32)
    if dtype == F32:
        return f32
    bits = f32.view(np.uint32).astype(np.uint64)
    bits = bits + 0x7FFF + ((bits >> 16) & 1)
    return (bits >> 16).astype(np.uint16)


def widen(stored: np.ndarray, dtype: int) -> np.ndarray:
    """Stored values -> fp64, exactly."""
    if dtype == F32:
        return stored.astype(np.float64)
    return (stored.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _zipf_row(rng: np.random.Generator, V: int, s: float, noise: float) -> np.ndarray:
    ranks = np.arange(V, dtype=np.float64)
    prof = -s * np.log(ranks + 1.0) + noise * rng.standard_normal(V)
    row = np.empty(V, dtype=np.float64)
    row[rng.permutation(V)] = prof
    return row


def _gumbel_argmax(rng: np.random.Generator, logits64: np.ndarray, T: float) -> int:
    return int(np.argmax(logits64 / T + rng.gumbel(size=logits64.shape[0])))


def _target_row(cfg: dict, rt: np.random.Generator, V: int) -> np.ndarray:
    kind = cfg["kind"]
    if kind in ("normal", "greedy"):
        return cfg["sigma_t"] * rt.standard_normal(V)
    if kind == "zipf":
        return _zipf_row(rt, V, cfg["zipf_s"], cfg["zipf_noise"])
    if kind == "mix":
        return cfg["sigma"] * rt.standard_normal(V)
    raise ValueError(kind)


def _draft_row(cfg: dict, rd: np.random.Generator, lt: np.ndarray, b: int, B: int) -> np.ndarray:
    kind, V = cfg["kind"], lt.shape[0]
    if kind in ("normal", "greedy"):
        return lt + cfg["sigma_noise"] * rd.standard_normal(V)
    if kind == "zipf":
        rho = cfg["rho"]
        return rho * lt + np.sqrt(1.0 - rho * rho) * _zipf_row(rd, V, cfg["zipf_s"],
                                                               cfg["zipf_noise"])
    # mix: draft distribution = w * softmax(target) + (1-w) * softmax(Q)
    from scipy.special import log_softmax
    w = cfg["weights"][min(len(cfg["weights"]) - 1, (len(cfg["weights"]) * b) // B)]
    q = cfg["sigma"] * rd.standard_normal(V)
    ld = np.logaddexp(np.log(w) + log_softmax(lt), np.log1p(-w) + log_softmax(q))
    return ld - ld.max()  # shift so the stored bf16 values keep their precision


def _draw_request(cfg: dict, seed: int, set_index: int, b: int, B: int, gamma: int, V: int,
                  dtype: int, T: float, Lt: np.ndarray, Ld: np.ndarray, x: np.ndarray) -> None:
    kind = cfg["kind"]
    for i in range(gamma + 1):
        lt = _target_row(cfg, rng_for(seed, set_index, _TAG_TARGET, b, i), V)
        Lt[b, i] = round_to_dtype(lt, dtype)
        if i == gamma:
            break
        ld = _draft_row(cfg, rng_for(seed, set_index, _TAG_DRAFT, b, i), lt, b, B)
        Ld[b, i] = round_to_dtype(ld, dtype)
        rx = rng_for(seed, set_index, _TAG_TOKEN, b, i)
        ld_stored = widen(Ld[b, i], dtype)
        if kind == "greedy":
            x[b, i] = int(np.argmax(ld_stored))
        else:
            x[b, i] = _gumbel_argmax(rx, ld_stored, T)


def make_inputs(cfg: dict | int, seed: int | None = None, set_index: int = 0,
                B: int | None = None, threads: int | None = None) -> Inputs:
    """Draw one batch of the given workload (a CONFIGS id or a dict with the
    same keys).  `B` overrides the batch size; the first B' requests of a
    batch are identical whatever B' is (rows are keyed by request index)."""
    if isinstance(cfg, int):
        cid = cfg
        cfg = CONFIGS[cfg]
        if seed is None:
            seed = BASE_SEED + cid
    if seed is None:
        seed = BASE_SEED
    B = cfg["B"] if B is None else B
    gamma, V = cfg["gamma"], cfg["V"]
    dtype = DTYPE_CODE[cfg["dtype"]] if isinstance(cfg["dtype"], str) else cfg["dtype"]
    st = np.float32 if dtype == F32 else np.uint16
    Lt = np.empty((B, gamma + 1, V), dtype=st)
    Ld = np.empty((B, gamma, V), dtype=st)
    x = np.empty((B, gamma), dtype=np.int32)
    ru = rng_for(seed, set_index, _TAG_UNIFORM)
    u_acc = ru.random((B, gamma), dtype=np.float32)
    u_res = ru.random((B, gamma + 1), dtype=np.float32)
    tcfg = cfg.get("temp", 1.0)
    if isinstance(tcfg, tuple):
        _, lo, hi = tcfg
        temp = rng_for(seed, set_index, _TAG_TEMP).uniform(lo, hi, B).astype(np.float32)
    else:
        temp = np.full(B, tcfg, dtype=np.float32)
    # the greedy workload samples nothing; its draft tokens are the draft argmax
    Tsample = [float(t) if t > 0 else 1.0 for t in temp]
    threads = threads or min(32, os.cpu_count() or 1)
    with np.errstate(divide="ignore", over="ignore"):
        if threads > 1 and B > 1:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(lambda b: _draw_request(cfg, seed, set_index, b, B, gamma, V, dtype,
                                                    Tsample[b], Lt, Ld, x), range(B)))
        else:
            for b in range(B):
                _draw_request(cfg, seed, set_index, b, B, gamma, V, dtype, Tsample[b], Lt, Ld, x)
    return Inputs(Lt, Ld, x, u_acc, u_res, temp, dtype, B, gamma, V, cfg.get("name", "custom"))


def custom_config(B: int, gamma: int, V: int, dtype: str = "bf16", kind: str = "normal",
                  temp=1.0, **kw) -> dict:
    """A workload dict with the given shape, for parity sweeps."""
    d = dict(name=f"custom_{kind}_B{B}_g{gamma}_V{V}_{dtype}", B=B, gamma=gamma, V=V,
             dtype=dtype, kind=kind, temp=temp)
    defaults = {"normal": dict(sigma_t=2.0, sigma_noise=0.5),
                "greedy": dict(sigma_t=3.0, sigma_noise=1.0),
                "zipf": dict(zipf_s=1.1, zipf_noise=0.3, rho=0.9),
                "mix": dict(sigma=2.5, weights=(0.3, 0.6, 0.9))}[kind]
    d.update(defaults)
    d.update(kw)
    return d


def draft_uniforms(B: int, n: int, seed: int, set_index: int = 0) -> np.ndarray:
    """u_draft [B][n]: fp32 uniforms in [0, 1) for sampling the draft rows."""
    return rng_for(seed, set_index, _TAG_DRAFT_UNIFORM).random((B, n), dtype=np.float32)


# ---------------------------------------------------------------- token trees

_TAG_TREE_TARGET, _TAG_TREE_DRAFT, _TAG_TREE_TOKEN, _TAG_TREE_UNIFORM, _TAG_TREE_SHAPE = (
    8, 9, 10, 11, 12)

# the token-tree workload: 64 requests, a tree with 3 root children, 2 below
# each of them, then two single-child levels (22 nodes, depth 4), the c4
# vocabulary and row model
TREE_WORKLOAD = dict(name="tree_b3211_B64_N22_V151936_bf16", B=64, branching=(3, 2, 1, 1),
                     V=151936, dtype="bf16", kind="mix", sigma=2.5, weights=(0.3, 0.6, 0.9),
                     temp=1.0)


def tree_parents(branching) -> np.ndarray:
    """Parent array (node order: level by level) of a tree whose nodes at
    depth d have branching[d] children each; the root's parent is -1."""
    parent, level = [-1], [0]
    for k in branching:
        nxt = []
        for p in level:
            for _ in range(k):
                parent.append(p)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.array(parent, np.int32)


def random_parents(N: int, seed: int, max_children: int = 4) -> np.ndarray:
    """A random tree on N nodes with parent[n] < n and at most max_children
    children per node."""
    rng = rng_for(seed, _TAG_TREE_SHAPE)
    parent = np.full(N, -1, np.int32)
    kids = np.zeros(N, np.int64)
    for n in range(1, N):
        while True:
            p = int(rng.integers(max(0, n - 8), n))
            if kids[p] < max_children:
                break
        parent[n] = p
        kids[p] += 1
    return parent


@dataclasses.dataclass
class TreeInputs:
    """One batch of token-tree verification inputs, host-resident.

    Lt, Ld [B][N][V]  target / draft logits (float32, or uint16 bf16 bits);
                      the draft rows of leaves are never read (filled with
                      `leaf_fill`)
    parent [B][N], tokens [B][N]  int32 (tokens[b][0] = 0, unused)
    u_acc, u_res [B][N]  float32 uniforms in [0, 1)
    temp [B]          float32
    """
    Lt: np.ndarray
    Ld: np.ndarray
    parent: np.ndarray
    tokens: np.ndarray
    u_acc: np.ndarray
    u_res: np.ndarray
    temp: np.ndarray
    dtype: int
    B: int
    N: int
    V: int
    name: str = "tree"

    def visited_bytes_bound(self) -> int:
        return (self.Lt.size + self.Ld.size) * ELEM_BYTES[self.dtype]


def _draw_tree_request(cfg, seed, set_index, b, B, parent, V, dtype, T, leaf_fill, Lt, Ld, tok):
    N = parent.shape[0]
    has_child = np.zeros(N, bool)
    has_child[parent[1:]] = True
    for n in range(N):
        lt = _target_row(cfg, rng_for(seed, set_index, _TAG_TREE_TARGET, b, n), V)
        Lt[b, n] = round_to_dtype(lt, dtype)
        if has_child[n]:
            ld = _draft_row(cfg, rng_for(seed, set_index, _TAG_TREE_DRAFT, b, n), lt, b, B)
            Ld[b, n] = round_to_dtype(ld, dtype)
        else:
            Ld[b, n] = round_to_dtype(np.full(V, leaf_fill), dtype)
    # every child's token is drawn from its parent's stored draft row
    # (Gumbel-max at the request's temperature), independently per sibling
    for n in range(1, N):
        rx = rng_for(seed, set_index, _TAG_TREE_TOKEN, b, n)
        tok[b, n] = _gumbel_argmax(rx, widen(Ld[b, parent[n]], dtype), T)


def make_tree_inputs(cfg: dict, parent, seed: int = BASE_SEED, set_index: int = 0,
                     B: int | None = None, leaf_fill: float = 0.0,
                     threads: int | None = None) -> TreeInputs:
    """Draw one batch of token-tree inputs: `cfg` a row model (the keys of
    custom_config or TREE_WORKLOAD), `parent` one parent array [N] shared by
    all requests or one per request [B][N]."""
    B = cfg["B"] if B is None else B
    V = cfg["V"]
    dtype = DTYPE_CODE[cfg["dtype"]] if isinstance(cfg["dtype"], str) else cfg["dtype"]
    parent = np.asarray(parent, np.int32)
    if parent.ndim == 1:
        parent = np.broadcast_to(parent, (B, parent.shape[0]))
    parent = np.ascontiguousarray(parent)
    N = parent.shape[1]
    st = np.float32 if dtype == F32 else np.uint16
    Lt = np.empty((B, N, V), dtype=st)
    Ld = np.empty((B, N, V), dtype=st)
    tok = np.zeros((B, N), dtype=np.int32)
    ru = rng_for(seed, set_index, _TAG_TREE_UNIFORM)
    u_acc = ru.random((B, N), dtype=np.float32)
    u_res = ru.random((B, N), dtype=np.float32)
    tcfg = cfg.get("temp", 1.0)
    if isinstance(tcfg, tuple):
        _, lo, hi = tcfg
        temp = rng_for(seed, set_index, _TAG_TEMP).uniform(lo, hi, B).astype(np.float32)
    else:
        temp = np.full(B, tcfg, dtype=np.float32)
    threads = threads or min(32, os.cpu_count() or 1)

    def one(b):
        _draw_tree_request(cfg, seed, set_index, b, B, parent[b], V, dtype, float(temp[b]),
                           leaf_fill, Lt, Ld, tok)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        if threads > 1 and B > 1:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(one, range(B)))
        else:
            for b in range(B):
                one(b)
    return TreeInputs(Lt, Ld, parent, tok, u_acc, u_res, temp, dtype, B, N, V,
                      cfg.get("name", "tree"))
