"""The C-ABI library on the host (no GPU needed): it loads, exports every
function include/specverify.h declares, sizes workspaces, and rejects bad
arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from speculative_decoding_verification_09_gb300 import binding
from speculative_decoding_verification_09_gb300._build_lib import ROOT

HEADERS = [os.path.join(ROOT, "include", f) for f in ("specverify.h", "svkv.h", "svtree.h")]


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()  # rebuilds only what is out of date
    return binding.lib()


def header_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*"
                                 r"([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


def test_header_symbols_exported(L):
    names = header_functions()
    assert set(names) == set(binding.EXPORTED), names
    for n in names:
        assert hasattr(L, n), n


def test_workspace_bytes(L):
    a = binding.sv_workspace_bytes(1, 4, 32000)
    b = binding.sv_workspace_bytes(256, 4, 151936)
    assert 0 < a < b and b % 256 == 0
    assert binding.sv_workspace_bytes(-1, 4, 10) == 0
    assert binding.sv_workspace_bytes(1, 33, 10) == 0
    assert binding.sv_workspace_bytes(1, 4, 0) == 0
    assert L.sv_version() >= 100
    assert L.sv_error_string(binding.SV_ERR_WORKSPACE) == b"SV_ERR_WORKSPACE"


FAKE = 0x10000000  # never dereferenced: every call below fails validation first


def _call(L, **kw):
    a = dict(Lt=FAKE, Ld=FAKE, x=FAKE, ua=FAKE, ur=FAKE, T=FAKE, B=2, g=3, V=100, dt=0,
             tok=FAKE, n=FAKE, p=None, Z=None, ws=FAKE, wsb=1 << 30, st=None, s=None)
    a.update(kw)
    return L.spec_verify_diag(a["Lt"], a["Ld"], a["x"], a["ua"], a["ur"], a["T"], a["B"], a["g"],
                              a["V"], a["dt"], a["tok"], a["n"], a["p"], a["Z"], a["ws"],
                              a["wsb"], a["st"], a["s"])


def test_argument_validation(L):
    assert _call(L, dt=7) == binding.SV_ERR_DTYPE
    assert _call(L, g=33) == binding.SV_ERR_INVALID_ARG
    assert _call(L, g=-1) == binding.SV_ERR_INVALID_ARG
    assert _call(L, B=-1) == binding.SV_ERR_INVALID_ARG
    assert _call(L, V=0) == binding.SV_ERR_INVALID_ARG
    assert _call(L, Lt=None) == binding.SV_ERR_INVALID_ARG
    assert _call(L, Ld=None) == binding.SV_ERR_INVALID_ARG
    assert _call(L, ur=None) == binding.SV_ERR_INVALID_ARG
    assert _call(L, tok=None) == binding.SV_ERR_INVALID_ARG
    assert _call(L, Lt=FAKE + 2) == binding.SV_ERR_INVALID_ARG   # fp32 logits need 4-byte alignment
    assert _call(L, x=FAKE + 1) == binding.SV_ERR_INVALID_ARG
    assert _call(L, ws=FAKE + 16) == binding.SV_ERR_WORKSPACE    # workspace needs 256-byte alignment
    assert _call(L, ws=None) == binding.SV_ERR_WORKSPACE
    assert _call(L, wsb=64) == binding.SV_ERR_WORKSPACE
    assert _call(L, B=0) == binding.SV_OK                        # empty batch: nothing launched
    # gamma = 0 needs no draft pointers; it still validates the rest
    assert _call(L, g=0, Ld=None, x=None, ua=None, wsb=64) == binding.SV_ERR_WORKSPACE
    assert L.spec_verify_greedy(FAKE, FAKE, 2, 3, 100, 5, FAKE, FAKE, FAKE, 1 << 30, None,
                                None) == binding.SV_ERR_DTYPE
    assert L.spec_verify_greedy(FAKE, None, 2, 3, 100, 1, FAKE, FAKE, FAKE, 1 << 30, None,
                                None) == binding.SV_ERR_INVALID_ARG
    assert L.spec_verify_greedy(FAKE + 1, FAKE, 2, 3, 100, 1, FAKE, FAKE, FAKE, 1 << 30, None,
                                None) == binding.SV_ERR_INVALID_ARG


def test_no_gpu_fails_loudly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid-looking arguments reach the device query, which must fail, not fall back
    assert _call(L) == binding.SV_ERR_CUDA


def test_stage_events_validation(L):
    arr = (ctypes.c_void_p * 6)(*([FAKE] * 6))
    assert L.sv_set_stage_events(arr, 6) == binding.SV_ERR_INVALID_ARG   # at most five
    assert L.sv_set_stage_events(arr, -1) == binding.SV_ERR_INVALID_ARG
    assert L.sv_set_stage_events(None, 2) == binding.SV_ERR_INVALID_ARG
    nul = (ctypes.c_void_p * 2)(FAKE, None)
    assert L.sv_set_stage_events(nul, 2) == binding.SV_ERR_INVALID_ARG   # a NULL handle
    assert L.sv_set_stage_events(None, 0) == binding.SV_OK               # off


def test_tail_selection_validation(L):
    assert L.sv_set_tail(4) == binding.SV_ERR_INVALID_ARG
    assert L.sv_set_tail(-1) == binding.SV_ERR_INVALID_ARG
    for mode in (1, 2, 3, 0):
        assert L.sv_set_tail(mode) == binding.SV_OK


def test_draft_and_cached_validation(L):
    ws = 1 << 30
    assert binding.sv_draft_workspace_bytes(4, 0, 100) == 0
    assert binding.sv_draft_workspace_bytes(4, 33, 100) == 0
    assert binding.sv_draft_workspace_bytes(4, 3, 100) == binding.sv_workspace_bytes(4, 2, 100)

    def draft(**kw):
        a = dict(L=FAKE, u=FAKE, T=FAKE, B=2, n=3, V=100, dt=1, col=0, ncols=3, tok=FAKE,
                 st=FAKE, ws=FAKE, wsb=ws)
        a.update(kw)
        return L.sv_draft_sample(a["L"], a["u"], a["T"], a["B"], a["n"], a["V"], a["dt"],
                                 a["col"], a["ncols"], a["tok"], a["st"], a["ws"], a["wsb"],
                                 None, None)
    assert draft(dt=3) == binding.SV_ERR_DTYPE
    assert draft(n=0) == binding.SV_ERR_INVALID_ARG
    assert draft(col=-1) == binding.SV_ERR_INVALID_ARG
    assert draft(col=1) == binding.SV_ERR_INVALID_ARG       # col + n > ncols
    assert draft(st=None) == binding.SV_ERR_INVALID_ARG
    assert draft(u=None) == binding.SV_ERR_INVALID_ARG
    assert draft(L=FAKE + 1) == binding.SV_ERR_INVALID_ARG  # bf16 needs 2-byte alignment
    assert draft(wsb=64) == binding.SV_ERR_WORKSPACE
    assert draft(B=0) == binding.SV_OK

    def cached(**kw):
        a = dict(Lt=FAKE, Ld=FAKE, x=FAKE, ds=FAKE, ua=FAKE, ur=FAKE, T=FAKE, B=2, g=3, V=100,
                 dt=0, tok=FAKE, n=FAKE, ws=FAKE, wsb=ws)
        a.update(kw)
        return L.spec_verify_cached(a["Lt"], a["Ld"], a["x"], a["ds"], a["ua"], a["ur"], a["T"],
                                    a["B"], a["g"], a["V"], a["dt"], a["tok"], a["n"], None,
                                    None, a["ws"], a["wsb"], None, None)
    assert cached(ds=None) == binding.SV_ERR_INVALID_ARG
    assert cached(ds=FAKE + 4) == binding.SV_ERR_INVALID_ARG  # stats pairs need 8-byte alignment
    assert cached(g=0, ds=None, Ld=None, x=None, ua=None, wsb=64) == binding.SV_ERR_WORKSPACE
    if not __import__("torch").cuda.is_available():
        assert cached() == binding.SV_ERR_CUDA
        assert draft() == binding.SV_ERR_CUDA


def test_kv_and_window_validation(L):
    assert L.sv_window_cols(64, 16) == 5 and L.sv_window_cols(100, 16) == 8
    assert L.sv_window_cols(5, 1) == 6 and L.sv_window_cols(0, 16) == -1
    assert L.sv_window_cols(16, 0) == -1
    # commit: row bytes a multiple of 16, window >= R, aligned buffers
    def commit(**kw):
        a = dict(kp=FAKE, vp=FAKE, kn=FAKE, vn=FAKE, na=FAKE, pos=FAKE, B=2, LH=3, R=4, rb=256,
                 S=4, W=8)
        a.update(kw)
        return L.sv_kv_commit(a["kp"], a["vp"], a["kn"], a["vn"], a["na"], a["pos"], a["B"],
                              a["LH"], a["R"], a["rb"], a["S"], a["W"], None, None)
    assert commit(rb=24) == binding.SV_ERR_INVALID_ARG
    assert commit(rb=8192 + 16) == binding.SV_ERR_INVALID_ARG   # rows of at most 8 KB
    assert commit(R=65, W=80) == binding.SV_ERR_INVALID_ARG     # at most 64 staged entries
    assert commit(W=3) == binding.SV_ERR_INVALID_ARG
    assert commit(S=-1) == binding.SV_ERR_INVALID_ARG
    assert commit(kp=FAKE + 8) == binding.SV_ERR_INVALID_ARG
    assert commit(pos=None) == binding.SV_ERR_INVALID_ARG
    assert commit(B=0) == binding.SV_OK
    assert L.sv_kv_valid_slots(FAKE, 2, 4, 0, FAKE, FAKE, None, None) == binding.SV_ERR_INVALID_ARG
    assert L.sv_window_block_table(FAKE, FAKE, 2, 4, 64, 16, -1, FAKE, FAKE, None, None,
                                   None) == binding.SV_ERR_INVALID_ARG
    assert L.sv_window_block_table(FAKE, FAKE, 2, 0, 64, 16, 3, FAKE, FAKE, None, None,
                                   None) == binding.SV_ERR_INVALID_ARG


def test_tree_validation(L):
    """sv_tree_verify rejects bad arguments before any CUDA call."""
    def tree(**kw):
        a = dict(dt=binding.SV_BF16, lt=FAKE, ld=FAKE, par=FAKE, tok=FAKE, ua=FAKE, ur=FAKE,
                 temp=FAKE, B=3, N=5, V=100, ot=FAKE, on=FAKE)
        a.update(kw)
        return L.sv_tree_verify(a["dt"], a["lt"], a["ld"], a["par"], a["tok"], a["ua"], a["ur"],
                                a["temp"], a["B"], a["N"], a["V"], a["ot"], a["on"], None, None,
                                None)
    assert tree(dt=2) == binding.SV_ERR_DTYPE
    assert tree(N=0) == binding.SV_ERR_INVALID_ARG
    assert tree(N=binding.SV_TREE_MAX_N + 1) == binding.SV_ERR_INVALID_ARG
    assert tree(V=0) == binding.SV_ERR_INVALID_ARG and tree(B=-1) == binding.SV_ERR_INVALID_ARG
    for k in ("lt", "par", "tok", "ur", "temp", "ot", "on", "ld", "ua"):
        assert tree(**{k: None}) == binding.SV_ERR_INVALID_ARG, k
    assert tree(lt=FAKE + 1) == binding.SV_ERR_INVALID_ARG        # bf16 needs 2-byte alignment
    assert tree(dt=binding.SV_F32, ld=FAKE + 2) == binding.SV_ERR_INVALID_ARG
    assert tree(B=0) == binding.SV_OK
    if not __import__("torch").cuda.is_available():
        # a single-node tree reads no draft row and no accept uniform: these
        # arguments are valid and fail only at the device query
        assert tree(N=1, ld=None, ua=None) == binding.SV_ERR_CUDA
    assert L.sv_tree_set_cluster(9) == binding.SV_ERR_INVALID_ARG
    assert L.sv_tree_set_cluster(-1) == binding.SV_ERR_INVALID_ARG
    assert L.sv_tree_set_cluster(0) == binding.SV_OK
    for w in (1, 12, 32, -8):
        assert L.sv_tree_set_warps(w) == binding.SV_ERR_INVALID_ARG
    for w in (8, 16, 0):
        assert L.sv_tree_set_warps(w) == binding.SV_OK


def test_window_host_mirror_matches_oracle():
    """The host windowing of lengths (the library's CPU code for length
    mirrors) against the oracle, including the page's unit-test example."""
    import numpy as np
    import oracle
    got = binding.sv_window_seq_lens_host([10, 60, 200, 64], 64, 16, 3)
    assert list(got) == [10, 60, 72, 64]
    rng = np.random.default_rng(3)
    for W, blk, K in ((64, 16, 3), (100, 16, 0), (7, 4, 2), (2048, 128, 5)):
        seq = rng.integers(-3, 100000, size=500).astype(np.int32)
        ref = oracle.window_block_table(seq, np.zeros((500, 1), np.int32), W, blk, K)
        assert np.array_equal(binding.sv_window_seq_lens_host(seq, W, blk, K), ref["seq"])
