"""Thin Python binding of libspecverify.so (argument marshalling only).

The functions carry the C ABI's names (include/specverify.h) and take torch
tensors for the device buffers; every step of the verification runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing,
loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build_lib import LIB_PATH

SV_F32, SV_BF16 = 0, 1
SV_OK, SV_ERR_INVALID_ARG, SV_ERR_DTYPE, SV_ERR_CUDA, SV_ERR_WORKSPACE = range(5)
SV_ST_NONFINITE, SV_ST_BAD_TOKEN, SV_ST_BAD_TEMP = 0x1, 0x2, 0x4
SV_ST_TIMEOUT, SV_ST_WORKSPACE, SV_ST_DEGENERATE = 0x8, 0x10, 0x20
SV_ST_BAD_LENGTH = 0x40
SV_MAX_GAMMA = 32

EXPORTED = ("sv_workspace_bytes", "sv_workspace_init", "spec_verify", "spec_verify_diag",
            "spec_verify_greedy", "spec_verify_noalloc", "spec_verify_cached",
            "sv_draft_workspace_bytes", "sv_draft_sample", "sv_set_tuning",
            "sv_set_stage_events", "sv_set_tail", "sv_test_withhold_slot", "sv_error_string",
            "sv_version",
            "sv_kv_commit", "sv_kv_valid_slots", "sv_window_cols", "sv_window_block_table",
            "sv_window_seq_lens_host", "sv_tree_verify", "sv_tree_set_cluster",
            "sv_tree_set_warps")
SV_TREE_MAX_N = 256
SV_NOALLOC_MAX_WORKSPACE = 16 << 20

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    """Load libspecverify.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise SpecVerifyError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.sv_workspace_bytes.argtypes = [I, I, I]
        L.sv_workspace_bytes.restype = Z
        L.sv_workspace_init.argtypes = [P, Z, P]
        L.spec_verify.argtypes = [P, P, P, P, P, P, I, I, I, I, P, P, P, Z, P, P]
        L.spec_verify_diag.argtypes = [P, P, P, P, P, P, I, I, I, I, P, P, P, P, P, Z, P, P]
        L.spec_verify_greedy.argtypes = [P, P, I, I, I, I, P, P, P, Z, P, P]
        L.spec_verify_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, P, P, P, P]
        L.spec_verify_cached.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, P, P, P, P, Z, P, P]
        L.sv_draft_workspace_bytes.argtypes = [I, I, I]
        L.sv_draft_workspace_bytes.restype = Z
        L.sv_draft_sample.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, Z, P, P]
        L.sv_kv_commit.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P]
        L.sv_kv_valid_slots.argtypes = [P, I, I, I, P, P, P, P]
        L.sv_window_cols.argtypes = [I, I]
        L.sv_window_block_table.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P]
        L.sv_window_seq_lens_host.argtypes = [P, I, I, I, I, P]
        L.sv_tree_verify.argtypes = [I, P, P, P, P, P, P, P, I, I, I, P, P, P, P, P]
        L.sv_tree_set_cluster.argtypes = [I]
        L.sv_tree_set_warps.argtypes = [I]
        L.sv_set_tuning.argtypes = [I]
        L.sv_set_tail.argtypes = [I]
        L.sv_set_stage_events.argtypes = [P, I]
        L.sv_test_withhold_slot.argtypes = [I]
        L.sv_error_string.argtypes = [I]
        L.sv_error_string.restype = ctypes.c_char_p
        for name in ("sv_workspace_init", "spec_verify", "spec_verify_diag",
                     "spec_verify_greedy", "spec_verify_noalloc", "spec_verify_cached",
                     "sv_draft_sample", "sv_set_tuning", "sv_set_stage_events", "sv_set_tail",
                     "sv_version",
                     "sv_test_withhold_slot",
                     "sv_kv_commit", "sv_kv_valid_slots", "sv_window_cols",
                     "sv_window_block_table", "sv_window_seq_lens_host", "sv_tree_verify",
                     "sv_tree_set_cluster", "sv_tree_set_warps"):
            getattr(L, name).restype = I
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != SV_OK:
        raise SpecVerifyError(lib().sv_error_string(rc).decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise SpecVerifyError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _dev(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise SpecVerifyError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise SpecVerifyError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise SpecVerifyError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def sv_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return int(lib().sv_workspace_bytes(B, gamma, V))


def sv_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _check(lib().sv_workspace_init(_dev(workspace, None, "workspace"), workspace.numel() *
                                   workspace.element_size(), _stream(stream, workspace.device)))


def make_workspace(B: int, gamma: int, V: int, device) -> torch.Tensor:
    """Allocate (torch caching allocator, 256-byte aligned) and zero a workspace."""
    ws = torch.empty(max(256, sv_workspace_bytes(B, gamma, V)), dtype=torch.uint8, device=device)
    sv_workspace_init(ws)
    return ws


def sv_set_tuning(chunk_elems: int = 0) -> None:
    """Elements per phase-1 chunk for the next calls (0 = automatic)."""
    _check(lib().sv_set_tuning(chunk_elems))


def sv_test_withhold_slot(enable: bool) -> None:
    """Failure-handling test aid: the next calls' streaming kernel leaves one
    slot unfilled, so its bounded wait runs out (SV_ST_TIMEOUT)."""
    _check(lib().sv_test_withhold_slot(1 if enable else 0))


def sv_set_tail(mode: int = 0) -> None:
    """Kernels of sampling calls: 0 automatic, 1 the reduce and the decide /
    residual / draw kernels, 2 the reduce and the fused tail, 3 one kernel
    (a cluster per request streams its rows, then decides and draws)."""
    _check(lib().sv_set_tail(mode))


def sv_set_stage_events(events) -> None:
    """Record these torch.cuda.Events (already recorded once, so they exist)
    around the kernels of the next calls; an empty list turns it off."""
    handles = (ctypes.c_void_p * max(1, len(events)))(*[e.cuda_event for e in events])
    _check(lib().sv_set_stage_events(handles if events else None, len(events)))


def _shapes(target_logits: torch.Tensor):
    if target_logits.dim() != 3:
        raise SpecVerifyError("target_logits must be [B][gamma+1][V]")
    B, R, V = target_logits.shape
    return B, R - 1, V


def spec_verify_diag(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                     temperature, out_tokens, out_num_accepted, out_p, out_Z, workspace,
                     dev_status=None, stream=None) -> None:
    B, g, V = _shapes(target_logits)
    dt = _dtype_code(target_logits)
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError("draft_logits must have the dtype of target_logits")
    _check(lib().spec_verify_diag(
        _dev(target_logits, None, "target_logits"), _dev(draft_logits, None, "draft_logits"),
        _dev(draft_tokens, torch.int32, "draft_tokens"), _dev(u_accept, torch.float32, "u_accept"),
        _dev(u_resample, torch.float32, "u_resample"),
        _dev(temperature, torch.float32, "temperature"), B, g, V, dt,
        _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_num_accepted, torch.int32, "out_num_accepted"),
        _dev(out_p, torch.float32, "out_p"), _dev(out_Z, torch.float32, "out_Z"),
        _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, target_logits.device)))


def spec_verify(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature,
                out_tokens, out_num_accepted, workspace, dev_status=None, stream=None) -> None:
    B, g, V = _shapes(target_logits)
    dt = _dtype_code(target_logits)
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError("draft_logits must have the dtype of target_logits")
    _check(lib().spec_verify(
        _dev(target_logits, None, "target_logits"), _dev(draft_logits, None, "draft_logits"),
        _dev(draft_tokens, torch.int32, "draft_tokens"), _dev(u_accept, torch.float32, "u_accept"),
        _dev(u_resample, torch.float32, "u_resample"),
        _dev(temperature, torch.float32, "temperature"), B, g, V, dt,
        _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_num_accepted, torch.int32, "out_num_accepted"),
        _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, target_logits.device)))


def spec_verify_greedy(target_logits, draft_tokens, out_tokens, out_num_accepted, workspace,
                       dev_status=None, stream=None) -> None:
    B, g, V = _shapes(target_logits)
    dt = _dtype_code(target_logits)
    _check(lib().spec_verify_greedy(
        _dev(target_logits, None, "target_logits"), _dev(draft_tokens, torch.int32, "draft_tokens"),
        B, g, V, dt, _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_num_accepted, torch.int32, "out_num_accepted"),
        _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, target_logits.device)))


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                        temperature, out_tokens, out_num_accepted, dev_status=None,
                        stream=None) -> None:
    """spec_verify without a workspace, for callers that may not allocate
    device memory: the library's built-in scratch (SV_NOALLOC_MAX_WORKSPACE
    bytes per device) is used instead.  Calls that may overlap on the GPU
    share that scratch and race; serialise them."""
    B, g, V = _shapes(target_logits)
    dt = _dtype_code(target_logits)
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError("draft_logits must have the dtype of target_logits")
    _check(lib().spec_verify_noalloc(
        _dev(target_logits, None, "target_logits"), _dev(draft_logits, None, "draft_logits"),
        _dev(draft_tokens, torch.int32, "draft_tokens"), _dev(u_accept, torch.float32, "u_accept"),
        _dev(u_resample, torch.float32, "u_resample"),
        _dev(temperature, torch.float32, "temperature"), B, g, V, dt,
        _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_num_accepted, torch.int32, "out_num_accepted"),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, target_logits.device)))


def sv_draft_workspace_bytes(B: int, n: int, V: int) -> int:
    return int(lib().sv_draft_workspace_bytes(B, n, V))


def make_draft_workspace(B: int, n: int, V: int, device) -> torch.Tensor:
    """Allocate and zero a workspace for sv_draft_sample."""
    ws = torch.empty(max(256, sv_draft_workspace_bytes(B, n, V)), dtype=torch.uint8,
                     device=device)
    sv_workspace_init(ws)
    return ws


def sv_draft_sample(draft_logits, u_draft, temperature, out_tokens, out_stats, workspace,
                    col: int = 0, dev_status=None, stream=None) -> None:
    """Sample one token per draft row of draft_logits [B][n][V] and report the
    rows' normalisers: out_tokens [B][ncols] int32 and out_stats [B][ncols][2]
    float32 get columns col .. col + n - 1 (ncols = out_tokens.shape[1])."""
    if draft_logits.dim() != 3:
        raise SpecVerifyError("draft_logits must be [B][n][V]")
    B, n, V = draft_logits.shape
    if out_tokens.dim() != 2 or out_tokens.shape[0] != B:
        raise SpecVerifyError("out_tokens must be [B][ncols]")
    ncols = out_tokens.shape[1]
    if tuple(out_stats.shape) != (B, ncols, 2):
        raise SpecVerifyError("out_stats must be [B][ncols][2]")
    _check(lib().sv_draft_sample(
        _dev(draft_logits, None, "draft_logits"), _dev(u_draft, torch.float32, "u_draft"),
        _dev(temperature, torch.float32, "temperature"), B, n, V, _dtype_code(draft_logits),
        col, ncols, _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_stats, torch.float32, "out_stats"), _dev(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, draft_logits.device)))


def spec_verify_cached(target_logits, draft_logits, draft_tokens, draft_stats, u_accept,
                       u_resample, temperature, out_tokens, out_num_accepted, workspace,
                       out_p=None, out_Z=None, dev_status=None, stream=None) -> None:
    """spec_verify with the draft rows' normalisers draft_stats [B][gamma][2]
    (as sv_draft_sample writes them): the draft rows are not streamed."""
    B, g, V = _shapes(target_logits)
    dt = _dtype_code(target_logits)
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError("draft_logits must have the dtype of target_logits")
    _check(lib().spec_verify_cached(
        _dev(target_logits, None, "target_logits"), _dev(draft_logits, None, "draft_logits"),
        _dev(draft_tokens, torch.int32, "draft_tokens"),
        _dev(draft_stats, torch.float32, "draft_stats"), _dev(u_accept, torch.float32, "u_accept"),
        _dev(u_resample, torch.float32, "u_resample"),
        _dev(temperature, torch.float32, "temperature"), B, g, V, dt,
        _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_num_accepted, torch.int32, "out_num_accepted"),
        _dev(out_p, torch.float32, "out_p"), _dev(out_Z, torch.float32, "out_Z"),
        _dev(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, target_logits.device)))


# ------------------------------------------------------------ KV-cache steps

def sv_kv_commit(k_pool, v_pool, k_new, v_new, num_accepted, pos, sink: int, window: int,
                 dev_status=None, stream=None) -> None:
    """Commit the accepted staged entries to a sink + ring KV cache.
    k_pool/v_pool [B][LH][sink+window][D], k_new/v_new [B][LH][R][D] (any
    element type, D * element size a multiple of 16); num_accepted [B] and
    pos [B] int32 (pos is advanced in place)."""
    if k_pool.dim() != 4 or k_new.dim() != 4:
        raise SpecVerifyError("pools must be [B][LH][sink+window][D], staged entries [B][LH][R][D]")
    B, LH, C, D = k_pool.shape
    R = k_new.shape[2]
    if (tuple(v_pool.shape) != tuple(k_pool.shape) or tuple(v_new.shape) != tuple(k_new.shape)
            or tuple(k_new.shape) != (B, LH, R, D) or C != sink + window):
        raise SpecVerifyError("KV shapes disagree")
    if len({k_pool.dtype, v_pool.dtype, k_new.dtype, v_new.dtype}) != 1:
        raise SpecVerifyError("KV buffers must share one dtype")
    _check(lib().sv_kv_commit(
        _dev(k_pool, None, "k_pool"), _dev(v_pool, None, "v_pool"), _dev(k_new, None, "k_new"),
        _dev(v_new, None, "v_new"), _dev(num_accepted, torch.int32, "num_accepted"),
        _dev(pos, torch.int32, "pos"), B, LH, R, D * k_pool.element_size(), sink, window,
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, k_pool.device)))


def sv_kv_valid_slots(pos, sink: int, window: int, out_slots, out_len, dev_status=None,
                      stream=None) -> None:
    """Valid physical slots of every request in logical order: out_slots
    [B][sink+window] (-1 padded) and out_len [B], int32."""
    B = pos.shape[0]
    _check(lib().sv_kv_valid_slots(
        _dev(pos, torch.int32, "pos"), B, sink, window, _dev(out_slots, torch.int32, "out_slots"),
        _dev(out_len, torch.int32, "out_len"), _dev(dev_status, torch.int32, "dev_status"),
        _stream(stream, pos.device)))


def sv_window_cols(window: int, block_size: int) -> int:
    return int(lib().sv_window_cols(window, block_size))


def sv_window_block_table(seq_lens, block_table, window: int, block_size: int,
                          future_offset: int, out_seq_lens, out_block_table,
                          out_start_block=None, dev_status=None, stream=None) -> None:
    """Draft KV sliding window on the device: windowed lengths and the
    zero-padded block-table clone [B][sv_window_cols(window, block_size)]."""
    B, full_cols = block_table.shape
    _check(lib().sv_window_block_table(
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(block_table, torch.int32, "block_table"),
        B, full_cols, window, block_size, future_offset,
        _dev(out_seq_lens, torch.int32, "out_seq_lens"),
        _dev(out_block_table, torch.int32, "out_block_table"),
        _dev(out_start_block, torch.int32, "out_start_block"),
        _dev(dev_status, torch.int32, "dev_status"), _stream(stream, seq_lens.device)))


def sv_window_seq_lens_host(seq_lens, window: int, block_size: int, future_offset: int):
    """The same windowing of lengths on the host (for host-side mirrors):
    an int32 numpy array in, a new one out."""
    import numpy as np
    src = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.empty_like(src)
    _check(lib().sv_window_seq_lens_host(
        src.ctypes.data_as(ctypes.c_void_p), int(src.size), window, block_size, future_offset,
        out.ctypes.data_as(ctypes.c_void_p)))
    return out


def sv_tree_verify(target_logits, draft_logits, parent, tokens, u_accept, u_residual,
                   temperature, out_tokens, out_num_accepted, out_nodes=None, dev_status=None,
                   stream=None) -> None:
    """Token-tree verification.  target_logits / draft_logits [B][N][V]
    (float32 or bfloat16; draft_logits may be None when N == 1), parent /
    tokens [B][N] int32, u_accept / u_residual [B][N] and temperature [B]
    float32; outputs out_tokens [B][N], out_num_accepted [B], out_nodes
    [B][N] (optional), all int32."""
    if target_logits.dim() != 3:
        raise SpecVerifyError("target_logits must be [B][N][V]")
    B, N, V = target_logits.shape
    dt = _dtype_code(target_logits)
    if draft_logits is not None and (draft_logits.dtype != target_logits.dtype
                                     or tuple(draft_logits.shape) != (B, N, V)):
        raise SpecVerifyError("draft_logits must match target_logits in shape and dtype")
    _check(lib().sv_tree_verify(
        dt, _dev(target_logits, None, "target_logits"), _dev(draft_logits, None, "draft_logits"),
        _dev(parent, torch.int32, "parent"), _dev(tokens, torch.int32, "tokens"),
        _dev(u_accept, torch.float32, "u_accept"), _dev(u_residual, torch.float32, "u_residual"),
        _dev(temperature, torch.float32, "temperature"), B, N, V,
        _dev(out_tokens, torch.int32, "out_tokens"),
        _dev(out_num_accepted, torch.int32, "out_num_accepted"),
        _dev(out_nodes, torch.int32, "out_nodes"), _dev(dev_status, torch.int32, "dev_status"),
        _stream(stream, target_logits.device)))


def sv_tree_set_cluster(ctas: int = 0) -> None:
    """CTAs per request for sv_tree_verify: 0 = automatic, 1..8 forced."""
    _check(lib().sv_tree_set_cluster(int(ctas)))


def sv_tree_set_warps(warps: int = 0) -> None:
    """Warps per CTA for sv_tree_verify: 0 = automatic, 8 or 16 forced."""
    _check(lib().sv_tree_set_warps(int(warps)))
