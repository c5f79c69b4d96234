"""GPU parity of the KV-cache steps (sv_kv_commit, sv_kv_valid_slots,
sv_window_block_table) through the C ABI against the oracle on the same
seeded inputs: integer and byte work, so every comparison is bit-exact."""
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_09_gb300 import binding

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _commit(kp, vp, kn, vn, k, pos, S, W):
    """Run sv_kv_commit on device copies; returns host pools, pos and status."""
    d = [_t(a) for a in (kp, vp, kn, vn)]
    kd, pd = _t(k.astype(np.int32)), _t(pos.astype(np.int32))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.sv_kv_commit(d[0], d[1], d[2], d[3], kd, pd, S, W, dev_status=st)
    torch.cuda.synchronize()
    return d[0].cpu().numpy(), d[1].cpu().numpy(), pd.cpu().numpy(), int(st.item())


def _valid(pos, S, W):
    pd = _t(pos.astype(np.int32))
    B = pos.shape[0]
    slots = torch.full((B, S + W), -7, dtype=torch.int32, device=DEV)
    ln = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.sv_kv_valid_slots(pd, S, W, slots, ln, dev_status=st)
    torch.cuda.synchronize()
    return slots.cpu().numpy(), ln.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("dtype,D", [(np.int16, 8), (np.float32, 4), (np.int16, 128)])
@pytest.mark.parametrize("S,W", [(0, 5), (4, 6), (3, 16)])
def test_commit_steps(dtype, D, S, W):
    """Twelve verification steps per request with random outcomes (including
    dropped requests, k = -1): pools, positions and the valid-slot lists
    equal the oracle's after every step."""
    rng = np.random.default_rng(100 + D + S + W)
    B, LH, R = 5, 3, 4
    C = S + W
    kp = rng.integers(0, 1 << 15, size=(B, LH, C, D)).astype(dtype)
    vp = rng.integers(0, 1 << 15, size=(B, LH, C, D)).astype(dtype)
    pos = np.zeros(B, np.int32)
    pos[1] = 2 * C + 3  # a request well into its ring
    for step in range(12):
        kn = rng.integers(0, 1 << 15, size=(B, LH, R, D)).astype(dtype)
        vn = rng.integers(0, 1 << 15, size=(B, LH, R, D)).astype(dtype)
        k = rng.integers(-1, R, size=B).astype(np.int32)
        ref = oracle.kv_commit(kp, vp, kn, vn, k, pos, S, W)
        gk, gv, gpos, st = _commit(kp, vp, kn, vn, k, pos, S, W)
        assert st == 0 and np.all(ref["flags"] == 0)
        assert np.array_equal(gpos, ref["pos"])
        assert np.array_equal(gk, ref["k_pool"]) and np.array_equal(gv, ref["v_pool"])
        kp, vp, pos = ref["k_pool"], ref["v_pool"], ref["pos"]
        slots, ln, st = _valid(pos, S, W)
        vref = oracle.kv_valid_slots(pos, S, W)
        assert st == 0
        assert np.array_equal(slots, vref["slots"]) and np.array_equal(ln, vref["len"])


def test_commit_model_sized():
    """A 1.8B-class target's KV rows (24 layers x 16 heads, head dim 128,
    16-bit elements: 384 rows of 256 bytes per token), 64 requests, gamma = 4, a ring of
    64 behind 4 sinks; positions spread over several laps of the ring."""
    rng = np.random.default_rng(7)
    B, LH, R, D, S, W = 64, 384, 5, 128, 4, 64
    kp = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, S + W, D), dtype=np.int16)
    vp = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, S + W, D), dtype=np.int16)
    kn = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, R, D), dtype=np.int16)
    vn = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, R, D), dtype=np.int16)
    k = rng.integers(0, R, size=B).astype(np.int32)
    pos = rng.integers(0, 5 * (S + W), size=B).astype(np.int32)
    ref = oracle.kv_commit(kp, vp, kn, vn, k, pos, S, W)
    gk, gv, gpos, st = _commit(kp, vp, kn, vn, k, pos, S, W)
    assert st == 0
    assert np.array_equal(gpos, ref["pos"])
    assert np.array_equal(gk, ref["k_pool"]) and np.array_equal(gv, ref["v_pool"])


def test_commit_invalid_requests_isolated():
    rng = np.random.default_rng(9)
    B, LH, R, D, S, W = 6, 2, 3, 4, 2, 5
    kp = rng.random((B, LH, S + W, D), dtype=np.float32)
    vp = rng.random((B, LH, S + W, D), dtype=np.float32)
    kn = rng.random((B, LH, R, D), dtype=np.float32)
    vn = rng.random((B, LH, R, D), dtype=np.float32)
    k = np.array([1, R, 0, -1, 2, 1], np.int32)       # k = R: past the staged entries
    pos = np.array([3, 4, -2, 5, 0, 9], np.int32)     # pos < 0: invalid
    ref = oracle.kv_commit(kp, vp, kn, vn, k, pos, S, W)
    gk, gv, gpos, st = _commit(kp, vp, kn, vn, k, pos, S, W)
    assert st == binding.SV_ST_BAD_LENGTH
    assert list(ref["flags"]) == [0, oracle.KV_INVALID, oracle.KV_INVALID, 0, 0, 0]
    assert np.array_equal(gpos, ref["pos"])
    assert np.array_equal(gk, ref["k_pool"]) and np.array_equal(gv, ref["v_pool"])
    slots, ln, st = _valid(gpos, S, W)
    assert st == binding.SV_ST_BAD_LENGTH and ln[2] == 0 and np.all(slots[2] == -1)


def _window(seq, table, W, blk, K):
    cols = binding.sv_window_cols(W, blk)
    B = table.shape[0]
    os_ = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    ot = torch.full((B, cols), -7, dtype=torch.int32, device=DEV)
    sb = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.sv_window_block_table(_t(seq.astype(np.int32)), _t(table.astype(np.int32)), W, blk, K,
                                  os_, ot, sb, dev_status=st)
    torch.cuda.synchronize()
    return os_.cpu().numpy(), ot.cpu().numpy(), sb.cpu().numpy(), int(st.item())


def test_window_page_example():
    table = np.arange(64, dtype=np.int32).reshape(4, 16) + 1000
    seq = np.array([10, 60, 200, 64], np.int32)
    got = _window(seq, table, 64, 16, 3)
    ref = oracle.window_block_table(seq, table, 64, 16, 3)
    assert list(got[0]) == [10, 60, 72, 64]
    assert np.array_equal(got[1], ref["table"]) and np.array_equal(got[2], ref["start_block"])


@pytest.mark.parametrize("W,blk,K", [(64, 16, 3), (100, 16, 0), (2048, 128, 4), (7, 4, 2),
                                     (512, 1, 1), (33, 64, 0)])
def test_window_random(W, blk, K):
    rng = np.random.default_rng(W + blk + K)
    B = 300
    full = 1 + (W + 4096) // blk
    seq = rng.integers(0, full * blk + 1, size=B).astype(np.int32)
    seq[:4] = [0, 1, full * blk, W + K]
    seq[4] = -5  # invalid
    table = rng.integers(1, 1 << 30, size=(B, full)).astype(np.int32)
    got = _window(seq, table, W, blk, K)
    ref = oracle.window_block_table(seq, table, W, blk, K)
    assert np.array_equal(got[0], ref["seq"])
    assert np.array_equal(got[1], ref["table"])
    assert np.array_equal(got[2], ref["start_block"])
    assert got[3] == binding.SV_ST_BAD_LENGTH
    # every length mirror is windowed alike: the host function gives the same lengths
    assert np.array_equal(binding.sv_window_seq_lens_host(seq, W, blk, K), got[0])


@pytest.mark.parametrize("seed", range(int(os.environ.get("SV_KV_FUZZ_SEEDS", "24"))))
def test_commit_fuzz(seed):
    """Random shapes (batch, layer-heads, staged entries, row size, sinks,
    window), positions near and far into the ring, accepted counts including
    dropped requests (-1): pools, positions and valid slots bit-exact with
    the oracle."""
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 20))
    LH = int(rng.integers(1, 6))
    R = int(rng.integers(1, 9))
    D = int(rng.choice([8, 16, 64, 256]))  # int16 elements: rows of 16 .. 512 bytes
    S = int(rng.integers(0, 5))
    W = int(rng.integers(R, R + 12))
    C = S + W
    kp = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, C, D)).astype(np.int16)
    vp = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, C, D)).astype(np.int16)
    kn = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, R, D)).astype(np.int16)
    vn = rng.integers(-(1 << 15), 1 << 15, size=(B, LH, R, D)).astype(np.int16)
    pos = rng.integers(0, 4 * C + 3, size=B).astype(np.int32)
    k = rng.integers(-1, R, size=B).astype(np.int32)
    gk, gv, gpos, st = _commit(kp, vp, kn, vn, k, pos, S, W)
    ref = oracle.kv_commit(kp, vp, kn, vn, k, pos, S, W)
    assert st == 0
    assert np.array_equal(gk, ref["k_pool"]) and np.array_equal(gv, ref["v_pool"])
    assert np.array_equal(gpos, ref["pos"])
    slots, ln, st2 = _valid(gpos, S, W)
    vref = oracle.kv_valid_slots(gpos, S, W)
    assert st2 == 0
    assert np.array_equal(ln, vref["len"])
    for b in range(B):
        assert np.array_equal(slots[b, :ln[b]], vref["slots"][b, :vref["len"][b]])
