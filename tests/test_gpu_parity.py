"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  See tests/gpu_util.py for the comparison rules."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, check_valid_draw, compare_greedy, compare_sampling, oracle_sampling,
                      run_greedy, run_sampling, to_dev)
from speculative_decoding_verification_09_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True, params=[1, 2, 3], ids=["tail3", "fused", "onecall"])
def _gpu(request):
    """Every test of the module runs three times: with the decide / residual /
    draw kernels after the reduce, with the fused tail (one cluster per
    request), and as one kernel (the cluster also streams its request's
    rows), whatever the batch size."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    binding.sv_set_tail(request.param)
    _TAIL[0] = request.param
    yield
    binding.sv_set_tail(0)
    _TAIL[0] = 0


_TAIL = [0]


def _gpu_tail() -> int:
    """The tail the module fixture selected for the running tests."""
    return _TAIL[0]


NEAR_LOG = []


def assert_same_or_valid(inp, got, ref):
    """Tokens and counts as the oracle's, or, at a flagged near-tie, a draw
    the rule allows within the 1e-6 window (check_valid_draw)."""
    near = (ref["flags"] & oracle.NEAR_ANY) != 0
    same = np.all(got["tokens"] == ref["tokens"], axis=1) & (got["n"] == ref["n"])
    assert np.all(same | near), np.argwhere(~(same | near)).ravel()
    for b in np.flatnonzero(~same):
        check_valid_draw(inp, got, ref, int(b))


# ------------------------------------------------------------ small sweeps

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("gamma", [0, 1, 3, 8])
@pytest.mark.parametrize("V", [1, 2, 3, 8, 33, 1000, 4099])
def test_small_sweep(V, gamma, dtype):
    cfg = synth.custom_config(5, gamma, V, dtype, "normal", temp=0.85)
    inp = synth.make_inputs(cfg, seed=1000 + V * 7 + gamma)
    stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    NEAR_LOG.append(stats)
    assert stats["mismatches"] <= max(1.0, 1e-4 * stats["positions"])


@pytest.mark.parametrize("kind", ["normal", "zipf", "mix"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_several_tiles_ragged(kind, dtype):
    """V = 20011 (odd: unaligned rows for both dtypes), 37 requests: several
    phase-1 chunks and three phase-2 chunks per row, each with a ragged tail."""
    cfg = synth.custom_config(37, 5, 20011, dtype, kind, temp=0.9)
    inp = synth.make_inputs(cfg, seed=77)
    stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    assert stats["mismatches"] <= 1


def test_per_request_temperature_and_low_acceptance():
    cfg = synth.custom_config(64, 4, 3001, "f32", "normal", temp=("uniform", 0.05, 3.0),
                              sigma_noise=3.0)
    inp = synth.make_inputs(cfg, seed=5)
    stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    assert stats["accepted"] < inp.B * inp.gamma  # rejections happened


# ------------------------------------------------------- the five workloads

@pytest.mark.parametrize("cid", [1, 3, 4, 5])
def test_workload_full_size(cid):
    inp = synth.make_inputs(cid)
    got = run_sampling(inp)
    ref = oracle_sampling(inp)
    stats = compare_sampling(inp, got, ref)
    print(f"\n{inp.name}: {stats}")
    # Flagged near-ties are reported, not bounded: the 1e-6 CDF-edge window
    # flags ~V * 1e-6 of the draws at LLM vocabularies.  Tokens that actually
    # differ must stay below 1e-4 of the positions (at most one here).
    assert stats["mismatches"] <= max(1.0, 1e-4 * stats["positions"])
    if cid == 4:  # acceptance rises with the mixture weight (0.3 / 0.6 / 0.9 per third)
        third = np.minimum(3 * np.arange(inp.B) // inp.B, 2)
        acc = [ref["n"][third == t].mean() for t in range(3)]
        assert acc[0] < acc[1] < acc[2]


def test_workload2_greedy_full_size():
    inp = synth.make_inputs(2)
    got = run_greedy(inp)
    ref = oracle.greedy(inp.Lt, inp.x, inp.dtype)
    compare_greedy(got, ref)
    assert 0 < ref["n"].sum() < inp.B * inp.gamma


# ------------------------------------------------------------------ greedy

@pytest.mark.parametrize("gamma", [2, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 513, 20011, 70000])
def test_greedy_planted_ties(V, dtype, gamma):
    """Ties inside a vector, across vectors and across phase-1 chunks; the
    lowest index must win; draft tokens equal to the argmax for a random
    prefix, then a mismatch.  gamma = 2 takes the decision kernel's
    four-warp form (R <= 4), gamma = 4 its sixteen-warp form."""
    cfg = synth.custom_config(24, gamma, V, dtype, "greedy")
    inp = synth.make_inputs(cfg, seed=V)
    wide = synth.widen(inp.Lt, inp.dtype)
    rng = np.random.default_rng(V)
    for b in range(inp.B):
        for i in range(inp.gamma + 1):
            a = int(np.argmax(wide[b, i]))
            for pos in rng.integers(0, V, size=3):
                inp.Lt[b, i, pos] = inp.Lt[b, i, a]
            if b % 2 and a > 0:
                inp.Lt[b, i, a - 1] = inp.Lt[b, i, a]
    wide = synth.widen(inp.Lt, inp.dtype)
    amax = np.argmax(wide, axis=2).astype(np.int32)
    x = amax[:, :inp.gamma].copy()
    kk = rng.integers(0, inp.gamma + 1, size=inp.B)
    for b in range(inp.B):
        if kk[b] < inp.gamma and V > 1:
            x[b, kk[b]] = (amax[b, kk[b]] + 1) % V
    ref = oracle.greedy(inp.Lt, x, inp.dtype)
    compare_greedy(run_greedy(inp, x=x), ref)


# ------------------------------------------------------------- edge cases

def test_invalid_requests_are_isolated():
    cfg = synth.custom_config(12, 2, 3000, "f32", "normal")
    inp = synth.make_inputs(cfg, seed=3)
    inp.Lt[1, 0, 5] = np.nan
    inp.Ld[2, 1, 0] = np.inf
    inp.Lt[3, 2, :] = -np.inf
    inp.x[4, 1] = inp.V
    inp.x[5, 0] = -1
    inp.temp[6], inp.temp[7], inp.temp[8], inp.temp[9] = 0.0, -1.0, np.nan, np.float32(1e-39)
    inp.temp[10] = np.inf
    inp.Lt[11, 1, :] = -np.inf
    inp.Lt[11, 1, 3] = 0.0
    got, ref = run_sampling(inp), oracle_sampling(inp)
    compare_sampling(inp, got, ref)
    assert got["status"] & (binding.SV_ST_NONFINITE | binding.SV_ST_BAD_TOKEN |
                            binding.SV_ST_BAD_TEMP) == 0x7


def test_invalid_bf16_and_greedy():
    cfg = synth.custom_config(6, 3, 5000, "bf16", "normal")
    inp = synth.make_inputs(cfg, seed=4)
    inp.Lt[0, 3, 4999] = 0x7FC0   # NaN in the bonus row
    inp.Ld[1, 0, 17] = 0x7F80     # +inf in a draft row
    inp.Lt[2, 1, :] = 0xFF80      # all -inf
    compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    ref = oracle.greedy(inp.Lt, inp.x, inp.dtype)
    compare_greedy(run_greedy(inp), ref)


def test_neg_inf_entries_are_legal():
    cfg = synth.custom_config(16, 4, 2500, "bf16", "normal")
    inp = synth.make_inputs(cfg, seed=8)
    rng = np.random.default_rng(8)
    mask_t = rng.random(inp.Lt.shape) < 0.3
    mask_d = rng.random(inp.Ld.shape) < 0.3
    inp.Lt[mask_t] = 0xFF80
    inp.Ld[mask_d] = 0xFF80
    for b in range(inp.B):  # keep the draft tokens possible under the draft
        for i in range(inp.gamma):
            inp.Ld[b, i, inp.x[b, i]] = 0
    got, ref = run_sampling(inp), oracle_sampling(inp)
    assert np.all((ref["flags"] & oracle.INVALID_ANY) == 0)
    compare_sampling(inp, got, ref)


def test_near_identical_rows():
    """Target and draft almost equal: tiny residual masses (the cancellation
    case); tokens must still match outside flagged near-ties."""
    cfg = synth.custom_config(32, 3, 4096, "f32", "normal", sigma_noise=1e-4, temp=1.0)
    inp = synth.make_inputs(cfg, seed=9)
    inp.u_acc[:] = 0.999999
    got, ref = run_sampling(inp), oracle_sampling(inp)
    stats = compare_sampling(inp, got, ref)
    print(f"\nnear-identical rows: {stats}")
    ok = (ref["flags"] & oracle.INVALID_ANY) == 0
    assert np.all((got["tokens"][ok] >= -1) & (got["tokens"][ok] < inp.V))
    assert stats["mismatches"] <= max(1.0, 1e-4 * stats["positions"])


def test_empty_batch_is_a_noop():
    ws = binding.make_workspace(1, 2, 10, DEV)
    z = torch.empty((0, 3, 10), dtype=torch.float32, device=DEV)
    e = torch.empty((0, 2), dtype=torch.int32, device=DEV)
    binding.spec_verify(z, torch.empty((0, 2, 10), device=DEV), e,
                        torch.empty((0, 2), device=DEV), torch.empty((0, 3), device=DEV),
                        torch.empty((0,), device=DEV), torch.empty((0, 3), dtype=torch.int32,
                                                                   device=DEV),
                        torch.empty((0,), dtype=torch.int32, device=DEV), ws)


def test_repeated_calls_reuse_workspace_and_streams():
    cfg = synth.custom_config(20, 4, 12345, "bf16", "mix")
    inp = synth.make_inputs(cfg, seed=10)
    d = to_dev(inp)
    ws = binding.make_workspace(64, 8, 20000, DEV)  # larger than needed, shared by shapes
    ref = oracle_sampling(inp)
    first = run_sampling(inp, d, ws)
    compare_sampling(inp, first, ref)
    s = torch.cuda.Stream()
    for _ in range(3):
        again = run_sampling(inp, d, ws, stream=s)
        assert np.array_equal(again["tokens"], first["tokens"]) and again["status"] == 0
    other = synth.make_inputs(synth.custom_config(3, 8, 777, "f32", "zipf"), seed=11)
    compare_sampling(other, run_sampling(other, ws=ws), oracle_sampling(other))
    g = run_greedy(inp, ws=ws)
    compare_greedy(g, oracle.greedy(inp.Lt, inp.x, inp.dtype))
    again = run_sampling(inp, d, ws)
    assert np.array_equal(again["tokens"], first["tokens"]) and again["status"] == 0


def test_overlapping_calls_on_three_streams():
    """Calls that overlap on the GPU (three streams, one workspace each, all
    queued before any is waited for, different batches and shapes per
    stream) each give the oracle's results."""
    cfgs = [synth.custom_config(12, 3, 9001, "bf16", "mix"),
            synth.custom_config(100, 2, 4099, "f32", "normal", temp=("uniform", 0.5, 1.5)),
            synth.custom_config(7, 5, 20011, "bf16", "zipf", temp=0.8)]
    inps = [synth.make_inputs(c, seed=60 + j) for j, c in enumerate(cfgs)]
    refs = [oracle_sampling(x) for x in inps]
    streams = [torch.cuda.Stream() for _ in inps]
    devs = [to_dev(x) for x in inps]
    wss = [binding.make_workspace(x.B, x.gamma, x.V, DEV) for x in inps]
    outs = []
    for x in inps:
        outs.append(dict(tok=torch.full((x.B, x.gamma + 1), -7, dtype=torch.int32, device=DEV),
                         n=torch.full((x.B,), -7, dtype=torch.int32, device=DEV),
                         st=torch.zeros(1, dtype=torch.int32, device=DEV)))
    torch.cuda.synchronize()
    for rep in range(4):  # each stream's calls queue behind one another
        for x, d, ws, o, s in zip(inps, devs, wss, outs, streams):
            binding.spec_verify(d["Lt"], d["Ld"], d["x"], d["u_acc"], d["u_res"], d["temp"],
                                o["tok"], o["n"], ws, o["st"], s)
    torch.cuda.synchronize()
    for x, o, ref in zip(inps, outs, refs):
        got = dict(tokens=o["tok"].cpu().numpy(), n=o["n"].cpu().numpy(),
                   p=np.zeros((x.B, x.gamma, 2), np.float32), Z=np.zeros(x.B, np.float32),
                   status=int(o["st"].item()))
        assert_same_or_valid(x, got, ref)
        assert got["status"] == 0


# Workspace layout facts used to poison it: the control block takes bytes
# 0..63 (the call-state word at byte 0, the reduce's pool-claim counter at
# byte 8, both 0 between calls); the partials start at byte 256.
def test_garbage_request_words_are_harmless():
    """Every workspace region past the control block is written before it is
    read within a call, so leftover or garbage words there (another shape's
    partials or records) cannot change the result."""
    cfg = synth.custom_config(8, 3, 6000, "bf16", "normal")
    inp = synth.make_inputs(cfg, seed=12)
    d = to_dev(inp)
    ws = binding.make_workspace(inp.B, inp.gamma, inp.V, DEV)
    ref = oracle_sampling(inp)
    ws[256:256 + 8 * 32].view(torch.int32).copy_(
        torch.randint(-2**31, 2**31 - 1, (8 * 8,), dtype=torch.int32, device=DEV))
    compare_sampling(inp, run_sampling(inp, d, ws), ref)
    ws[256:264].view(torch.int64).fill_(3)  # request 0: a stale decision flag
    compare_sampling(inp, run_sampling(inp, d, ws), ref)


def test_poisoned_task_counter_is_detected_and_repaired():
    cfg = synth.custom_config(4, 2, 3000, "f32", "normal")
    inp = synth.make_inputs(cfg, seed=13)
    d = to_dev(inp)
    ws = binding.make_workspace(inp.B, inp.gamma, inp.V, DEV)
    ref = oracle_sampling(inp)
    ws[0:8].view(torch.int64).fill_(1 << 40)  # the control block is not in its ready state
    bad = run_sampling(inp, d, ws)
    assert bad["status"] & binding.SV_ST_WORKSPACE
    compare_sampling(inp, run_sampling(inp, d, ws), ref)
    ws[8:16].view(torch.int64).fill_(5)  # a stale pool-claim count
    bad = run_sampling(inp, d, ws)
    assert bad["status"] & binding.SV_ST_WORKSPACE
    compare_sampling(inp, run_sampling(inp, d, ws), ref)


def test_small_calls_in_a_loop_report_no_workspace_error():
    """Many back-to-back calls of the smallest workload (one request of
    V = 32000: about one reduce task per CTA, so every CTA reaches the pool
    claims at its first chunk) on one workspace: none may report
    SV_ST_WORKSPACE (the ready-state check must not race with the claims of
    the call's own CTAs), and every call gives the oracle's tokens."""
    inp = synth.make_inputs(1)
    d = to_dev(inp)
    ws = binding.make_workspace(inp.B, inp.gamma, inp.V, DEV)
    ref = oracle_sampling(inp)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok = torch.full((inp.B, inp.gamma + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((inp.B,), -7, dtype=torch.int32, device=DEV)
    for _ in range(300):
        binding.spec_verify(d["Lt"], d["Ld"], d["x"], d["u_acc"], d["u_res"], d["temp"], tok, n,
                            ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_same_or_valid(inp, dict(tokens=tok.cpu().numpy(), n=n.cpu().numpy()), ref)


def test_bounded_wait_reports_timeout_and_context_recovers():
    """Failure handling without a fault: with one reduce slot withheld, that
    slot's waits run out after their one-second limit; the call reports
    SV_ST_TIMEOUT, and the next calls (sampling and greedy) are correct."""
    import time
    cfg = synth.custom_config(6, 3, 5000, "bf16", "normal")
    inp = synth.make_inputs(cfg, seed=15)
    d = to_dev(inp)
    ws = binding.make_workspace(inp.B, inp.gamma, inp.V, DEV)
    ref = oracle_sampling(inp)
    binding.sv_test_withhold_slot(True)
    try:
        t0 = time.perf_counter()
        bad = run_sampling(inp, d, ws)
        waited = time.perf_counter() - t0
    finally:
        binding.sv_test_withhold_slot(False)
    assert bad["status"] & binding.SV_ST_TIMEOUT
    assert 0.5 < waited < 30.0
    compare_sampling(inp, run_sampling(inp, d, ws), ref)
    compare_greedy(run_greedy(inp, ws=ws), oracle.greedy(inp.Lt, inp.x, inp.dtype))


def test_gamma_zero_is_plain_sampling():
    cfg = synth.custom_config(50, 0, 700, "f32", "normal", temp=1.3)
    inp = synth.make_inputs(cfg, seed=14)
    got, ref = run_sampling(inp), oracle_sampling(inp)
    compare_sampling(inp, got, ref)
    assert np.all(got["n"] == 0) and np.all(got["tokens"][:, 0] >= 0)


def test_near_tie_rate_small_sweep():
    if not NEAR_LOG:
        pytest.skip("sweep not run")
    pos = sum(s["positions"] for s in NEAR_LOG)
    near = sum(s["near"] for s in NEAR_LOG)
    print(f"\nsmall sweep: {near} near-ties over {pos} positions")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_maximum_gamma(dtype):
    """gamma = SV_MAX_GAMMA (33 rows per request: lane 0 also handles row 32)."""
    cfg = synth.custom_config(5, binding.SV_MAX_GAMMA, 3001, dtype, "normal", temp=0.7,
                              sigma_noise=0.2)
    inp = synth.make_inputs(cfg, seed=21)
    stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    assert stats["mismatches"] <= 1
    compare_greedy(run_greedy(inp), oracle.greedy(inp.Lt, inp.x, inp.dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_maximum_gamma_all_accepted(dtype):
    """gamma = SV_MAX_GAMMA with u_accept = 0, so every draft is accepted and
    the bonus token is drawn from target row 32 with u_resample[b][32] (the
    one uniform past the first 32 lanes)."""
    cfg = synth.custom_config(6, binding.SV_MAX_GAMMA, 2003, dtype, "normal", temp=0.9)
    inp = synth.make_inputs(cfg, seed=24)
    inp.u_acc[:] = 0.0
    ref = oracle_sampling(inp)
    assert np.all(ref["n"] == binding.SV_MAX_GAMMA)
    got = run_sampling(inp)
    assert np.all(got["n"] == binding.SV_MAX_GAMMA)
    stats = compare_sampling(inp, got, ref)
    assert stats["mismatches"] == 0


def test_vocabulary_of_a_million():
    """V = 1000003 (odd: unaligned rows; ~40 phase-1 chunks and 41 phase-2
    chunks per row, several rounds of partials in the draw)."""
    cfg = synth.custom_config(3, 2, 1000003, "bf16", "normal", temp=1.0)
    inp = synth.make_inputs(cfg, seed=22)
    stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    assert stats["mismatches"] <= 1


def test_many_requests_small_rows():
    """B = 3000 requests of V = 257: one chunk per row, many rows per CTA."""
    cfg = synth.custom_config(3000, 3, 257, "f32", "normal", temp=("uniform", 0.5, 1.5))
    inp = synth.make_inputs(cfg, seed=23)
    stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    assert stats["mismatches"] <= 1


@pytest.mark.parametrize("B", [75, 76, 77, 152, 153])
def test_automatic_tail_around_its_boundary(B):
    """The automatic choice (fused tail while B * 2 <= SMs, so up to B = 76 on
    152 SMs; three kernels above), checked on both sides of the boundary and
    where one SM per request is left or fewer, against the oracle."""
    cfg = synth.custom_config(B, 3, 3001, "bf16", "normal", temp=("uniform", 0.6, 1.4))
    inp = synth.make_inputs(cfg, seed=50 + B)
    binding.sv_set_tail(0)
    try:
        stats = compare_sampling(inp, run_sampling(inp), oracle_sampling(inp))
    finally:
        binding.sv_set_tail(_gpu_tail())
    assert stats["mismatches"] <= 1


def test_cuda_graph_capture_and_replay():
    """A verification call captured in a CUDA graph (its programmatic launches
    become graph edges) and replayed on new inputs copied into the captured
    buffers gives the oracle's results each time."""
    cfg = synth.custom_config(9, 4, 6007, "bf16", "mix", temp=0.9)
    inps = [synth.make_inputs(cfg, seed=40 + k) for k in range(3)]
    d = to_dev(inps[0])
    B, g = inps[0].B, inps[0].gamma
    tok = torch.full((B, g + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = binding.make_workspace(B, g, inps[0].V, DEV)
    binding.spec_verify(d["Lt"], d["Ld"], d["x"], d["u_acc"], d["u_res"], d["temp"], tok, n, ws,
                        st)  # first call outside the capture (per-device set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            binding.spec_verify(d["Lt"], d["Ld"], d["x"], d["u_acc"], d["u_res"], d["temp"], tok,
                                n, ws, st)
    torch.cuda.synchronize()
    for inp in inps:
        nd = to_dev(inp)
        for k in d:
            d[k].copy_(nd[k])
        graph.replay()
        torch.cuda.synchronize()
        got = dict(tokens=tok.cpu().numpy(), n=n.cpu().numpy(),
                   p=np.zeros((B, g, 2), np.float32), Z=np.zeros(B, np.float32),
                   status=int(st.item()))
        ref = oracle_sampling(inp)
        assert_same_or_valid(inp, got, ref)
        assert got["status"] == 0
