"""GPU parity of the draft side: sv_draft_sample (draft-row sampling with the
rows' normalisers) and spec_verify_cached (verification that takes those
normalisers instead of streaming the draft rows), through the C ABI, against
the fp64 oracle on the same seeded inputs.  See tests/gpu_util.py for the
comparison rules."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, compare_draft, compare_sampling, oracle_sampling, run_cached,
                      run_draft, run_sampling, to_dev)
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
    yield
    binding.sv_set_tail(0)


def _draft_case(B, n, V, dtype, kind="normal", temp=0.85, seed=0):
    inp = synth.make_inputs(synth.custom_config(B, n, V, dtype, kind, temp=temp), seed=seed)
    u = synth.draft_uniforms(B, n, seed)
    return inp, u


# ------------------------------------------------------------ draft sampling

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 3])
@pytest.mark.parametrize("V", [1, 2, 33, 1000, 4099, 20011])
def test_draft_sample_sweep(V, n, dtype):
    inp, u = _draft_case(6, n, V, dtype, seed=300 + V + n)
    got = run_draft(inp.Ld, u, inp.temp, inp.dtype)
    ref = oracle.draft_sample(inp.Ld, u, inp.temp, inp.dtype)
    stats = compare_draft(got, ref)
    assert stats["mismatches"] == 0 or stats["mismatches"] <= stats["near"]


def test_draft_sample_many_chunks_and_extreme_u():
    """Many phase-1 chunks per row (B = 1 spreads the row over every SM) and
    uniforms at the ends of [0, 1): u = 0 picks the first token with mass,
    u just below 1 the last one."""
    V = 151936
    inp, u = _draft_case(2, 4, V, "bf16", kind="mix", temp=1.0, seed=9)
    u[0, 0] = 0.0
    u[0, 1] = np.float32(1.0) - np.float32(2 ** -24)
    u[1, :] = [0.5, 1e-7, 0.999, 0.25]
    got = run_draft(inp.Ld, u, inp.temp, inp.dtype)
    ref = oracle.draft_sample(inp.Ld, u, inp.temp, inp.dtype)
    compare_draft(got, ref)


def test_draft_sample_columns():
    """One call per draft position into column i of [B][gamma] outputs gives
    what one call over all positions gives (the normaliser up to fp32
    rounding: a row's 16-byte alignment, and so the split of its elements over
    the lanes, differs between the two layouts)."""
    B, g, V = 9, 4, 3001
    inp, u = _draft_case(B, g, V, "f32", temp=("uniform", 0.5, 1.5), seed=4)
    whole = run_draft(inp.Ld, u, inp.temp, inp.dtype)
    out = (torch.full((B, g), -7, dtype=torch.int32, device=DEV),
           torch.full((B, g, 2), -7.0, dtype=torch.float32, device=DEV))
    for i in range(g):
        step = run_draft(np.ascontiguousarray(inp.Ld[:, i:i + 1]), u[:, i:i + 1], inp.temp,
                         inp.dtype, ncols=g, col=i, out=out)
    assert np.array_equal(step["tokens"], whole["tokens"])
    assert np.array_equal(step["stats"][..., 0], whole["stats"][..., 0])
    assert np.allclose(step["stats"][..., 1], whole["stats"][..., 1], rtol=1e-6, atol=0)


def test_draft_sample_invalid_rows():
    B, n, V = 5, 3, 700
    inp, u = _draft_case(B, n, V, "f32", seed=12)
    L = inp.Ld.copy()
    L[0, 1, 17] = np.nan
    L[1, 0, :] = -np.inf
    L[2, 2, 5] = np.inf
    L[3, :, ::3] = -np.inf  # legal: some entries -inf
    T = inp.temp.copy()
    T[4] = 0.0
    got = run_draft(L, u, T, inp.dtype)
    ref = oracle.draft_sample(L, u, T, inp.dtype)
    compare_draft(got, ref)
    assert np.all(got["tokens"][3] % 3 != 0)


@pytest.mark.parametrize("cid", [4, 5])
def test_draft_sample_workload_rows(cid):
    """The draft rows of the full-size workloads, sampled at the workload's
    temperature: c4 (256 x 4 rows of 151936 bf16) and c5 (1024 x 3 rows of
    50257 fp32, per-request T)."""
    inp = synth.make_inputs(cid)
    u = synth.draft_uniforms(inp.B, inp.gamma, synth.BASE_SEED + cid)
    got = run_draft(inp.Ld, u, inp.temp, inp.dtype)
    ref = oracle.draft_sample(inp.Ld, u, inp.temp, inp.dtype)
    # rows whose chosen token sits within 1e-6 of u in the CDF are flagged
    # (at low temperature most of the vocabulary has probability far below
    # 1e-6, so c5 flags several percent of its rows); a token that differs
    # there must still be a valid draw for u
    stats = compare_draft(got, ref, L=inp.Ld, dtype=inp.dtype, temp=inp.temp, u=u)
    print(f"\n{inp.name} draft rows: {stats}")
    assert stats["mismatches"] <= max(1, 0.05 * stats["near"])


# ------------------------------------------------------- cached verification

def _with_tokens(inp: synth.Inputs, x: np.ndarray) -> synth.Inputs:
    return dataclasses.replace(inp, x=np.ascontiguousarray(x, dtype=np.int32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("gamma", [0, 1, 4])
@pytest.mark.parametrize("V", [1, 33, 4099, 20011])
def test_cached_verify_with_oracle_stats(V, gamma, dtype):
    """spec_verify_cached given the oracle's draft normalisers (rounded to
    fp32) matches the oracle's verification."""
    inp = synth.make_inputs(synth.custom_config(7, gamma, V, dtype, "normal", temp=0.9),
                            seed=500 + V + gamma)
    ds = oracle.draft_sample(inp.Ld, np.zeros((inp.B, gamma), np.float32), inp.temp, inp.dtype)
    stats = np.stack([ds["m"], ds["S"]], axis=-1).astype(np.float32)
    compare_sampling(inp, run_cached(inp, stats), oracle_sampling(inp))


@pytest.mark.parametrize("cid", [1, 3, 4, 5])
def test_draft_then_cached_verify_pipeline(cid):
    """The draft side and verification chained on the GPU: sv_draft_sample
    draws x and the normalisers from the draft rows, spec_verify_cached
    verifies with them; the oracle draws x from the same rows and uniforms
    (the tokens must agree) and verifies them the plain way."""
    inp = synth.make_inputs(cid)
    u = synth.draft_uniforms(inp.B, inp.gamma, synth.BASE_SEED + cid)
    ds_gpu = run_draft(inp.Ld, u, inp.temp, inp.dtype)
    ds_ref = oracle.draft_sample(inp.Ld, u, inp.temp, inp.dtype)
    dstats = compare_draft(ds_gpu, ds_ref, L=inp.Ld, dtype=inp.dtype, temp=inp.temp, u=u)
    same_x = np.all(ds_gpu["tokens"] == ds_ref["tokens"], axis=1)
    ref_inp = _with_tokens(inp, ds_ref["tokens"])
    got = run_cached(_with_tokens(inp, ds_gpu["tokens"]), ds_gpu["stats"])
    ref = oracle_sampling(ref_inp)
    keep = same_x  # requests whose draft tokens differ (near CDF edges) are compared no further
    sub = dataclasses.replace(ref_inp, B=int(keep.sum()))
    got_k = {k: (v[keep] if isinstance(v, np.ndarray) else v) for k, v in got.items()}
    ref_k = {k: v[keep] for k, v in ref.items()}
    stats = compare_sampling(sub, got_k, ref_k)
    print(f"\n{inp.name} draft+cached: draft {dstats} verify {stats}")
    assert keep.sum() >= inp.B - max(1, dstats["near"])
    assert stats["mismatches"] <= max(1.0, 1e-4 * stats["positions"])


def test_cached_equals_streaming_path():
    """With the GPU's own normalisers, the cached path and the streaming path
    verify the same tokens (c4 rows at B = 64; both checked against the oracle)."""
    inp = synth.make_inputs(4, B=64)
    u = synth.draft_uniforms(inp.B, inp.gamma, synth.BASE_SEED + 4)
    ds = run_draft(inp.Ld, u, inp.temp, inp.dtype)  # the normalisers do not depend on u
    inp = _with_tokens(inp, oracle.draft_sample(inp.Ld, u, inp.temp, inp.dtype)["tokens"])
    ref = oracle_sampling(inp)
    a = compare_sampling(inp, run_sampling(inp), ref)
    b = compare_sampling(inp, run_cached(inp, ds["stats"]), ref)
    assert a["mismatches"] <= 1 and b["mismatches"] <= 1


def test_cached_invalid_stats_isolated():
    B, g, V = 6, 3, 900
    inp = synth.make_inputs(synth.custom_config(B, g, V, "f32", "normal", temp=1.0), seed=8)
    ds = oracle.draft_sample(inp.Ld, np.zeros((B, g), np.float32), inp.temp, inp.dtype)
    stats = np.stack([ds["m"], ds["S"]], axis=-1).astype(np.float32)
    stats[1, 0, 1] = np.nan
    stats[2, 2, 1] = 0.0
    stats[3, 1, 0] = np.inf
    got = run_cached(inp, stats)
    ref = oracle_sampling(inp)
    for b in (1, 2, 3):
        assert got["n"][b] == 0 and np.all(got["tokens"][b] == -1)
    assert got["status"] == binding.SV_ST_NONFINITE
    ok = np.array([0, 4, 5])
    assert np.array_equal(got["tokens"][ok], ref["tokens"][ok]) or \
        np.all(ref["flags"][ok] & oracle.NEAR_ANY)


def test_draft_sample_limits():
    """n = SV_MAX_GAMMA rows per request, a vocabulary of a million (many
    rounds of partials in the sampler), and many small rows."""
    for (B, n, V, dt, seed) in ((3, binding.SV_MAX_GAMMA, 2003, "f32", 31),
                                (2, 2, 1000003, "bf16", 32), (1500, 2, 129, "bf16", 33)):
        inp, u = _draft_case(B, n, V, dt, seed=seed)
        got = run_draft(inp.Ld, u, inp.temp, inp.dtype)
        ref = oracle.draft_sample(inp.Ld, u, inp.temp, inp.dtype)
        compare_draft(got, ref, L=inp.Ld, dtype=inp.dtype, temp=inp.temp, u=u)
