"""GPU parity of token-tree verification (sv_tree_verify) through the C ABI
against the fp64 oracle on the same seeded inputs.

Comparison rule: requests the oracle does not flag match exactly (accepted
count, emitted tokens, accepted nodes, status).  A flagged request (an accept
test with |u - ratio| < 1e-6, a draw within 1e-6 of a CDF boundary, or a
vanished residual) may take another branch; its GPU result must still be a
valid walk: a chain of children from the root, each emitting its own token,
then one token in [0, V).  The same 1e-6 as the chain rule: the kernel sums
each row in float pairs over fp32 vector sums, so a residual mass S_j carries
a relative error near 1e-7, which the next ratio divides by S_j.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_09_gb300 import binding, synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TREE_EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield
    binding.sv_tree_set_cluster(0)
    binding.sv_tree_set_warps(0)


def _t(a):
    return torch.from_numpy(np.array(a, order="C", copy=True)).to(DEV)


def run_tree(ti: synth.TreeInputs, ld_offset: int = 0, no_draft: bool = False) -> dict:
    Lt, Ld = _t(ti.Lt), _t(ti.Ld)
    if ld_offset:  # the draft rows at a shifted address (another 16-byte alignment)
        buf = torch.empty(Ld.numel() + ld_offset, dtype=Ld.dtype, device=DEV)
        buf[ld_offset:].copy_(Ld.reshape(-1))
        Ld = buf[ld_offset:].view(Ld.shape)
    if ti.dtype == synth.BF16:
        Lt, Ld = Lt.view(torch.bfloat16), Ld.view(torch.bfloat16)
    B, N = ti.B, ti.N
    tok = torch.full((B, N), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    nodes = torch.full((B, N), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.sv_tree_verify(Lt, None if no_draft else Ld, _t(ti.parent), _t(ti.tokens),
                           None if no_draft else _t(ti.u_acc), _t(ti.u_res), _t(ti.temp), tok, n,
                           nodes, st)
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), n=n.cpu().numpy(), nodes=nodes.cpu().numpy(),
                status=int(st.item()))


def oracle_tree(ti: synth.TreeInputs) -> dict:
    return oracle.tree_verify(ti.Lt, ti.Ld, ti.parent, ti.tokens, ti.u_acc, ti.u_res, ti.temp,
                              ti.dtype, near_eps=TREE_EPS)


def _valid_walk(ti, b, got):
    k = int(got["n"][b])
    if not (0 <= k < ti.N):
        return False
    prev = 0
    for i in range(k):
        c = int(got["nodes"][b, i])
        if not (0 < c < ti.N and ti.parent[b, c] == prev and got["tokens"][b, i] == ti.tokens[b, c]):
            return False
        prev = c
    return (0 <= got["tokens"][b, k] < ti.V and np.all(got["tokens"][b, k + 1:] == -1)
            and np.all(got["nodes"][b, k:] == -1))


def compare_tree(ti, got, ref) -> dict:
    near = (ref["flags"] & oracle.NEAR_ANY) != 0
    invalid = (ref["flags"] & oracle.INVALID_ANY) != 0
    same = ((got["n"] == ref["n"]) & np.all(got["tokens"] == ref["tokens"], axis=1)
            & np.all(got["nodes"] == ref["nodes"], axis=1))
    bad = ~same & ~near
    assert not bad.any(), (np.nonzero(bad)[0][:8], got["tokens"][bad][:2], ref["tokens"][bad][:2],
                           got["nodes"][bad][:2], ref["nodes"][bad][:2])
    for b in np.nonzero(~same & near & ~invalid)[0]:
        assert _valid_walk(ti, b, got), b
    want = 0
    if (ref["flags"] & oracle.INVALID_NONFINITE).any():
        want |= binding.SV_ST_NONFINITE
    if (ref["flags"] & oracle.INVALID_TOKEN).any():
        want |= binding.SV_ST_BAD_TOKEN
    if (ref["flags"] & oracle.INVALID_TEMP).any():
        want |= binding.SV_ST_BAD_TEMP
    assert got["status"] & ~binding.SV_ST_DEGENERATE == want
    return dict(requests=ti.B, near=int(near.sum()), differ=int((~same).sum()),
                accepted=float(ref["n"][~invalid].mean()) if (~invalid).any() else 0.0)


SHAPES = {
    "chain4": np.arange(-1, 4, dtype=np.int32),
    "b3211": synth.tree_parents((3, 2, 1, 1)),
    "star6": np.array([-1, 0, 0, 0, 0, 0, 0], np.int32),
    "random20": synth.random_parents(20, 5),
}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("V", [1, 2, 33, 1000, 4099, 20011])
def test_tree_sweep(V, shape, dtype):
    cfg = synth.custom_config(6, 0, V, dtype, "normal", temp=("uniform", 0.6, 1.4))
    ti = synth.make_tree_inputs(cfg, SHAPES[shape], seed=700 + V)
    compare_tree(ti, run_tree(ti), oracle_tree(ti))


@pytest.mark.parametrize("warps", [8, 16])
@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 8])
def test_tree_cluster_sizes(ctas, warps):
    """Every cluster size and CTA width gives the oracle's walk (the segment
    split differs, so only rounding may move; flagged requests excepted)."""
    cfg = synth.custom_config(12, 0, 30011, "bf16", "mix", temp=1.0)
    ti = synth.make_tree_inputs(cfg, SHAPES["b3211"], seed=71)
    binding.sv_tree_set_cluster(ctas)
    binding.sv_tree_set_warps(warps)
    try:
        compare_tree(ti, run_tree(ti), oracle_tree(ti))
    finally:
        binding.sv_tree_set_cluster(0)
        binding.sv_tree_set_warps(0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("V", [1, 33, 4099, 20011])
def test_tree_sweep_sixteen_warps(V, shape, dtype):
    """The sweep's cases with CTAs of 16 warps (the automatic choice takes 8
    at these batch sizes)."""
    cfg = synth.custom_config(6, 0, V, dtype, "normal", temp=("uniform", 0.6, 1.4))
    ti = synth.make_tree_inputs(cfg, SHAPES[shape], seed=700 + V)
    binding.sv_tree_set_warps(16)
    try:
        compare_tree(ti, run_tree(ti), oracle_tree(ti))
    finally:
        binding.sv_tree_set_warps(0)



def test_tree_star_many_rejections():
    """A root with 12 children and a weak draft: most requests reject several
    siblings in a row, so many residuals are formed one after another."""
    parent = np.array([-1] + [0] * 12, np.int32)
    cfg = synth.custom_config(40, 0, 5003, "f32", "mix", temp=1.0, weights=(0.05, 0.2))
    ti = synth.make_tree_inputs(cfg, parent, seed=72)
    stats = compare_tree(ti, run_tree(ti), oracle_tree(ti))
    print(f"\nstar12: {stats}")


def test_tree_unaligned_draft_rows():
    """Draft rows at an address whose 16-byte alignment differs from the
    target rows' (the scalar path) give the same walks."""
    for dtype, V in (("bf16", 4099), ("f32", 1001)):
        cfg = synth.custom_config(5, 0, V, dtype, "normal", temp=0.9)
        ti = synth.make_tree_inputs(cfg, SHAPES["random20"], seed=73)
        ref = oracle_tree(ti)
        compare_tree(ti, run_tree(ti, ld_offset=1), ref)
        compare_tree(ti, run_tree(ti, ld_offset=3), ref)


def test_tree_single_node():
    """N = 1: one draw from the root's target row; no draft rows needed."""
    cfg = synth.custom_config(9, 0, 3001, "bf16", "normal", temp=1.1)
    ti = synth.make_tree_inputs(cfg, np.array([-1], np.int32), seed=74)
    got = run_tree(ti, no_draft=True)
    compare_tree(ti, got, oracle_tree(ti))
    assert np.all(got["n"] == 0)


def test_tree_invalid_and_unread_rows():
    """Readings T2/T3: malformed trees, bad tokens and temperatures, and NaN
    in a row the walk reads invalidate only their request; NaN in the rows of
    nodes the walk never visits, and in every leaf's draft row, changes
    nothing."""
    cfg = synth.custom_config(8, 0, 2000, "f32", "normal", temp=1.0)
    ti = synth.make_tree_inputs(cfg, SHAPES["b3211"], seed=75, leaf_fill=np.nan)
    ref0 = oracle_tree(ti)
    # NaN in every row off request 0's walk: its result must not change
    visited = {0} | {int(c) for c in ref0["nodes"][0] if c >= 0}
    for n in range(ti.N):
        if n not in visited:
            ti.Lt[0, n, 7] = np.nan
            ti.Ld[0, n, 9] = np.nan
    ti.parent[1, 5] = 7        # a parent after the node
    ti.tokens[2, 3] = ti.V     # token out of range
    ti.Lt[3, 0, 11] = np.inf   # the root row is always read
    ti.temp[4] = np.nan
    ti.Ld[5, 0, :] = -np.inf   # the root's draft row is read (it has children)
    ref = oracle_tree(ti)
    assert ref["n"][0] == ref0["n"][0] and np.array_equal(ref["tokens"][0], ref0["tokens"][0])
    got = run_tree(ti)
    compare_tree(ti, got, ref)
    for b in (1, 2, 3, 4, 5):
        assert got["n"][b] == 0 and np.all(got["tokens"][b] == -1)
    assert got["status"] == (binding.SV_ST_BAD_TOKEN | binding.SV_ST_NONFINITE
                             | binding.SV_ST_BAD_TEMP)


def test_tree_limits():
    """The largest tree (SV_TREE_MAX_N nodes, up to 8 children), many requests
    in several waves of CTAs, and a vocabulary of a million."""
    cfg = synth.custom_config(3, 0, 257, "bf16", "normal", temp=0.8)
    ti = synth.make_tree_inputs(cfg, synth.random_parents(binding.SV_TREE_MAX_N, 6, 8), seed=76)
    compare_tree(ti, run_tree(ti), oracle_tree(ti))
    cfg = synth.custom_config(700, 0, 100, "f32", "normal", temp=1.0)
    ti = synth.make_tree_inputs(cfg, SHAPES["b3211"], seed=77)
    compare_tree(ti, run_tree(ti), oracle_tree(ti))
    cfg = synth.custom_config(2, 0, 1000003, "bf16", "normal", temp=1.0)
    ti = synth.make_tree_inputs(cfg, SHAPES["chain4"], seed=78)
    compare_tree(ti, run_tree(ti), oracle_tree(ti))


def test_tree_chain_matches_spec_verify():
    """A chain tree is plain verification: the tree kernel and the chain
    kernels give the same tokens on the same rows (both checked against the
    oracle)."""
    from gpu_util import compare_sampling, oracle_sampling, run_sampling
    inp = synth.make_inputs(synth.custom_config(16, 4, 20011, "bf16", "mix", temp=1.0), seed=79)
    B, g, V = inp.B, inp.gamma, inp.V
    Ldt = np.concatenate([inp.Ld, np.zeros((B, 1, V), inp.Ld.dtype)], axis=1)
    ti = synth.TreeInputs(inp.Lt, Ldt, np.ascontiguousarray(
        np.broadcast_to(np.arange(-1, g, dtype=np.int32), (B, g + 1))),
        np.concatenate([np.zeros((B, 1), np.int32), inp.x], axis=1),
        np.concatenate([np.zeros((B, 1), np.float32), inp.u_acc], axis=1), inp.u_res,
        inp.temp, inp.dtype, B, g + 1, V)
    ref = oracle_sampling(inp)
    chain = run_sampling(inp)
    compare_sampling(inp, chain, ref)
    tree = run_tree(ti)
    compare_tree(ti, tree, oracle_tree(ti))
    near = (ref["flags"] & oracle.NEAR_ANY) != 0
    assert np.array_equal(tree["tokens"][~near], chain["tokens"][~near])


def test_tree_workload():
    """The token-tree workload at full size: 64 requests, 22-node trees
    (3, 2, 1, 1 children per level), V = 151936 bf16, draft mixtures
    w = 0.3 / 0.6 / 0.9 of the target."""
    ti = synth.make_tree_inputs(synth.TREE_WORKLOAD, synth.tree_parents(
        synth.TREE_WORKLOAD["branching"]))
    stats = compare_tree(ti, run_tree(ti), oracle_tree(ti))
    print(f"\n{ti.name}: {stats}")
    assert stats["near"] <= ti.B // 8


@pytest.mark.parametrize("seed", range(int(os.environ.get("SV_TREE_FUZZ_SEEDS", "24"))))
def test_tree_fuzz(seed):
    """Random trees, batches, vocabularies, dtypes, recipes, temperatures and
    kernel shapes (CTA width, cluster size: automatic or forced) against the
    oracle."""
    rng = np.random.default_rng(4000 + seed)
    B = int(rng.integers(1, 40))
    N = int(rng.integers(1, 48))
    V = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 5000)),
                        int(rng.integers(5000, 40000))]))
    dtype = str(rng.choice(["f32", "bf16"]))
    kind = str(rng.choice(["normal", "zipf", "mix"]))
    temp = ("uniform", 0.3, 2.0) if rng.random() < 0.5 else float(rng.uniform(0.2, 3.0))
    cfg = synth.custom_config(B, 0, V, dtype, kind, temp=temp)
    parents = synth.random_parents(N, 5000 + seed, int(rng.integers(1, 6)))
    ti = synth.make_tree_inputs(cfg, parents, seed=6000 + seed)
    warps = int(rng.choice([0, 8, 16]))
    ctas = int(rng.choice([0, 0, 1, 2, 3, 4, 8]))
    binding.sv_tree_set_warps(warps)
    binding.sv_tree_set_cluster(ctas)
    try:
        compare_tree(ti, run_tree(ti), oracle_tree(ti))
    finally:
        binding.sv_tree_set_warps(0)
        binding.sv_tree_set_cluster(0)
