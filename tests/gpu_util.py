"""Helpers shared by the GPU parity tests: move synthetic inputs to the
device, call the library through its C ABI (binding), and compare with the
oracle under the parity rules:

  * tokens and accepted counts bit-exact, except at requests the oracle flags
    as near-ties (|u_acc - r| < 1e-6 at a decided position, the u_resample
    CDF boundary within 1e-6, or a vanished residual);
  * P_t(x_i), P_d(x_i) within relative 1e-5;
  * the final draw's mass Z within relative 1e-5 plus absolute 1e-6 (the
    residual max(0, P_t - P_d) loses relative precision by cancellation where
    the two rows agree; each fp32 term carries ~1e-7 relative error);
  * invalid requests: accepted count 0, tokens all -1, matching status bits;
  * greedy: bit-exact everywhere.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_verification_09_gb300 import binding, synth

DEV = torch.device("cuda:0")
P_RTOL = 1e-5
Z_RTOL, Z_ATOL = 1e-5, 1e-6


def to_dev(inp: synth.Inputs, device=DEV) -> dict:
    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    Lt, Ld = t(inp.Lt), t(inp.Ld)
    if inp.dtype == synth.BF16:
        Lt, Ld = Lt.view(torch.bfloat16), Ld.view(torch.bfloat16)
    return dict(Lt=Lt, Ld=Ld, x=t(inp.x), u_acc=t(inp.u_acc), u_res=t(inp.u_res), temp=t(inp.temp))


def run_sampling(inp: synth.Inputs, d: dict | None = None, ws=None, stream=None) -> dict:
    d = d or to_dev(inp)
    B, g = inp.B, inp.gamma
    tok = torch.full((B, g + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    p = torch.full((B, g, 2), -7.0, dtype=torch.float32, device=DEV)
    Z = torch.full((B,), -7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = binding.make_workspace(B, g, inp.V, DEV)
    binding.spec_verify_diag(d["Lt"], d["Ld"] if g > 0 else None, d["x"] if g > 0 else None,
                             d["u_acc"] if g > 0 else None, d["u_res"], d["temp"], tok, n, p, Z,
                             ws, st, stream)
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), n=n.cpu().numpy(), p=p.cpu().numpy(),
                Z=Z.cpu().numpy(), status=int(st.item()))


def run_greedy(inp: synth.Inputs, x=None, d: dict | None = None, ws=None) -> dict:
    d = d or to_dev(inp)
    B, g = inp.B, inp.gamma
    xd = d["x"] if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    tok = torch.full((B, g + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = binding.make_workspace(B, g, inp.V, DEV)
    binding.spec_verify_greedy(d["Lt"], xd if g > 0 else None, tok, n, ws, st)
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), n=n.cpu().numpy(), status=int(st.item()))


def oracle_sampling(inp: synth.Inputs) -> dict:
    return oracle.verify(inp.Lt, inp.Ld, inp.x, inp.u_acc, inp.u_res, inp.temp, inp.dtype)


def expected_status(flags: np.ndarray) -> int:
    s = 0
    if np.any(flags & oracle.INVALID_NONFINITE):
        s |= binding.SV_ST_NONFINITE
    if np.any(flags & oracle.INVALID_TOKEN):
        s |= binding.SV_ST_BAD_TOKEN
    if np.any(flags & oracle.INVALID_TEMP):
        s |= binding.SV_ST_BAD_TEMP
    return s


def _row_probs(L, dtype: int, T: float) -> np.ndarray:
    """softmax(l / T) of one stored logit row, in fp64."""
    w = synth.widen(L, dtype).astype(np.float64) / float(T)
    m = np.max(w)
    if not np.isfinite(m):
        return np.zeros_like(w)
    p = np.exp(w - m)
    return p / p.sum()


def check_valid_draw(inp: synth.Inputs, got: dict, ref: dict, b: int) -> None:
    """A request whose GPU result differs from the oracle's at a flagged
    near-tie must still be a result the rule allows, decided within the
    1e-6 window:
      * the outputs have the rule's shape: the accepted drafts, one drawn
        token, then -1;
      * where the accepted counts differ, the first position decided
        differently has |u_accept - r| < 1e-6 (r the oracle's fp64 ratio);
      * the drawn token's interval of the fp64 CDF it is drawn from (the
        residual of row k, the target row gamma for the bonus, the target
        row k when the residual vanishes) contains u_resample[b][k] to
        within 1e-6."""
    g, tok = inp.gamma, got["tokens"][b]
    kg, kr = int(got["n"][b]), int(ref["n"][b])
    assert 0 <= kg <= g, (b, kg)
    assert np.array_equal(tok[:kg], inp.x[b, :kg]) and np.all(tok[kg + 1:] == -1), (b, tok)
    if kg != kr:
        i = min(kg, kr)
        pt, pd = float(ref["pt"][b, i]), float(ref["pd"][b, i])
        r = 1.0 if pd == 0.0 else min(1.0, pt / pd)
        assert abs(float(inp.u_acc[b, i]) - r) < oracle.NEAR_EPS, (b, i, float(inp.u_acc[b, i]), r)
    T = float(inp.temp[b])
    row_t = inp.Lt[b, kg]
    w = _row_probs(row_t, inp.dtype, T)
    if kg < g:
        res = np.maximum(0.0, w - _row_probs(inp.Ld[b, kg], inp.dtype, T))
        if res.sum() > 0.0:
            w = res
    c = np.cumsum(w) / w.sum()
    v = int(tok[kg])
    assert 0 <= v < inp.V and w[v] > 0.0, (b, v)
    lo, hi = (c[v - 1] if v > 0 else 0.0), c[v]
    u = float(inp.u_res[b, kg])
    assert lo - oracle.NEAR_EPS <= u < hi + oracle.NEAR_EPS, (b, kg, v, lo, u, hi)


def compare_sampling(inp: synth.Inputs, got: dict, ref: dict) -> dict:
    flags = ref["flags"]
    inv = (flags & oracle.INVALID_ANY) != 0
    near = (flags & oracle.NEAR_ANY) != 0
    assert np.all(got["n"][inv] == 0) and np.all(got["tokens"][inv] == -1)
    same = np.all(got["tokens"] == ref["tokens"], axis=1) & (got["n"] == ref["n"])
    bad = ~inv & ~near & ~same
    assert not bad.any(), (f"{int(bad.sum())} mismatching requests, e.g. b={int(np.argmax(bad))}: "
                           f"gpu {got['tokens'][bad][0]} n={got['n'][bad][0]} vs oracle "
                           f"{ref['tokens'][bad][0]} n={ref['n'][bad][0]}")
    # a flagged request that differs must still be a valid draw
    for b in np.flatnonzero(~inv & near & ~same):
        check_valid_draw(inp, got, ref, int(b))
    ok = ~inv
    if inp.gamma > 0 and ok.any():
        for j, key in ((0, "pt"), (1, "pd")):
            g_, r_ = got["p"][ok, :, j].astype(np.float64), ref[key][ok]
            err = np.abs(g_ - r_) - P_RTOL * np.abs(r_) - 1e-30
            assert np.all(err <= 0), f"{key}: max rel err {np.max(np.abs(g_ - r_) / np.abs(r_))}"
    samek = ok & (got["n"] == ref["n"])
    if samek.any():
        gz, rz = got["Z"][samek].astype(np.float64), ref["Z"][samek]
        assert np.all(np.abs(gz - rz) <= Z_RTOL * np.abs(rz) + Z_ATOL), \
            f"Z: max abs err {np.max(np.abs(gz - rz))}"
    want = expected_status(flags)
    st = got["status"] & ~binding.SV_ST_DEGENERATE
    assert st == want, f"status {st:#x} != expected {want:#x}"
    near_bits = (((flags & oracle.NEAR_ACCEPT) != 0).astype(int)
                 + ((flags & oracle.NEAR_SAMPLE) != 0).astype(int)
                 + ((flags & oracle.DEGENERATE) != 0).astype(int))
    mism = ~inv & ~same
    dist = np.min(ref["dist"], axis=1)
    return dict(requests=inp.B, positions=inp.B * inp.gamma, near=int(near_bits.sum()),
                near_requests=int(near.sum()), mismatches=int(mism.sum()),
                max_mismatch_dist=float(dist[mism].max()) if mism.any() else 0.0,
                accepted=int(ref["n"][~inv].sum()))


def compare_greedy(got: dict, ref: dict) -> None:
    assert np.array_equal(got["tokens"], ref["tokens"]), "greedy tokens differ"
    assert np.array_equal(got["n"], ref["n"]), "greedy counts differ"
    want = expected_status(ref["flags"])
    assert got["status"] == want, f"status {got['status']:#x} != {want:#x}"


# ------------------------------------------------------------ draft side

S_RTOL = 1e-5  # the draft rows' normaliser S


def run_draft(L, u, temp, dtype: int, ncols: int | None = None, col: int = 0, ws=None,
              out=None) -> dict:
    """sv_draft_sample on host arrays L [B][n][V] (float32 or bf16 bits), u [B][n], temp [B];
    returns tokens [B][ncols], stats [B][ncols][2] and the status word."""
    B, n, V = L.shape
    ncols = n if ncols is None else ncols
    Ld = torch.from_numpy(np.ascontiguousarray(L)).to(DEV)
    if dtype == synth.BF16:
        Ld = Ld.view(torch.bfloat16)
    ud = torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).to(DEV)
    td = torch.from_numpy(np.ascontiguousarray(temp, dtype=np.float32)).to(DEV)
    if out is None:
        out = (torch.full((B, ncols), -7, dtype=torch.int32, device=DEV),
               torch.full((B, ncols, 2), -7.0, dtype=torch.float32, device=DEV))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = binding.make_draft_workspace(B, n, V, DEV)
    binding.sv_draft_sample(Ld, ud, td, out[0], out[1], ws, col=col, dev_status=st)
    torch.cuda.synchronize()
    return dict(tokens=out[0].cpu().numpy(), stats=out[1].cpu().numpy(), status=int(st.item()),
                out=out)


def _cdf_edges(L, dtype, temp, b, i, v):
    """fp64 CDF of draft row (b, i) of the stored logits just before and at
    token v, normalised: the interval of u that selects v."""
    w = synth.widen(L[b, i], dtype) / float(temp[b])
    p = np.exp(w - w.max())
    c = np.cumsum(p) / p.sum()
    return (c[v - 1] if v > 0 else 0.0), c[v]


def compare_draft(got: dict, ref: dict, col: int = 0, L=None, dtype=None, temp=None,
                  u=None) -> dict:
    """Draft tokens bit-exact except at rows the oracle flags as near a CDF
    edge; m exact (the stored maximum); S within relative S_RTOL; invalid rows
    -1 with NaN stats.  Given the rows (L, dtype, temp, u), a differing token
    must still be a valid draw: u within 1e-6 of the token's CDF interval."""
    n = ref["tokens"].shape[1]
    tok = got["tokens"][:, col:col + n]
    m, S = got["stats"][:, col:col + n, 0], got["stats"][:, col:col + n, 1]
    inv = (ref["flags"] & oracle.INVALID_ANY) != 0
    near = (ref["flags"] & oracle.NEAR_SAMPLE) != 0
    assert np.all(tok[inv] == -1) and np.all(np.isnan(S[inv])) and np.all(np.isnan(m[inv]))
    ok = ~inv
    assert np.all(m[ok].astype(np.float64) == ref["m"][ok]), "row maxima differ"
    rel = np.abs(S[ok].astype(np.float64) - ref["S"][ok]) / ref["S"][ok]
    assert np.all(rel <= S_RTOL), f"S: max rel err {rel.max()}"
    mism = ok & (tok != ref["tokens"])
    bad = mism & ~near
    assert not bad.any(), (f"{int(bad.sum())} draft tokens differ, e.g. "
                           f"{np.argwhere(bad)[0]}: gpu {tok[bad][0]} oracle {ref['tokens'][bad][0]}")
    if L is not None:
        for b, i in np.argwhere(mism):
            lo, hi = _cdf_edges(L, dtype, temp, b, i, int(tok[b, i]))
            uu = float(u[b, i])
            assert lo - 1e-6 <= uu < hi + 1e-6, (b, i, lo, uu, hi)
    want = 0
    if np.any(ref["flags"] & oracle.INVALID_NONFINITE):
        want |= binding.SV_ST_NONFINITE
    if np.any(ref["flags"] & oracle.INVALID_TEMP):
        want |= binding.SV_ST_BAD_TEMP
    assert got["status"] == want, f"status {got['status']:#x} != {want:#x}"
    return dict(rows=int(ok.sum()), near=int(near.sum()), mismatches=int(mism.sum()),
                max_rel_S=float(rel.max()) if rel.size else 0.0)


def run_cached(inp: synth.Inputs, stats: np.ndarray, d: dict | None = None, ws=None) -> dict:
    """spec_verify_cached with the draft normalisers `stats` [B][gamma][2]."""
    d = d or to_dev(inp)
    B, g = inp.B, inp.gamma
    tok = torch.full((B, g + 1), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    p = torch.full((B, g, 2), -7.0, dtype=torch.float32, device=DEV)
    Z = torch.full((B,), -7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd = torch.from_numpy(np.ascontiguousarray(stats, dtype=np.float32)).to(DEV)
    if ws is None:
        ws = binding.make_workspace(B, g, inp.V, DEV)
    binding.spec_verify_cached(d["Lt"], d["Ld"] if g > 0 else None, d["x"] if g > 0 else None,
                               sd if g > 0 else None, d["u_acc"] if g > 0 else None, d["u_res"],
                               d["temp"], tok, n, ws, out_p=p, out_Z=Z, dev_status=st)
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), n=n.cpu().numpy(), p=p.cpu().numpy(),
                Z=Z.cpu().numpy(), status=int(st.item()))
