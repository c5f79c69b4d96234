"""The no-allocation entry point, spec_verify_noalloc, against the regular
spec_verify (GPU).

spec_verify_noalloc serves callers that may not allocate device memory (a
plugin inside a framework that owns all GPU memory, a loop that cannot afford
cudaMalloc's implicit synchronisation): it runs the same verification kernel
on a scratch array built into the library instead of a caller workspace.  It
must give exactly the tokens and counts of spec_verify, call after call, on
the same inputs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_09_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    return torch.device("cuda:0")


def _inputs(inp, dev):
    t = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).to(dev)
         for k in ("Lt", "Ld", "x", "u_acc", "u_res", "temp")}
    if inp.dtype == synth.BF16:
        t["Lt"], t["Ld"] = t["Lt"].view(torch.bfloat16), t["Ld"].view(torch.bfloat16)
    return t


def _outputs(inp, dev):
    return (torch.full((inp.B, inp.gamma + 1), -7, dtype=torch.int32, device=dev),
            torch.full((inp.B,), -7, dtype=torch.int32, device=dev),
            torch.zeros(1, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("cfg", [
    synth.custom_config(16, 5, 20011, "bf16", "zipf", temp=0.8),
    synth.custom_config(40, 3, 7001, "f32", "normal", temp=("uniform", 0.5, 1.5)),
], ids=["bf16_zipf", "f32_normal"])
def test_noalloc_matches_spec_verify_twice(cfg, dev):
    inp = synth.make_inputs(cfg, seed=31)
    t = _inputs(inp, dev)
    tok, n, st = _outputs(inp, dev)
    ws = binding.make_workspace(inp.B, inp.gamma, inp.V, dev)
    binding.spec_verify(t["Lt"], t["Ld"], t["x"], t["u_acc"], t["u_res"], t["temp"], tok, n, ws,
                        st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for _ in range(2):  # two calls in a row on the shared scratch
        tok2, n2, st2 = _outputs(inp, dev)
        binding.spec_verify_noalloc(t["Lt"], t["Ld"], t["x"], t["u_acc"], t["u_res"], t["temp"],
                                    tok2, n2, st2)
        torch.cuda.synchronize()
        assert st2.item() == 0
        assert torch.equal(tok2, tok) and torch.equal(n2, n)


def test_noalloc_rejects_sizes_beyond_its_scratch(dev):
    B, g, V = 4096, 8, 262144
    assert binding.sv_workspace_bytes(B, g, V) > binding.SV_NOALLOC_MAX_WORKSPACE
    fake = ctypes.c_void_p(0x10000000)  # never dereferenced: the size check comes first
    rc = binding.lib().spec_verify_noalloc(fake, fake, fake, fake, fake, fake, B, g, V,
                                           binding.SV_BF16, fake, fake, None, None)
    assert rc == binding.SV_ERR_WORKSPACE
