"""GB300 (sm_103a) speculative-decoding verification.

The product is libspecverify.so (C ABI in include/specverify.h, kernels in
csrc/specverify.cu); `binding` is its thin Python marshalling layer and
`synth` draws seeded synthetic inputs.  Importing the package loads nothing;
the binding's names are resolved on first use.
"""
_BINDING_NAMES = {"spec_verify", "spec_verify_diag", "spec_verify_greedy", "sv_workspace_bytes",
                  "sv_workspace_init", "sv_set_tuning", "make_workspace", "lib",
                  "SpecVerifyError"}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
