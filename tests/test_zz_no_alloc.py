"""The allocation-free entry point, for callers that may not allocate device memory.

fa_constrained_step_noalloc takes the same inputs and outputs as fa_constrained_step but
no workspace: an engine whose memory pool owns the device, or a loop where cudaMalloc
would synchronise the GPU, can still run the step.  Its scratch is a fixed array built
into the library.  This file sorts last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

from constrained_decoding_diffusion_gb300 import synth

pytestmark = pytest.mark.gpu

LOGZ_RTOL = 1e-5
MARG_ATOL = 1e-5


def _outputs(B, L, k):
    import torch
    return dict(tokens=torch.empty((B, L), dtype=torch.int32, device="cuda"),
                logZ=torch.empty((B,), dtype=torch.float64, device="cuda"),
                marg=torch.empty((B, L), dtype=torch.float32, device="cuda"),
                commit_idx=torch.empty((B, k), dtype=torch.int32, device="cuda"),
                row_status=torch.empty((B,), dtype=torch.int32, device="cuda"))


def _same(a, b):
    assert np.array_equal(a["row_status"].cpu().numpy(), b["row_status"].cpu().numpy())
    assert np.array_equal(a["tokens"].cpu().numpy(), b["tokens"].cpu().numpy())
    assert np.array_equal(a["commit_idx"].cpu().numpy(), b["commit_idx"].cpu().numpy())
    la, lb = a["logZ"].cpu().numpy(), b["logZ"].cpu().numpy()
    assert np.all(np.abs(la - lb) <= LOGZ_RTOL * np.maximum(1.0, np.abs(lb)))
    np.testing.assert_allclose(a["marg"].cpu().numpy(), b["marg"].cpu().numpy(), rtol=0, atol=MARG_ATOL)


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    """Three calls in a row on the shared scratch: the larger random-DFA layout, then the
    small real-number one over its leftovers, then the random DFA again over the real-number
    call's leftovers.  Each matches the workspace entry point: bit for bit on tokens, commit
    set and status, within the oracle tolerances on logZ and the marginals."""
    import torch
    from constrained_decoding_diffusion_gb300 import native
    assert torch.cuda.is_available()
    native.load()
    first = synth.workload("random_dfa_S64_L128")
    cases = [first, synth.workload("real_number_L6", B=3), first]
    for call, w in enumerate(cases):
        aut = native.fa_compile(w.fa)
        probs = torch.from_numpy(w.probs(step=call)).cuda()
        com = torch.from_numpy(w.committed).cuda()
        ref = _outputs(w.B, w.L, w.k)
        ws = torch.empty(native.fa_step_workspace_bytes(aut, w.B, w.L), dtype=torch.uint8, device="cuda")
        native.fa_constrained_step(aut, probs, com, 77, call, w.k, 0, w.window, ws, ref["tokens"], ref["logZ"],
                                   ref["marg"], ref["commit_idx"], ref["row_status"])
        got = _outputs(w.B, w.L, w.k)
        native.fa_constrained_step_noalloc(aut, probs, com, 77, call, w.k, 0, w.window, got["tokens"], got["logZ"],
                                           got["marg"], got["commit_idx"], got["row_status"])
        torch.cuda.synchronize()
        assert (ref["row_status"].cpu().numpy() == 0).all()
        _same(got, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    from constrained_decoding_diffusion_gb300 import native
    native.load()
    w = synth.workload("random_dfa_S64_L128")
    aut = native.fa_compile(w.fa)
    B = 8                                           # 8 sequences of L=128 need ~35 MB of scratch
    assert native.fa_step_workspace_bytes(aut, B, w.L) > native.NOALLOC_SCRATCH_BYTES
    probs = torch.full((B, w.L, w.V), 1.0 / w.V, device="cuda")
    com = torch.full((B, w.L), -1, dtype=torch.int32, device="cuda")
    out = _outputs(B, w.L, w.k)
    with pytest.raises(native.FaError) as ei:
        native.fa_constrained_step_noalloc(aut, probs, com, 1, 0, w.k, 0, w.L, out["tokens"], out["logZ"],
                                           out["marg"], out["commit_idx"], out["row_status"])
    assert ei.value.code == native.FA_ERR_WORKSPACE_TOO_SMALL
    assert "scratch" in str(ei.value)


def test_noalloc_rejects_out_of_range_batch_as_invalid():
    import torch
    from constrained_decoding_diffusion_gb300 import native
    native.load()
    w = synth.workload("real_number_L6")
    aut = native.fa_compile(w.fa)
    lib = native._lib
    rc = lib.fa_constrained_step_noalloc(aut.handle, 70000, w.L, None, None, 1, 0, w.k, 0, w.L, None, None, None,
                                         None, None, None)
    assert rc == native.FA_ERR_INVALID_ARG
    assert "out of range" in lib.fa_last_error().decode()
    rc = lib.fa_constrained_step_noalloc(aut.handle, 1, w.L, None, None, 1, 0, -1, 0, w.L, None, None, None,
                                         None, None, None)
    assert rc == native.FA_ERR_INVALID_ARG
