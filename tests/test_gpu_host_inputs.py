"""fa_constrained_step_host: the step with the probabilities and committed tokens in host
memory, copied in up to eight pieces of consecutive positions (the first a thirty-second
of the batch, each next one 1.4 times larger) that overlap the emission reweighting.  Its outputs must equal those of fa_constrained_step
on the same inputs already on the device, bit for bit (the same kernels and row-block layout
over the same values), for batches split into pieces that start and end inside sequences, on
the shared-memory-row reweight (random DFA) and the cell-store one (layered chain)."""
import numpy as np
import pytest

from constrained_decoding_diffusion_gb300 import synth

pytestmark = pytest.mark.gpu


def _outputs(B, L, k):
    import torch
    return dict(tokens=torch.empty((B, L), dtype=torch.int32, device="cuda"),
                logZ=torch.empty((B,), dtype=torch.float64, device="cuda"),
                marg=torch.empty((B, L), dtype=torch.float32, device="cuda"),
                commit_idx=torch.empty((B, k), dtype=torch.int32, device="cuda"),
                row_status=torch.empty((B,), dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("name,B", [("random_dfa_S64_L128", 5), ("layered_chain_S256_L256", 4),
                                    ("real_number_L6", 11)])
def test_host_inputs_match_device_inputs(name, B):
    import torch
    from constrained_decoding_diffusion_gb300 import native
    native.load()
    w = synth.workload(name, B=B)
    aut = native.fa_compile(w.fa)
    probs = w.probs()
    h_probs = torch.from_numpy(probs).pin_memory()
    h_com = torch.from_numpy(np.ascontiguousarray(w.committed, np.int32)).pin_memory()
    ws = torch.empty(native.fa_step_workspace_bytes(aut, w.B, w.L), dtype=torch.uint8, device="cuda")
    ref = _outputs(w.B, w.L, w.k)
    native.fa_constrained_step(aut, h_probs.cuda(), h_com.cuda(), 9, 2, w.k, 0, w.window, ws, ref["tokens"],
                               ref["logZ"], ref["marg"], ref["commit_idx"], ref["row_status"])
    got = _outputs(w.B, w.L, w.k)
    d_probs = torch.full(probs.shape, float("nan"), dtype=torch.float32, device="cuda")
    d_com = torch.full(w.committed.shape, -7, dtype=torch.int32, device="cuda")
    for _ in range(2):          # twice in a row: the copy stream and its events are reused
        native.fa_constrained_step_host(aut, h_probs, h_com, d_probs, d_com, 9, 2, w.k, 0, w.window, ws,
                                        got["tokens"], got["logZ"], got["marg"], got["commit_idx"],
                                        got["row_status"])
        torch.cuda.synchronize()
        assert torch.equal(d_probs.cpu(), h_probs) and torch.equal(d_com.cpu(), h_com)
        for key in ref:
            assert torch.equal(got[key], ref[key]), key
    assert (ref["row_status"].cpu().numpy() == 0).all()


def test_host_inputs_reject_null_buffers():
    from constrained_decoding_diffusion_gb300 import native
    native.load()
    w = synth.workload("real_number_L6")
    aut = native.fa_compile(w.fa)
    rc = native._lib.fa_constrained_step_host(aut.handle, 1, w.L, None, None, None, None, 1, 0, w.k, 0, w.L, None, 0,
                                              None, None, None, None, None, None)
    assert rc == native.FA_ERR_INVALID_ARG
