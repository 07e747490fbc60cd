"""The timeout path of the persistent full-vocabulary chain kernel, made to
run out without faulting anything: the idle limit (how many polls a warp
makes while none of its work is ready) is set to one poll, so warps give up
while others still work.  A warp leaves only after the bulk copies it has in
flight have landed; the call reports SPEC_FLAG_TIMEOUT in the workspace's
status word.  With a fresh workspace and the default limit the results are
exact again.  No wait on a bulk copy is made to run out."""
import pytest
import torch

from parity import compare_chain, full_path_used, run_chain
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_idle_limit_reports_timeout_and_a_fresh_workspace_recovers():
    spec = W.ChainSpec("timeout B=64 g=4 V=32768", B=64, gamma=4, V=32768, dtype="f32",
                       target_sigma=3.0, temperature=1.0, top_k=0, draft_sigma=1.0)
    batch = W.make_chain(spec, seed=7)
    assert api.chain_workspace_kind(True, 0, spec.V) == L.SPEC_WS_CHAIN_FULL
    dev = "cuda"
    ws = L.new_workspace(L.SPEC_WS_CHAIN_FULL, spec.B, spec.gamma, spec.V, dev)  # this call's own
    try:
        L.spec_set_idle_limit(1)
        api.verify_chain(batch.target.to(dev), torch.from_numpy(batch.draft_tokens).to(dev),
                         gamma=spec.gamma, temperature=spec.temperature, draft=batch.draft.to(dev),
                         uniforms=torch.from_numpy(batch.uniforms).to(dev), ws=ws)
        torch.cuda.synchronize()
    finally:
        L.spec_set_idle_limit(0)
    assert L.spec_get_status(ws) & L.SPEC_FLAG_TIMEOUT
    # the call's outputs are not valid and its workspace is not clean; a fresh
    # one (and the default limit) gives exact results
    del ws
    api.clear_workspaces()
    gpu = run_chain(batch, residual=False)
    assert full_path_used(spec.B, spec.gamma, spec.V)
    assert compare_chain(batch, gpu, range(spec.B)).boundary <= 1
