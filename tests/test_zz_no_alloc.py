"""spec_verify_chain_static: chain verification without any device allocation.

Callers that cannot allocate device memory where they verify a round (code
under a pool or arena allocator that owns every device byte, framework
plug-ins that forbid allocation on the hot path, callers that must avoid an
allocation's implicit synchronisation) use this entry point: its scratch is
a fixed array inside the library.  These tests call it through the C ABI
and compare it with spec_verify_chain, which uses a caller-allocated
workspace, on two calls in a row (the array keeps the previous call's
contents, so the second call checks that it is cleared correctly).
"""
import ctypes

import numpy as np
import pytest
import torch

from parity import PROB_TOL
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import api
from speculative_decoding_verification_37_gb300 import build as _build
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(B, g, sampled, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(n_acc=torch.full((B,), -7, **i32), out_tokens=torch.full((B, g + 1), -7, **i32),
                n_out=torch.full((B,), -7, **i32), flags=torch.full((B,), -7, **i32),
                accept_prob=torch.full((B, g), -7.0, device=dev) if sampled else None,
                residual_mass=torch.full((B, g), -7.0, device=dev) if sampled else None)


CASES = {
    "topk": W.ChainSpec("topk", B=16, gamma=4, V=128256, dtype="bf16", target_sigma=3.0,
                        zipf_bias=True, draft_sigma=1.0, temperature=0.8, top_k=50),
    "full": W.WORKLOADS[1],
    "greedy": W.ChainSpec("greedy", B=32, gamma=8, V=152064, dtype="bf16", target_sigma=3.0,
                          temperature=0.0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_workspace_entry_point_twice(name):
    _build.build()
    spec = CASES[name]
    dev = "cuda"
    batch = W.make_chain(spec, seed=3)
    g, B = spec.gamma, spec.B
    sampled = not spec.greedy
    tgt = batch.target.to(dev)
    tok = torch.from_numpy(batch.draft_tokens).to(dev)
    drf = batch.draft.to(dev) if sampled else None
    unif = torch.from_numpy(batch.uniforms).to(dev) if sampled else None
    common = dict(target_logits=tgt, draft_tokens=tok, gamma=g, temperature=spec.temperature,
                  draft_logits=drf, uniforms=unif, top_k=spec.top_k)

    ref = _outputs(B, g, sampled, dev)
    ws = api.workspace(L.SPEC_WS_CHAIN, B, g, spec.V, dev)
    L.spec_verify_chain(workspace=ws, **common, **ref)
    outs = [_outputs(B, g, sampled, dev) for _ in range(2)]
    torch.cuda.synchronize()
    # the device's free memory is read with every buffer of the test already
    # allocated: the static calls must not change it
    free0 = torch.cuda.mem_get_info()[0]
    for call in range(2):
        got = outs[call]
        L.spec_verify_chain_static(**common, **got)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, call
        for key in ("n_acc", "n_out", "out_tokens", "flags"):
            assert torch.equal(got[key], ref[key]), (call, key)
        if sampled:
            for key in ("accept_prob", "residual_mass"):
                err = (got[key] - ref[key]).abs().max().item()
                assert err <= PROB_TOL, (call, key, err)
        assert int(got["n_out"].min()) >= 1


def test_static_scratch_rejects_oversized_batches():
    _build.build()
    need = L.spec_workspace_bytes(L.SPEC_WS_CHAIN, 100000, 8, 1000)
    assert need > L.SPEC_STATIC_WORKSPACE_BYTES
    a = L.SpecChainArgs(B=100000, gamma=8, V=1000, dtype=L.SPEC_DTYPE_F32, target_logits=4096,
                        target_row_stride=1000, draft_tokens=256, temperature=0.0,
                        n_acc=1024, out_tokens=2048, n_out=3072)
    # rejected on the host, before anything is enqueued
    assert L.lib().spec_verify_chain_static(ctypes.byref(a), None) == L.SPEC_ERR_TOO_LARGE
    assert b"static workspace" in L.lib().spec_error_string(L.SPEC_ERR_TOO_LARGE)
    assert np.isfinite(need)


def test_static_scratch_with_top_p_matches_the_workspace_entry_point():
    """Top-p through the fixed array: the exact path, with the same results
    as the workspace entry point taking that path with a plain workspace."""
    _build.build()
    spec = CASES["topk"]
    dev = "cuda"
    batch = W.make_chain(spec, seed=3)
    common = dict(target_logits=batch.target.to(dev),
                  draft_tokens=torch.from_numpy(batch.draft_tokens).to(dev), gamma=spec.gamma,
                  temperature=spec.temperature, draft_logits=batch.draft.to(dev),
                  uniforms=torch.from_numpy(batch.uniforms).to(dev), top_k=spec.top_k, top_p=0.9)
    ref = _outputs(spec.B, spec.gamma, True, dev)
    L.spec_verify_chain(workspace=api.workspace(L.SPEC_WS_CHAIN, spec.B, spec.gamma, spec.V, dev),
                        **common, **ref)
    got = _outputs(spec.B, spec.gamma, True, dev)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    L.spec_verify_chain_static(**common, **got)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    for key in ("n_acc", "n_out", "out_tokens", "flags"):
        assert torch.equal(got[key], ref[key]), key
    assert int(got["n_out"].min()) >= 1
