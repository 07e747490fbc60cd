"""The C ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/spec_verify.h declares, matches the C struct layouts, and
rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from conftest import ROOT
from speculative_decoding_verification_37_gb300 import _lib as L
from speculative_decoding_verification_37_gb300 import build as B

HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(L.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (spec_\w+)", out.stdout))
    assert set(names) <= exported


def test_build_targets_sm_103a_only():
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_struct_layouts_match_c(lib):
    src = r"""
    #include <stdio.h>
    #include <stddef.h>
    #include "spec_verify.h"
    #define P(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
    int main(void) {
        printf("SpecChainArgs %zu\nSpecTreeArgs %zu\nSpecCommitArgs %zu\nSpecTreeLevelArgs %zu\n",
               sizeof(SpecChainArgs), sizeof(SpecTreeArgs), sizeof(SpecCommitArgs),
               sizeof(SpecTreeLevelArgs));
        P(SpecTreeLevelArgs, k) P(SpecTreeLevelArgs, logits) P(SpecTreeLevelArgs, row_stride)
        P(SpecTreeLevelArgs, flags) P(SpecTreeLevelArgs, next_row0)
        P(SpecChainArgs, flags) P(SpecChainArgs, fallback_eps) P(SpecChainArgs, uniforms)
        P(SpecChainArgs, committed_len) P(SpecChainArgs, block_size) P(SpecChainArgs, kv_capacity)
        P(SpecChainArgs, eos_enabled) P(SpecChainArgs, max_new) P(SpecChainArgs, top_p)
        P(SpecChainArgs, gamma_per_request) P(SpecChainArgs, temperature_per_request)
        P(SpecChainArgs, top_k_per_request) P(SpecChainArgs, top_p_per_request)
        P(SpecTreeArgs, flags) P(SpecTreeArgs, committed_len) P(SpecTreeArgs, row_stride)
        P(SpecCommitArgs, flags) P(SpecCommitArgs, num_blocks) P(SpecCommitArgs, slots_stride)
        return 0;
    }
    """
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.split() for line in lines if line)
    structs = {"SpecChainArgs": L.SpecChainArgs, "SpecTreeArgs": L.SpecTreeArgs,
               "SpecCommitArgs": L.SpecCommitArgs, "SpecTreeLevelArgs": L.SpecTreeLevelArgs}
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
    for key, val in got.items():
        if "." in key:
            s, f = key.split(".")
            assert getattr(structs[s], f).offset == int(val), key


def test_workspace_sizes(lib):
    assert L.spec_workspace_bytes(L.SPEC_WS_CHAIN, 64, 4, 128256) >= 256 + 64 * 4 + 64 * 5 * 16
    assert L.spec_workspace_bytes(L.SPEC_WS_TREE, 128, 5, 128256) >= 256 + 128 * 4 + 128 * 5 * 8
    assert L.spec_workspace_bytes(L.SPEC_WS_COMMIT, 512, 0, 0) >= 256 + 512 * 4
    base = L.spec_workspace_bytes(L.SPEC_WS_CHAIN, 64, 4, 128256)
    # the chain workspace exactly: a 256-byte header, two per-request words,
    # a 16-byte record per position, each region rounded up to 256 bytes
    al = lambda x: (x + 255) // 256 * 256
    rows = 64 * 5
    assert base == 256 + 2 * al(64 * 4) + al(rows * 16)
    # the top-k path adds, per position and row slot: 256 thread maxima and
    # 4 x 256 packed groups (4 bytes each) from the pass, then a 32-byte kept-set
    # header and 256 kept entries of 8 bytes, and one arrival counter per
    # position; none of it depends on V
    topk = base + al(rows * 2 * 256 * 4) + al(rows * 2 * 4 * 256 * 4) + al(rows * 2 * 32) + \
        al(rows * 2 * 256 * 8) + al(rows * 4)
    assert L.spec_workspace_bytes(L.SPEC_WS_CHAIN_TOPK, 64, 4, 128256) == topk
    assert L.spec_workspace_bytes(L.SPEC_WS_CHAIN_TOPK, 64, 4, 1000) == topk
    assert L.spec_workspace_bytes(99, 1, 1, 1) == 0
    assert L.spec_workspace_bytes(L.SPEC_WS_CHAIN, -1, 1, 1) == 0


def _chain_args(**over):
    a = L.SpecChainArgs(B=2, gamma=2, V=16, dtype=L.SPEC_DTYPE_F32, target_logits=4096,
                        target_row_stride=16, draft_logits=8192, draft_row_stride=16,
                        draft_tokens=256, uniforms=512, temperature=1.0, top_k=0,
                        fallback_eps=1e-6, n_acc=1024, out_tokens=2048, n_out=3072,
                        accept_prob=None, residual_mass=None, flags=None)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(V=0), dict(gamma=-1), dict(B=-1), dict(dtype=7), dict(temperature=-1.0),
    dict(temperature=float("nan")), dict(top_k=-2), dict(fallback_eps=-1.0),
    dict(target_logits=None), dict(target_row_stride=15), dict(n_acc=None),
    dict(draft_tokens=None), dict(uniforms=None), dict(draft_logits=None),
    dict(draft_row_stride=3), dict(target_logits=4097),
    dict(blocks_in_use=4096),                                   # needs committed_len
    dict(committed_len=4096, blocks_in_use=4352, block_size=0),  # needs block_size >= 1
    dict(draft_len=4096), dict(committed_len=4096, kv_capacity=-1),
    dict(eos_enabled=1, eos_token=-1), dict(eos_enabled=1, eos_token=16),   # EOS outside [0, V)
    dict(top_p=-0.5), dict(top_p=float("nan")),
])
def test_chain_host_validation(lib, bad):
    a = _chain_args(**bad)
    ws = ctypes.create_string_buffer(1 << 16)
    # host buffers stand in for device pointers: validation must reject first
    assert lib.spec_verify_chain(ctypes.byref(a), ws, 1 << 16, None) == L.SPEC_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [
    dict(V=0), dict(dtype=7), dict(temperature=float("nan")), dict(top_k=-2),
    dict(target_logits=None), dict(uniforms=None), dict(draft_row_stride=3),
    dict(eos_enabled=1, eos_token=16), dict(top_p=float("nan")),
])
def test_static_entry_point_checks_arguments_first(lib, bad):
    """spec_verify_chain_static refuses every bad call before it touches
    CUDA: on this GPU-less host any CUDA call (the device lookup, the memset
    of its array) would fail with SPEC_ERR_CUDA instead."""
    a = _chain_args(**bad)
    assert lib.spec_verify_chain_static(ctypes.byref(a), None) == L.SPEC_ERR_INVALID_ARG
    a = _chain_args(gamma_per_request=8192, eos_enabled=1, eos_token=3)
    assert lib.spec_verify_chain_static(ctypes.byref(a), None) == L.SPEC_ERR_UNSUPPORTED
    assert lib.spec_verify_chain_static(ctypes.byref(_chain_args(B=0)), None) == L.SPEC_OK


def test_chain_workspace_validation(lib):
    a = _chain_args()
    assert lib.spec_verify_chain(ctypes.byref(a), None, 0, None) == L.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_chain(ctypes.byref(a), ctypes.c_void_p(4096), 16, None) == L.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_chain(ctypes.byref(a), ctypes.c_void_p(4097), 1 << 20, None) == L.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_chain(None, None, 0, None) == L.SPEC_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    a = _chain_args(B=0)
    assert lib.spec_verify_chain(ctypes.byref(a), None, 0, None) == L.SPEC_OK
    t = L.SpecTreeArgs(B=0, N=3, R=1, V=10, dtype=0)
    assert lib.spec_verify_tree(ctypes.byref(t), None, 0, None) == L.SPEC_OK
    c = L.SpecCommitArgs(B=0, L=1, H=1, D=8, S=1, block_size=16, elem_bytes=2, num_blocks=1,
                         max_blocks=1)
    assert lib.spec_commit_kv(ctypes.byref(c), None, 0, None) == L.SPEC_OK


def test_tree_and_commit_host_validation(lib):
    ws = ctypes.create_string_buffer(1 << 16)
    t = L.SpecTreeArgs(B=1, N=2000, R=1, V=10, dtype=0, logits=4096, row_stride=10)
    assert lib.spec_verify_tree(ctypes.byref(t), ws, 1 << 16, None) == L.SPEC_ERR_INVALID_ARG
    t = L.SpecTreeArgs(B=1, N=3, R=0, V=10, dtype=0, logits=4096, row_stride=10)
    assert lib.spec_verify_tree(ctypes.byref(t), ws, 1 << 16, None) == L.SPEC_ERR_INVALID_ARG
    t = L.SpecTreeArgs(B=1, N=3, R=1, V=10, dtype=0, logits=4096, row_stride=10, node_token=256,
                       node_parent=512, row_of_node=768, path=1024, n_acc=1280, out_tokens=1536,
                       n_out=1792, pos=2048, committed_len=None)
    assert lib.spec_verify_tree(ctypes.byref(t), ws, 1 << 16, None) == L.SPEC_ERR_INVALID_ARG
    c = L.SpecCommitArgs(B=1, L=1, H=1, D=7, S=1, block_size=16, elem_bytes=2, num_blocks=1,
                         max_blocks=1, temp_kv=4096, cache=8192, block_table=256, n_slots=512,
                         committed_len=768)
    assert lib.spec_commit_kv(ctypes.byref(c), ws, 1 << 16, None) == L.SPEC_ERR_UNSUPPORTED
    c.D, c.elem_bytes = 8, 3
    assert lib.spec_commit_kv(ctypes.byref(c), ws, 1 << 16, None) == L.SPEC_ERR_INVALID_ARG
    c.elem_bytes, c.cache = 2, 8200
    assert lib.spec_commit_kv(ctypes.byref(c), ws, 1 << 16, None) == L.SPEC_ERR_INVALID_ARG


def test_error_strings(lib):
    assert lib.spec_error_string(L.SPEC_ERR_INVALID_ARG) == b"invalid argument"
    assert lib.spec_error_string(12345) == b"unknown error code"


def _level_args(**over):
    k = (ctypes.c_int32 * L.SPEC_TREE_MAX_HEADS)(*([2, 2] + [0] * (L.SPEC_TREE_MAX_HEADS - 2)))
    a = L.SpecTreeLevelArgs(B=2, V=100, dtype=L.SPEC_DTYPE_F32, H=2, k=k, n_next=2, N=12, n_before=6,
                            next_row0=3, logits=4096, row_stride=100, parents=256, node_token=512,
                            node_parent=768, node_logp=1024, row_of_node=1280, next_parents=1536,
                            flags=None)
    for key, v in over.items():
        setattr(a, key, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(H=0), dict(H=65), dict(V=0), dict(dtype=5), dict(n_next=-1), dict(n_next=5), dict(n_next=65),
    dict(n_before=-1), dict(N=9), dict(next_row0=0), dict(parents=None), dict(logits=None),
    dict(logits=4098), dict(row_stride=99), dict(node_logp=None), dict(next_parents=None),
])
def test_tree_level_host_validation(lib, bad):
    a = _level_args(**bad)
    ws = ctypes.create_string_buffer(1 << 20)
    assert lib.spec_tree_level(ctypes.byref(a), ws, 1 << 20, None) == L.SPEC_ERR_INVALID_ARG


def test_tree_level_children_limits(lib):
    ws = ctypes.create_string_buffer(1 << 20)
    for ks in ([0, 2], [17, 2], [101, 1]):
        a = _level_args()
        a.k[0], a.k[1] = ks
        assert lib.spec_tree_level(ctypes.byref(a), ws, 1 << 20, None) == L.SPEC_ERR_INVALID_ARG
    a = _level_args(H=20, N=400, n_next=0)
    for j in range(20):
        a.k[j] = 16                                       # 320 children > 256 per level
    assert lib.spec_tree_level(ctypes.byref(a), ws, 1 << 20, None) == L.SPEC_ERR_INVALID_ARG
    a = _level_args()
    assert lib.spec_tree_level(ctypes.byref(a), None, 0, None) == L.SPEC_ERR_INVALID_ARG
    assert lib.spec_tree_level(ctypes.byref(a), ctypes.c_void_p(4096), 64, None) == L.SPEC_ERR_INVALID_ARG
    assert lib.spec_tree_level(ctypes.byref(_level_args(B=0)), None, 0, None) == L.SPEC_OK
    assert L.spec_workspace_bytes(L.SPEC_WS_TREE_LEVEL, 128, 2, 128256) >= 128 * 2 * 32 * 144


def test_per_request_rounds_have_no_early_end(lib):
    """Per-request settings go with neither the early end of a round nor the
    in-place commit: refused before anything is launched."""
    ws = ctypes.create_string_buffer(1 << 16)
    for over in (dict(eos_enabled=1, eos_token=3), dict(max_new=4096), dict(committed_len=4096)):
        a = _chain_args(gamma_per_request=8192, **over)
        assert lib.spec_verify_chain(ctypes.byref(a), ws, 1 << 16, None) == L.SPEC_ERR_UNSUPPORTED


def test_workspace_cache_and_clear(lib):
    from speculative_decoding_verification_37_gb300 import api
    w = api.workspace(L.SPEC_WS_COMMIT, 4, 0, 0, "cpu")
    assert api.workspace(L.SPEC_WS_COMMIT, 4, 0, 0, "cpu") is w
    assert int(w.sum()) == 0 and w.numel() >= L.spec_workspace_bytes(L.SPEC_WS_COMMIT, 4, 0, 0)
    api.clear_workspaces()
    assert api.workspace(L.SPEC_WS_COMMIT, 4, 0, 0, "cpu") is not w
