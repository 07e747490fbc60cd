"""GB300-native (sm_103a) batched target-side verify-and-commit step of
speculative decoding: chain and tree verification plus paged-KV commit,
plus the draft-side tree builder and n-gram drafter, behind a small C ABI (include/spec_verify.h) with a thin ctypes binding."""
from ._lib import (EXPORTED, SPEC_DTYPE_BF16, SPEC_DTYPE_F32, SPEC_ERR_CUDA,  # noqa: F401
                   SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_FLAG_BAD_INPUT,
                   SPEC_FLAG_BAD_ROW, SPEC_FLAG_EOS, SPEC_FLAG_FALLBACK, SPEC_FLAG_LIMIT, SPEC_FLAG_TIMEOUT, SPEC_OK, SPEC_WS_CHAIN,
                   SPEC_WS_CHAIN_FULL, SPEC_WS_CHAIN_TOPK, SPEC_WS_COMMIT,
                   SPEC_WS_TREE, SPEC_WS_TREE_LEVEL, SpecError, lib, new_workspace, spec_commit_kv,
                   spec_get_status, spec_ngram_draft, spec_tree_level, spec_verify_chain,
                   spec_verify_tree, spec_workspace_bytes)
from .api import (ChainOut, NgramOut, TreeBuilder, TreeOut, chain_workspace_kind,  # noqa: F401
                  clear_workspaces, commit_kv, ngram_draft, verify_chain, verify_tree, workspace)
