"""ctypes binding of libspecverify.so.

Argument marshalling only: every step of the verify-and-commit path runs in
the library's CUDA kernels.  PyTorch tensors serve as owners of device memory
and streams.  If the library is missing, loading fails loudly; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint32, c_void_p
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspecverify.so")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA, SPEC_ERR_TOO_LARGE = 0, 1, 2, 3, 4
SPEC_STATIC_WORKSPACE_BYTES = 1 << 20
SPEC_DTYPE_BF16, SPEC_DTYPE_F32 = 0, 1
SPEC_FLAG_BAD_INPUT, SPEC_FLAG_FALLBACK, SPEC_FLAG_BAD_ROW, SPEC_FLAG_TIMEOUT = 1, 2, 4, 8
SPEC_WS_CHAIN, SPEC_WS_TREE, SPEC_WS_COMMIT, SPEC_WS_CHAIN_TOPK, SPEC_WS_CHAIN_FULL = 0, 1, 2, 3, 4
SPEC_WS_TREE_LEVEL = 5
SPEC_FLAG_EOS, SPEC_FLAG_LIMIT = 16, 32
SPEC_TREE_MAX_HEADS = 64
TOPK_FAST_MAX = 128   # top_k served by the candidate-pool path when the workspace holds it

EXPORTED = ("spec_verify_chain", "spec_verify_tree", "spec_commit_kv", "spec_workspace_bytes",
            "spec_get_status", "spec_error_string", "spec_last_cuda_error",
            "spec_verify_chain_static", "spec_selftest_ex2", "spec_ngram_draft", "spec_tree_level",
            "spec_set_idle_limit")


class SpecChainArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("gamma", c_int32), ("V", c_int32), ("dtype", c_int32),
                ("target_logits", c_void_p), ("target_row_stride", c_int64),
                ("draft_logits", c_void_p), ("draft_row_stride", c_int64),
                ("draft_tokens", c_void_p), ("uniforms", c_void_p),
                ("temperature", c_float), ("top_k", c_int32), ("fallback_eps", c_float),
                ("n_acc", c_void_p), ("out_tokens", c_void_p), ("n_out", c_void_p),
                ("accept_prob", c_void_p), ("residual_mass", c_void_p), ("flags", c_void_p),
                ("committed_len", c_void_p), ("draft_len", c_void_p), ("blocks_in_use", c_void_p),
                ("block_size", c_int32), ("kv_capacity", c_int64), ("eos_enabled", c_int32),
                ("eos_token", c_int32), ("max_new", c_void_p), ("top_p", c_float),
                ("gamma_per_request", c_void_p), ("temperature_per_request", c_void_p),
                ("top_k_per_request", c_void_p), ("top_p_per_request", c_void_p)]


class SpecTreeArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("N", c_int32), ("R", c_int32), ("V", c_int32), ("dtype", c_int32),
                ("logits", c_void_p), ("row_stride", c_int64),
                ("node_token", c_void_p), ("node_parent", c_void_p), ("row_of_node", c_void_p),
                ("committed_len", c_void_p), ("path", c_void_p), ("n_acc", c_void_p),
                ("out_tokens", c_void_p), ("n_out", c_void_p), ("tree_mask", c_void_p),
                ("pos", c_void_p), ("commit_slots", c_void_p), ("n_commit", c_void_p),
                ("flags", c_void_p)]


class SpecCommitArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("L", c_int32), ("H", c_int32), ("D", c_int32), ("S", c_int32),
                ("block_size", c_int32), ("elem_bytes", c_int32),
                ("temp_kv", c_void_p), ("cache", c_void_p), ("num_blocks", c_int64),
                ("block_table", c_void_p), ("max_blocks", c_int32),
                ("slots", c_void_p), ("slots_stride", c_int32),
                ("n_slots", c_void_p), ("committed_len", c_void_p),
                ("blocks_in_use", c_void_p), ("flags", c_void_p)]


class SpecNgramArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("gamma", c_int32), ("n_min", c_int32), ("n_max", c_int32),
                ("history", c_void_p), ("history_stride", c_int64), ("hist_len", c_void_p),
                ("draft_tokens", c_void_p), ("n_draft", c_void_p), ("match_n", c_void_p),
                ("match_start", c_void_p), ("flags", c_void_p)]


class SpecTreeLevelArgs(ctypes.Structure):
    _fields_ = [("B", c_int32), ("V", c_int32), ("dtype", c_int32), ("H", c_int32),
                ("k", c_int32 * SPEC_TREE_MAX_HEADS), ("n_next", c_int32), ("N", c_int32),
                ("n_before", c_int32), ("next_row0", c_int32), ("logits", c_void_p),
                ("row_stride", c_int64), ("parents", c_void_p), ("node_token", c_void_p),
                ("node_parent", c_void_p), ("node_logp", c_void_p), ("row_of_node", c_void_p),
                ("next_parents", c_void_p), ("flags", c_void_p)]


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = f"{fn} returned {code} ({lib().spec_error_string(code).decode()})"
        if code == SPEC_ERR_CUDA:
            msg += ": " + lib().spec_last_cuda_error().decode()
        super().__init__(msg)
        self.code = code


_LIB = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "speculative_decoding_verification_37_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.spec_verify_chain.argtypes = [POINTER(SpecChainArgs), c_void_p, c_size_t, c_void_p]
        L.spec_verify_tree.argtypes = [POINTER(SpecTreeArgs), c_void_p, c_size_t, c_void_p]
        L.spec_commit_kv.argtypes = [POINTER(SpecCommitArgs), c_void_p, c_size_t, c_void_p]
        for f in ("spec_verify_chain", "spec_verify_tree", "spec_commit_kv"):
            getattr(L, f).restype = c_int
        L.spec_workspace_bytes.argtypes = [c_int, c_int32, c_int32, c_int32]
        L.spec_workspace_bytes.restype = c_size_t
        L.spec_get_status.argtypes = [c_void_p, c_void_p, POINTER(c_uint32)]
        L.spec_get_status.restype = c_int
        L.spec_error_string.argtypes = [c_int]
        L.spec_error_string.restype = c_char_p
        L.spec_verify_chain_static.argtypes = [POINTER(SpecChainArgs), c_void_p]
        L.spec_verify_chain_static.restype = c_int
        L.spec_last_cuda_error.argtypes = []
        L.spec_last_cuda_error.restype = c_char_p
        L.spec_selftest_ex2.argtypes = [POINTER(ctypes.c_float)]
        L.spec_selftest_ex2.restype = c_int
        L.spec_set_idle_limit.argtypes = [c_int64]
        L.spec_set_idle_limit.restype = c_int
        L.spec_ngram_draft.argtypes = [POINTER(SpecNgramArgs), c_void_p]
        L.spec_ngram_draft.restype = c_int
        L.spec_tree_level.argtypes = [POINTER(SpecTreeLevelArgs), c_void_p, c_size_t, c_void_p]
        L.spec_tree_level.restype = c_int
        _LIB = L
    return _LIB


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream) -> c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_DTYPE_BF16
    if t.dtype == torch.float32:
        return SPEC_DTYPE_F32
    raise TypeError(f"logits must be bfloat16 or float32, not {t.dtype}")


def _check(fn: str, code: int):
    if code != SPEC_OK:
        raise SpecError(fn, code)


def spec_workspace_bytes(kind: int, B: int, n: int, V: int) -> int:
    return int(lib().spec_workspace_bytes(kind, B, n, V))


def new_workspace(kind: int, B: int, n: int, V: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (torch allocates it; the library never does)."""
    nbytes = max(spec_workspace_bytes(kind, B, n, V), 256)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def spec_ngram_draft(*, history: torch.Tensor, hist_len: torch.Tensor, gamma: int, n_min: int,
                     n_max: int, draft_tokens: torch.Tensor, n_draft: torch.Tensor,
                     match_n: Optional[torch.Tensor] = None, match_start: Optional[torch.Tensor] = None,
                     flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """Marshals one spec_ngram_draft call: history int32 [B, stride] (rows may
    be strided), hist_len int32 [B], draft_tokens int32 [B, gamma]."""
    a = SpecNgramArgs(B=history.shape[0], gamma=gamma, n_min=n_min, n_max=n_max, history=_ptr(history),
                      history_stride=history.stride(0), hist_len=_ptr(hist_len),
                      draft_tokens=_ptr(draft_tokens), n_draft=_ptr(n_draft), match_n=_ptr(match_n),
                      match_start=_ptr(match_start), flags=_ptr(flags))
    _check("spec_ngram_draft", lib().spec_ngram_draft(ctypes.byref(a), _stream(stream)))


def spec_tree_level(*, logits: torch.Tensor, H: int, k, n_next: int, n_before: int, next_row0: int,
                    node_token: torch.Tensor, node_parent: torch.Tensor, node_logp: torch.Tensor,
                    row_of_node: torch.Tensor, workspace: torch.Tensor,
                    parents: Optional[torch.Tensor] = None, next_parents: Optional[torch.Tensor] = None,
                    flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """Marshals one spec_tree_level call: logits [B*H, V] (row stride =
    stride(0)), node arrays [B, N] / [B, N+1], parents [B, H] or None at the
    root, next_parents [B, n_next]."""
    B = logits.shape[0] // H
    kk = (c_int32 * SPEC_TREE_MAX_HEADS)(*[int(x) for x in k])
    a = SpecTreeLevelArgs(B=B, V=logits.shape[-1], dtype=_dtype_code(logits), H=H, k=kk,
                          n_next=n_next, N=node_token.shape[-1], n_before=n_before,
                          next_row0=next_row0, logits=_ptr(logits), row_stride=logits.stride(0),
                          parents=_ptr(parents), node_token=_ptr(node_token),
                          node_parent=_ptr(node_parent), node_logp=_ptr(node_logp),
                          row_of_node=_ptr(row_of_node), next_parents=_ptr(next_parents),
                          flags=_ptr(flags))
    _check("spec_tree_level", lib().spec_tree_level(ctypes.byref(a), _ptr(workspace),
                                                    workspace.numel(), _stream(stream)))


def spec_selftest_ex2() -> float:
    """Largest relative error of the GPU's hardware exponential over [-126, 1]
    (the certified fp32 draw assumes 1.5e-7)."""
    out = ctypes.c_float(0.0)
    _check("spec_selftest_ex2", lib().spec_selftest_ex2(ctypes.byref(out)))
    return float(out.value)


def spec_set_idle_limit(polls: int) -> None:
    """Idle polls before a warp of the persistent full-vocabulary path gives
    up (SPEC_FLAG_TIMEOUT); 0 restores the default.  Process-wide."""
    _check("spec_set_idle_limit", lib().spec_set_idle_limit(int(polls)))


def spec_get_status(workspace: torch.Tensor, stream=None) -> int:
    out = c_uint32(0)
    _check("spec_get_status", lib().spec_get_status(_ptr(workspace), _stream(stream), ctypes.byref(out)))
    return int(out.value)


def spec_verify_chain(*, target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                      n_acc: torch.Tensor, out_tokens: torch.Tensor, n_out: torch.Tensor,
                      workspace: torch.Tensor, gamma: int, temperature: float,
                      draft_logits: Optional[torch.Tensor] = None,
                      uniforms: Optional[torch.Tensor] = None, top_k: int = 0,
                      fallback_eps: float = 1e-6, accept_prob: Optional[torch.Tensor] = None,
                      residual_mass: Optional[torch.Tensor] = None,
                      flags: Optional[torch.Tensor] = None,
                      committed_len: Optional[torch.Tensor] = None,
                      draft_len: Optional[torch.Tensor] = None,
                      blocks_in_use: Optional[torch.Tensor] = None, block_size: int = 0,
                      kv_capacity: int = 0, eos_token: Optional[int] = None,
                      max_new: Optional[torch.Tensor] = None, top_p: float = 0.0,
                      gamma_per_request: Optional[torch.Tensor] = None,
                      temperature_per_request: Optional[torch.Tensor] = None,
                      top_k_per_request: Optional[torch.Tensor] = None,
                      top_p_per_request: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    """Marshals one spec_verify_chain call.  Logits are 2-D [rows, V] views
    (row stride = stride(0)); every tensor must already be on the device.
    The *_per_request tensors (int32 / float32 [B]) give each request its
    own gamma, temperature, top-k and top-p."""
    V = target_logits.shape[-1]
    B = target_logits.shape[0] // (gamma + 1)
    a = SpecChainArgs(B=B, gamma=gamma, V=V, dtype=_dtype_code(target_logits),
                      target_logits=_ptr(target_logits), target_row_stride=target_logits.stride(0),
                      draft_logits=_ptr(draft_logits),
                      draft_row_stride=draft_logits.stride(0) if draft_logits is not None else 0,
                      draft_tokens=_ptr(draft_tokens), uniforms=_ptr(uniforms),
                      temperature=float(temperature), top_k=int(top_k),
                      fallback_eps=float(fallback_eps), n_acc=_ptr(n_acc),
                      out_tokens=_ptr(out_tokens), n_out=_ptr(n_out),
                      accept_prob=_ptr(accept_prob), residual_mass=_ptr(residual_mass),
                      flags=_ptr(flags), committed_len=_ptr(committed_len),
                      draft_len=_ptr(draft_len), blocks_in_use=_ptr(blocks_in_use),
                      block_size=int(block_size), kv_capacity=int(kv_capacity),
                      eos_enabled=0 if eos_token is None else 1,
                      eos_token=0 if eos_token is None else int(eos_token), max_new=_ptr(max_new),
                      top_p=float(top_p), gamma_per_request=_ptr(gamma_per_request),
                      temperature_per_request=_ptr(temperature_per_request),
                      top_k_per_request=_ptr(top_k_per_request),
                      top_p_per_request=_ptr(top_p_per_request))
    _check("spec_verify_chain", lib().spec_verify_chain(
        ctypes.byref(a), _ptr(workspace), workspace.numel(), _stream(stream)))


def spec_verify_tree(*, logits: torch.Tensor, R: int, node_token: torch.Tensor,
                     node_parent: torch.Tensor, row_of_node: torch.Tensor, path: torch.Tensor,
                     n_acc: torch.Tensor, out_tokens: torch.Tensor, n_out: torch.Tensor,
                     workspace: torch.Tensor, committed_len: Optional[torch.Tensor] = None,
                     tree_mask: Optional[torch.Tensor] = None, pos: Optional[torch.Tensor] = None,
                     commit_slots: Optional[torch.Tensor] = None,
                     n_commit: Optional[torch.Tensor] = None, flags: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    V = logits.shape[-1]
    B = logits.shape[0] // R
    N = node_token.shape[-1]
    a = SpecTreeArgs(B=B, N=N, R=R, V=V, dtype=_dtype_code(logits), logits=_ptr(logits),
                     row_stride=logits.stride(0), node_token=_ptr(node_token),
                     node_parent=_ptr(node_parent), row_of_node=_ptr(row_of_node),
                     committed_len=_ptr(committed_len), path=_ptr(path), n_acc=_ptr(n_acc),
                     out_tokens=_ptr(out_tokens), n_out=_ptr(n_out), tree_mask=_ptr(tree_mask),
                     pos=_ptr(pos), commit_slots=_ptr(commit_slots), n_commit=_ptr(n_commit),
                     flags=_ptr(flags))
    _check("spec_verify_tree", lib().spec_verify_tree(
        ctypes.byref(a), _ptr(workspace), workspace.numel(), _stream(stream)))


def spec_commit_kv(*, temp_kv: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
                   n_slots: torch.Tensor, committed_len: torch.Tensor, block_size: int,
                   workspace: torch.Tensor, slots: Optional[torch.Tensor] = None,
                   blocks_in_use: Optional[torch.Tensor] = None,
                   flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """temp_kv [B, L, 2, S, H, D]; cache [L, 2, num_blocks, block_size, H, D]."""
    B, L, two, S, H, D = temp_kv.shape
    a = SpecCommitArgs(B=B, L=L, H=H, D=D, S=S, block_size=block_size,
                       elem_bytes=temp_kv.element_size(), temp_kv=_ptr(temp_kv), cache=_ptr(cache),
                       num_blocks=cache.shape[2], block_table=_ptr(block_table),
                       max_blocks=block_table.shape[-1], slots=_ptr(slots),
                       slots_stride=slots.stride(0) if slots is not None else 0,
                       n_slots=_ptr(n_slots), committed_len=_ptr(committed_len),
                       blocks_in_use=_ptr(blocks_in_use), flags=_ptr(flags))
    _check("spec_commit_kv", lib().spec_commit_kv(
        ctypes.byref(a), _ptr(workspace), workspace.numel(), _stream(stream)))


def spec_verify_chain_static(*, target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                             n_acc: torch.Tensor, out_tokens: torch.Tensor, n_out: torch.Tensor,
                             gamma: int, temperature: float,
                             draft_logits: Optional[torch.Tensor] = None,
                             uniforms: Optional[torch.Tensor] = None, top_k: int = 0,
                             fallback_eps: float = 1e-6, accept_prob: Optional[torch.Tensor] = None,
                             residual_mass: Optional[torch.Tensor] = None,
                             flags: Optional[torch.Tensor] = None,
                             committed_len: Optional[torch.Tensor] = None,
                             draft_len: Optional[torch.Tensor] = None,
                             blocks_in_use: Optional[torch.Tensor] = None, block_size: int = 0,
                             kv_capacity: int = 0, eos_token: Optional[int] = None,
                             max_new: Optional[torch.Tensor] = None, top_p: float = 0.0,
                             stream=None) -> None:
    """Marshals one spec_verify_chain_static call: the same as
    spec_verify_chain, but the library's fixed device array is the scratch,
    for callers that cannot allocate device memory."""
    V = target_logits.shape[-1]
    B = target_logits.shape[0] // (gamma + 1)
    a = SpecChainArgs(B=B, gamma=gamma, V=V, dtype=_dtype_code(target_logits),
                      target_logits=_ptr(target_logits), target_row_stride=target_logits.stride(0),
                      draft_logits=_ptr(draft_logits),
                      draft_row_stride=draft_logits.stride(0) if draft_logits is not None else 0,
                      draft_tokens=_ptr(draft_tokens), uniforms=_ptr(uniforms),
                      temperature=float(temperature), top_k=int(top_k),
                      fallback_eps=float(fallback_eps), n_acc=_ptr(n_acc),
                      out_tokens=_ptr(out_tokens), n_out=_ptr(n_out),
                      accept_prob=_ptr(accept_prob), residual_mass=_ptr(residual_mass),
                      flags=_ptr(flags), committed_len=_ptr(committed_len),
                      draft_len=_ptr(draft_len), blocks_in_use=_ptr(blocks_in_use),
                      block_size=int(block_size), kv_capacity=int(kv_capacity),
                      eos_enabled=0 if eos_token is None else 1,
                      eos_token=0 if eos_token is None else int(eos_token), max_new=_ptr(max_new),
                      top_p=float(top_p))
    _check("spec_verify_chain_static", lib().spec_verify_chain_static(ctypes.byref(a), _stream(stream)))
