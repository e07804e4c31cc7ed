"""Python binding of the CUDA library ``_lib/libtv.so`` (argument marshalling only).

Every function has the name of the C entry point it calls (``include/tv.h``), takes torch
tensors that live on the GPU, and passes their data pointers, sizes and dtype codes.  All of
the work runs in the library's kernels; there is no CPU fallback.  Importing this package
raises ``ImportError`` when the library has not been built
(``python tree_speculative_verification_gdn_gb300/_build.py``).

Non-OK return codes raise :class:`TVError`.  Per-sequence, data-dependent errors land in the
caller's ``err`` tensor (read it after synchronising).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtv.so")

# Status codes and enums of include/tv.h.
TV_OK = 0
TV_ERR_INVALID_ARG = -1
TV_ERR_BAD_TREE = -2
TV_ERR_BAD_PATH = -3
TV_ERR_UNSUPPORTED = -4
TV_ERR_CUDA = -5
TV_ERR_TIMEOUT = -6
TV_ERR_CAPACITY = -7
TV_ERR_BAD_BLOCK = -8
TV_ERR_SCRATCH = -9
TV_F32 = 0
TV_BF16 = 1
TV_MODE_FORK = 0
TV_MODE_WY = 1
TV_MAX_NODES = 256
TV_BLOCK_SIZE = 16
TV_STATIC_SCRATCH_BYTES = 64 << 20

EXPORTED = ("tv_status_string", "tv_last_cuda_error", "tv_version", "tv_tree_prepare",
            "tv_gdn_tree_verify_fork", "tv_gdn_tree_verify_wy", "tv_gdn_commit",
            "tv_tree_attn_workspace_size", "tv_tree_attn", "tv_tree_attn_static", "tv_kv_compact",
            "tv_accept_walk", "tv_gdn_tree_verify_fork_selective", "tv_gdn_commit_selective",
            "tv_gdn_tree_verify_wy_lazy", "tv_gdn_fork_workspace_size", "tv_gdn_tree_verify_fork_ws",
            "tv_gdn_fork_materialize", "tv_gdn_fork_materialize_selective", "tv_gdn_commit_layers",
            "tv_kv_compact_remap", "tv_test_bounded_wait")

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

_SIGNATURES = {
    "tv_status_string": (ctypes.c_char_p, [_I]),
    "tv_last_cuda_error": (_I, []),
    "tv_version": (_I, []),
    "tv_tree_prepare": (_I, [_P, _I, _I, _P, _P, _P, _I, _P, _P, _P]),
    "tv_gdn_tree_verify_fork": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "tv_gdn_tree_verify_wy": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "tv_gdn_commit": (_I, [_I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "tv_gdn_commit_layers": (_I, [_I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "tv_tree_attn_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "tv_tree_attn": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _P, _P, _Z,
                          _P, _P]),
    "tv_tree_attn_static": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _P,
                                 _P, _P]),
    "tv_gdn_tree_verify_fork_selective": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I, _I,
                                              _F, _P, _P, _P, _P, _P]),
    "tv_gdn_commit_selective": (_I, [_P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                    _P, _P]),
    "tv_gdn_tree_verify_wy_lazy": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                       _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "tv_gdn_fork_workspace_size": (_Z, [_I, _I, _I, _I]),
    "tv_gdn_tree_verify_fork_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _Z,
                                       _P, _P]),
    "tv_gdn_fork_materialize": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "tv_gdn_fork_materialize_selective": (_I, [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                               _P, _P, _P, _P]),
    "tv_accept_walk": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tv_kv_compact": (_I, [_P, _P, _I, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "tv_kv_compact_remap": (_I, [_P, _P, _I, _P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                 _P]),
    "tv_test_bounded_wait": (_I, [ctypes.c_uint, _I, _P, _P, _P]),
}


class TVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.tv_status_string(status).decode()
        if status == TV_ERR_CUDA:
            msg += f" (cudaError {lib.tv_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first with "
                          "python tree_speculative_verification_gdn_gb300/_build.py or "
                          "__graft_entry__.build()")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


lib = _load()

_DTYPES = {torch.float32: TV_F32, torch.bfloat16: TV_BF16}


def _ptr(t):
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors passed to the library must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != TV_OK:
        raise TVError(status, where)


def status_string(status: int) -> str:
    return lib.tv_status_string(status).decode()


def tv_tree_prepare(parents, depth, mask_bits, err, paths=None, max_depth=None, stream=None) -> None:
    """parents [B,N] int32 -> depth [B,N] int32, mask_bits [B,N,ceil(N/32)] int32 (bit pattern
    of uint32 words), err [B] int32; optionally paths [B,N,cap] int32 (root-to-node, -1 padded)
    and max_depth [B] int32."""
    B, N = parents.shape
    cap = paths.shape[-1] if paths is not None else 0
    _check(lib.tv_tree_prepare(_ptr(parents), B, N, _ptr(depth), _ptr(mask_bits), _ptr(paths), cap,
                               _ptr(max_depth), _ptr(err), _stream(stream)), "tv_tree_prepare")


def tv_gdn_tree_verify_fork(q, k, v, alpha, beta, S0, parents, out, node_states, err,
                            q_scale: float = 1.0, stream=None) -> None:
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    _check(lib.tv_gdn_tree_verify_fork(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(parents), B, N, H, dk, dv,
        _DTYPES[q.dtype], _DTYPES[S0.dtype], float(q_scale), _ptr(out), _ptr(node_states), _ptr(err),
        _stream(stream)), "tv_gdn_tree_verify_fork")


def tv_gdn_fork_workspace_size(B, N, H, dv) -> int:
    return int(lib.tv_gdn_fork_workspace_size(B, N, H, dv))


def tv_gdn_tree_verify_fork_ws(q, k, v, alpha, beta, S0, parents, out, node_states, workspace, err,
                               q_scale: float = 1.0, stream=None) -> None:
    """Fork mode in two passes (TreeWY outputs and w, then the snapshots) with a workspace."""
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    _check(lib.tv_gdn_tree_verify_fork_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(parents), B, N, H, dk, dv,
        _DTYPES[q.dtype], _DTYPES[S0.dtype], float(q_scale), _ptr(out), _ptr(node_states), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)), "tv_gdn_tree_verify_fork_ws")


def tv_gdn_fork_materialize(k, alpha, S0, parents, pseudo_v, node_states, err, max_ctas_per_sm: int = 0,
                            stream=None) -> None:
    """Every fork-mode snapshot from the w of a preceding tv_gdn_tree_verify_wy (same inputs)."""
    B, N, H, dk = k.shape
    dv = pseudo_v.shape[-1]
    _check(lib.tv_gdn_fork_materialize(
        _ptr(k), _ptr(alpha), _ptr(S0), _ptr(parents), _ptr(pseudo_v), B, N, H, dk, dv, _DTYPES[k.dtype],
        _DTYPES[S0.dtype], int(max_ctas_per_sm), _ptr(node_states), _ptr(err), _stream(stream)),
        "tv_gdn_fork_materialize")


def tv_gdn_fork_materialize_selective(k, alpha, S0, parents, pseudo_v, confidence, threshold: float, node_states,
                                      slot, err, max_ctas_per_sm: int = 0, stream=None) -> None:
    """The selected fork-mode snapshots (confidence <= threshold) from the w of a preceding
    tv_gdn_tree_verify_wy: node_states [B, capacity, H, dv, dk], slot [B, N] int32."""
    B, N, H, dk = k.shape
    dv = pseudo_v.shape[-1]
    _check(lib.tv_gdn_fork_materialize_selective(
        _ptr(k), _ptr(alpha), _ptr(S0), _ptr(parents), _ptr(pseudo_v), _ptr(confidence), float(threshold),
        node_states.shape[1], B, N, H, dk, dv, _DTYPES[k.dtype], _DTYPES[S0.dtype], int(max_ctas_per_sm),
        _ptr(node_states), _ptr(slot), _ptr(err), _stream(stream)), "tv_gdn_fork_materialize_selective")


def tv_gdn_tree_verify_fork_selective(q, k, v, alpha, beta, S0, parents, confidence, threshold: float, out,
                                      node_states, slot, err, q_scale: float = 1.0, stream=None) -> None:
    """Fork mode keeping snapshots only of nodes with confidence <= threshold: node_states
    [B, capacity, H, dv, dk] (capacity = node_states.shape[1]), slot [B, N] int32."""
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    _check(lib.tv_gdn_tree_verify_fork_selective(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(parents), _ptr(confidence),
        float(threshold), node_states.shape[1], B, N, H, dk, dv, _DTYPES[q.dtype], _DTYPES[S0.dtype],
        float(q_scale), _ptr(out), _ptr(node_states), _ptr(slot), _ptr(err), _stream(stream)),
        "tv_gdn_tree_verify_fork_selective")


def tv_gdn_commit_selective(accepted_path, accepted_len, parents, node_states, slot, k, v, alpha, beta, S0, err,
                            stream=None) -> None:
    """Commit after tv_gdn_tree_verify_fork_selective (replays from the deepest kept snapshot)."""
    B, H, dv, dk = S0.shape
    N = parents.shape[1]
    _check(lib.tv_gdn_commit_selective(
        _ptr(accepted_path), _ptr(accepted_len), accepted_path.shape[1], _ptr(parents), _ptr(node_states),
        _ptr(slot), node_states.shape[1], _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), B, N, H, dk, dv,
        _DTYPES[k.dtype], _DTYPES[S0.dtype], _ptr(err), _stream(stream)), "tv_gdn_commit_selective")


def tv_gdn_tree_verify_wy_lazy(prev_path, prev_len, prev_parents, prev_pseudo_v, prev_log_gamma, prev_k,
                               q, k, v, alpha, beta, S0, parents, out, pseudo_v, log_gamma, err,
                               q_scale: float = 1.0, stream=None) -> None:
    """The previous round's TreeWY commit applied to S0 (in place) inside this round's verify."""
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    _check(lib.tv_gdn_tree_verify_wy_lazy(
        _ptr(prev_path), _ptr(prev_len), prev_path.shape[1], _ptr(prev_parents), prev_parents.shape[1],
        _ptr(prev_pseudo_v), _ptr(prev_log_gamma), _ptr(prev_k), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
        _ptr(beta), _ptr(S0), _ptr(parents), B, N, H, dk, dv, _DTYPES[q.dtype], _DTYPES[S0.dtype],
        float(q_scale), _ptr(out), _ptr(pseudo_v), _ptr(log_gamma), _ptr(err), _stream(stream)),
        "tv_gdn_tree_verify_wy_lazy")


def tv_gdn_tree_verify_wy(q, k, v, alpha, beta, S0, parents, out, pseudo_v, log_gamma, err,
                          q_scale: float = 1.0, stream=None) -> None:
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    _check(lib.tv_gdn_tree_verify_wy(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(parents), B, N, H, dk, dv,
        _DTYPES[q.dtype], _DTYPES[S0.dtype], float(q_scale), _ptr(out), _ptr(pseudo_v), _ptr(log_gamma),
        _ptr(err), _stream(stream)), "tv_gdn_tree_verify_wy")


def tv_gdn_commit(mode: int, accepted_path, accepted_len, parents, S0, err, *, node_states=None,
                  pseudo_v=None, log_gamma=None, k=None, io_dtype=None, N=None, stream=None) -> None:
    """Fork mode reads ``node_states``; WY mode reads ``pseudo_v``, ``log_gamma`` and ``k``."""
    B, H, dv, dk = S0.shape
    Lmax = accepted_path.shape[1]
    N = parents.shape[1] if N is None else N
    io = _DTYPES[k.dtype] if k is not None else (_DTYPES[io_dtype] if io_dtype is not None else
                                                  _DTYPES[S0.dtype])
    _check(lib.tv_gdn_commit(
        int(mode), _ptr(accepted_path), _ptr(accepted_len), Lmax, _ptr(parents), _ptr(node_states),
        _ptr(pseudo_v), _ptr(log_gamma), _ptr(k), _ptr(S0), B, N, H, dk, dv, io, _DTYPES[S0.dtype],
        _ptr(err), _stream(stream)), "tv_gdn_commit")


def tv_gdn_commit_layers(mode: int, accepted_path, accepted_len, parents, S0, err, *, node_states=None,
                         pseudo_v=None, log_gamma=None, k=None, io_dtype=None, N=None, stream=None) -> None:
    """One launch commits every layer: S0 [layers, B, H, dv, dk] and the mode's per-layer tensors
    with a leading layer dimension; path, lengths, parents and err are shared by the layers."""
    layers, B, H, dv, dk = S0.shape
    Lmax = accepted_path.shape[1]
    N = parents.shape[1] if N is None else N
    io = _DTYPES[k.dtype] if k is not None else (_DTYPES[io_dtype] if io_dtype is not None else
                                                  _DTYPES[S0.dtype])
    _check(lib.tv_gdn_commit_layers(
        int(mode), _ptr(accepted_path), _ptr(accepted_len), Lmax, _ptr(parents), _ptr(node_states),
        _ptr(pseudo_v), _ptr(log_gamma), _ptr(k), _ptr(S0), layers, B, N, H, dk, dv, io, _DTYPES[S0.dtype],
        _ptr(err), _stream(stream)), "tv_gdn_commit_layers")


def tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size=TV_BLOCK_SIZE) -> int:
    return int(lib.tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size))


def tv_tree_attn(q, k_new, v_new, k_cache, v_cache, block_table, prefix_len, parents, out,
                 workspace, err, rope_theta: float, sm_scale: float | None = None, stream=None) -> None:
    B, N, Hq, hd = q.shape
    Hkv = k_new.shape[2]
    num_blocks, _, bs, _ = k_cache.shape
    max_blocks = block_table.shape[1]
    scale = hd ** -0.5 if sm_scale is None else sm_scale
    _check(lib.tv_tree_attn(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table),
        max_blocks, _ptr(prefix_len), _ptr(parents), B, N, Hq, Hkv, hd, bs, float(rope_theta), float(scale),
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err),
        _stream(stream)), "tv_tree_attn")


def tv_tree_attn_static(q, k_new, v_new, k_cache, v_cache, block_table, prefix_len, parents, out,
                        err, rope_theta: float, sm_scale: float | None = None, stream=None) -> None:
    """``tv_tree_attn`` on the library's static scratch (no workspace, no allocation).  Raises
    TVError with TV_ERR_SCRATCH when the call needs more than TV_STATIC_SCRATCH_BYTES."""
    B, N, Hq, hd = q.shape
    Hkv = k_new.shape[2]
    num_blocks, _, bs, _ = k_cache.shape
    max_blocks = block_table.shape[1]
    scale = hd ** -0.5 if sm_scale is None else sm_scale
    _check(lib.tv_tree_attn_static(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table),
        max_blocks, _ptr(prefix_len), _ptr(parents), B, N, Hq, Hkv, hd, bs, float(rope_theta), float(scale),
        _ptr(out), _ptr(err), _stream(stream)), "tv_tree_attn_static")


def tv_kv_compact(k_cache, v_cache, block_table, prefix_len, parents, accepted_path, accepted_len,
                  slot_map, new_len, err, stream=None) -> None:
    num_blocks, Hkv, bs, hd = k_cache.shape
    B, max_blocks = block_table.shape
    N = parents.shape[1]
    Lmax = accepted_path.shape[1]
    _check(lib.tv_kv_compact(
        _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table), max_blocks, _ptr(prefix_len),
        _ptr(parents), N, _ptr(accepted_path), _ptr(accepted_len), Lmax, B, Hkv, hd, bs, _ptr(slot_map),
        _ptr(new_len), _ptr(err), _stream(stream)), "tv_kv_compact")


def tv_kv_compact_remap(k_cache, v_cache, block_table, block_table_out, prefix_len, parents, accepted_path,
                        accepted_len, slot_map, new_len, remapped, err, stream=None) -> None:
    """Compaction that exchanges whole blocks of ``block_table`` where it can (result rows in
    ``block_table_out``) and moves the other kept entries; ``remapped [B]`` counts exchanges."""
    num_blocks, Hkv, bs, hd = k_cache.shape
    B, max_blocks = block_table.shape
    N = parents.shape[1]
    Lmax = accepted_path.shape[1]
    _check(lib.tv_kv_compact_remap(
        _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table), _ptr(block_table_out), max_blocks,
        _ptr(prefix_len), _ptr(parents), N, _ptr(accepted_path), _ptr(accepted_len), Lmax, B, Hkv, hd, bs,
        _ptr(slot_map), _ptr(new_len), _ptr(remapped), _ptr(err), _stream(stream)), "tv_kv_compact_remap")


def tv_accept_walk(parents, draft_tokens, target_tokens, accepted_path, accepted_len, next_token, err,
                   stream=None) -> None:
    """parents, draft_tokens, target_tokens [B,N] int32 -> accepted_path [B,Lmax], accepted_len [B],
    next_token [B], err [B] (all int32)."""
    B, N = parents.shape
    _check(lib.tv_accept_walk(_ptr(parents), _ptr(draft_tokens), _ptr(target_tokens), B, N, accepted_path.shape[1],
                              _ptr(accepted_path), _ptr(accepted_len), _ptr(next_token), _ptr(err), _stream(stream)),
           "tv_accept_walk")


def tv_test_bounded_wait(max_polls: int, arrive: bool, status, elapsed_ns, stream=None) -> None:
    """One thread waits on a shared-memory barrier with the library's bounded wait (nothing
    arrives unless ``arrive``): status [1] int32 gets TV_OK or TV_ERR_TIMEOUT, elapsed_ns [1]
    int64 the device time of the wait.  max_polls 0 = the limit the kernels use."""
    _check(lib.tv_test_bounded_wait(int(max_polls), int(bool(arrive)), _ptr(status), _ptr(elapsed_ns),
                                    _stream(stream)), "tv_test_bounded_wait")
