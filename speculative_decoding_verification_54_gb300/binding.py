"""Thin ctypes binding of libspecverify (spec_verify.h), same names as the C ABI.

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of the shared library.  Tensors are torch CUDA tensors (PyTorch is
used for device memory and streams); raw integer device addresses are also
accepted where noted.  A missing or unloadable library raises immediately —
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

SPEC_F32, SPEC_BF16 = 0, 1
SPEC_OK = 0
SPEC_ERR_INVALID_ARG = -1
SPEC_ERR_UNSUPPORTED = -2
SPEC_ERR_ALIGNMENT = -3
SPEC_ERR_WORKSPACE = -4
SPEC_ERR_CUDA = -5
SPEC_ERR_TIMEOUT = -6
SPEC_ERR_DEVICE_INPUT = -7
SPEC_ERR_STATE = -8
SPEC_ERR_DEVICE_BOUNDS = -9
MAX_GAMMA = 31

EXPORTED = (
    "spec_verify_workspace_bytes", "spec_verify_workspace_init", "spec_verify_greedy",
    "spec_verify_sample", "spec_verify_status", "spec_verify_error_string",
    "spec_verify_version", "spec_verify_selftest_timeout", "spec_verify_sample_reduce_only",
    "spec_verify_sample_noalloc", "spec_verify_lmhead_sample", "spec_verify_lmhead_gemm_only",
    "spec_verify_greedy_multi", "spec_round_update", "spec_verify_topkp_workspace_bytes",
    "spec_verify_sample_topkp", "spec_centroid_head_workspace_bytes", "spec_centroid_head",
    "spec_verify_sparse_workspace_bytes", "spec_verify_sample_sparse",
)


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})" if what else f"{error_string(code)} ({code})")


_lib = None
_vp, _sz, _i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libspecverify not built ({path} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    lib.spec_verify_workspace_bytes.argtypes = [_i, _i, _i, _i, ctypes.POINTER(_sz)]
    lib.spec_verify_workspace_init.argtypes = [_vp, _sz, _vp]
    lib.spec_verify_greedy.argtypes = [_vp, _i, _vp, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]
    lib.spec_verify_greedy_multi.argtypes = [_vp, _i, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_verify_sample.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i,
                                       _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_verify_sample_reduce_only.argtypes = list(lib.spec_verify_sample.argtypes)
    lib.spec_verify_sample_noalloc.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i,
                                               _vp, _vp, _vp, _vp]
    lib.spec_verify_lmhead_sample.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                              _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_verify_lmhead_gemm_only.argtypes = list(lib.spec_verify_lmhead_sample.argtypes)
    lib.spec_round_update.argtypes = [_vp, _vp, _i, _i, _i, _vp, _vp]
    lib.spec_verify_topkp_workspace_bytes.argtypes = [_i, _i, _i, ctypes.POINTER(_sz)]
    lib.spec_verify_sample_topkp.argtypes = [_vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, ctypes.c_float,
                                             _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_centroid_head_workspace_bytes.argtypes = [_i, _i, _i, ctypes.POINTER(_sz)]
    lib.spec_centroid_head.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                                       _vp, _sz, _vp]
    lib.spec_verify_sparse_workspace_bytes.argtypes = [_i, _i, _i, ctypes.POINTER(_sz)]
    lib.spec_verify_sample_sparse.argtypes = [_vp, _i, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i,
                                              _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_verify_status.argtypes = [_vp, _vp]
    lib.spec_verify_error_string.argtypes = [_i]
    lib.spec_verify_error_string.restype = ctypes.c_char_p
    lib.spec_verify_version.argtypes = []
    lib.spec_verify_selftest_timeout.argtypes = [_vp, _sz, _vp]
    for name in EXPORTED:
        if name not in ("spec_verify_error_string",):
            getattr(lib, name).restype = _i
    _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().spec_verify_error_string(int(code)).decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t):
    """Device address of a tensor (or an int address), None for None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, f"logits dtype {t.dtype}")


def _check(code: int, what: str) -> int:
    if code != SPEC_OK:
        raise SpecVerifyError(code, what)
    return code


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


# ---------------------------------------------------------------------------
# the C ABI, one wrapper per entry point
# ---------------------------------------------------------------------------
def spec_verify_workspace_bytes(B: int, gamma: int, V: int, H: int = 0) -> int:
    out = _sz(0)
    _check(load().spec_verify_workspace_bytes(B, gamma, V, H, ctypes.byref(out)),
           "spec_verify_workspace_bytes")
    return out.value


def spec_verify_workspace_init(workspace, stream=None) -> None:
    _check(load().spec_verify_workspace_init(_ptr(workspace), _nbytes(workspace), _stream(stream)),
           "spec_verify_workspace_init")


def make_workspace(B: int, gamma: int, V: int, H: int = 0, device="cuda"):
    """Allocate (torch) and zero a workspace big enough for (B, gamma, V, H)."""
    import torch
    n = spec_verify_workspace_bytes(B, gamma, V, H)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def spec_verify_greedy(target_logits, draft_tokens, out_tokens, out_num_accepted, workspace,
                       stream=None) -> None:
    """target_logits [B, gamma+1, V] (fp32/bf16), draft_tokens [B, gamma] int32."""
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    _check(load().spec_verify_greedy(_ptr(target_logits), _dtype_code(target_logits),
                                     _ptr(draft_tokens), B, gamma, V, _ptr(out_tokens),
                                     _ptr(out_num_accepted), _ptr(workspace), _nbytes(workspace),
                                     _stream(stream)), "spec_verify_greedy")


def spec_verify_greedy_multi(target_logits, draft_tokens, out_tokens, out_num_accepted, workspace,
                             out_choice=None, stream=None) -> None:
    """target_logits [B, n_cand, gamma+1, V] (fp32/bf16), draft_tokens
    [B, n_cand, gamma] int32; out_tokens [B, gamma+1], out_num_accepted [B],
    optional out_choice [B] int32.  Workspace: make_workspace(B * n_cand, gamma, V)."""
    B, n_cand, g1, V = target_logits.shape
    _check(load().spec_verify_greedy_multi(_ptr(target_logits), _dtype_code(target_logits),
                                           _ptr(draft_tokens), B, n_cand, g1 - 1, V, _ptr(out_tokens),
                                           _ptr(out_num_accepted), _ptr(out_choice), _ptr(workspace),
                                           _nbytes(workspace), _stream(stream)), "spec_verify_greedy_multi")


def spec_verify_sample(target_logits, draft_logits, draft_tokens, temperature, u_accept,
                       u_resample, out_tokens, out_num_accepted, workspace, out_debug=None,
                       stream=None) -> None:
    """target_logits [B, gamma+1, V], draft_logits [B, gamma, V] (same dtype),
    draft_tokens [B, gamma] int32, temperature [B], u_accept [B, gamma],
    u_resample [B] (float32); out_tokens [B, gamma+1], out_num_accepted [B]
    int32; optional out_debug [B, gamma+1, 4] float32."""
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, "target and draft logits differ in dtype")
    _check(load().spec_verify_sample(_ptr(target_logits), _ptr(draft_logits),
                                     _dtype_code(target_logits), _ptr(draft_tokens),
                                     _ptr(temperature), _ptr(u_accept), _ptr(u_resample), B, gamma, V,
                                     _ptr(out_tokens), _ptr(out_num_accepted), _ptr(out_debug),
                                     _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "spec_verify_sample")


def spec_verify_topkp_workspace_bytes(B: int, gamma: int, V: int) -> int:
    out = _sz(0)
    _check(load().spec_verify_topkp_workspace_bytes(B, gamma, V, ctypes.byref(out)),
           "spec_verify_topkp_workspace_bytes")
    return out.value


def make_topkp_workspace(B: int, gamma: int, V: int, device="cuda"):
    """Allocate (torch) and zero a workspace for spec_verify_sample_topkp."""
    import torch
    n = spec_verify_topkp_workspace_bytes(B, gamma, V)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def spec_verify_sample_topkp(target_logits, draft_logits, draft_tokens, temperature, u_accept,
                             u_resample, top_k, top_p, out_tokens, out_num_accepted, workspace,
                             out_debug=None, stream=None) -> None:
    """spec_verify_sample with top-k / top-p truncation of p and q (same
    arguments plus top_k, top_p).  Workspace: make_topkp_workspace(B, gamma, V)."""
    B, g1, V = target_logits.shape
    if draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, "target and draft logits differ in dtype")
    _check(load().spec_verify_sample_topkp(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_tokens),
        _ptr(temperature), _ptr(u_accept), _ptr(u_resample), B, g1 - 1, V, int(top_k), float(top_p),
        _ptr(out_tokens), _ptr(out_num_accepted), _ptr(out_debug), _ptr(workspace), _nbytes(workspace),
        _stream(stream)), "spec_verify_sample_topkp")


def spec_verify_sample_reduce_only(target_logits, draft_logits, draft_tokens, temperature,
                                   u_accept, u_resample, out_tokens, out_num_accepted, workspace,
                                   out_debug=None, stream=None) -> None:
    """Enqueue only the row-reducer kernel of spec_verify_sample (timing aid)."""
    B, g1, V = target_logits.shape
    _check(load().spec_verify_sample_reduce_only(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_tokens),
        _ptr(temperature), _ptr(u_accept), _ptr(u_resample), B, g1 - 1, V, _ptr(out_tokens),
        _ptr(out_num_accepted), _ptr(out_debug), _ptr(workspace), _nbytes(workspace),
        _stream(stream)), "spec_verify_sample_reduce_only")


def spec_verify_sample_noalloc(target_logits, draft_logits, draft_tokens, temperature, u_accept,
                               u_resample, out_tokens, out_num_accepted, out_debug=None,
                               stream=None) -> None:
    """spec_verify_sample for callers that cannot allocate device memory: no
    workspace, the library's built-in 16 MiB scratch instead.  Calls must not
    overlap on the GPU (they share that scratch)."""
    B, g1, V = target_logits.shape
    if draft_logits.dtype != target_logits.dtype:
        raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, "target and draft logits differ in dtype")
    _check(load().spec_verify_sample_noalloc(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_tokens),
        _ptr(temperature), _ptr(u_accept), _ptr(u_resample), B, g1 - 1, V, _ptr(out_tokens),
        _ptr(out_num_accepted), _ptr(out_debug), _stream(stream)), "spec_verify_sample_noalloc")


def _lmhead_call(fn, name, hidden, W, draft_logits, draft_tokens, temperature, u_accept,
                 u_resample, out_tokens, out_num_accepted, workspace, out_debug, stream):
    import torch
    B, gamma, V = draft_logits.shape
    H = W.shape[1]
    for t, what in ((hidden, "hidden"), (W, "W"), (draft_logits, "draft_logits")):
        if t.dtype != torch.bfloat16:
            raise SpecVerifyError(SPEC_ERR_UNSUPPORTED, f"{what} must be bfloat16, got {t.dtype}")
    if tuple(hidden.shape) != (B * (gamma + 1), H) or W.shape[0] != V:
        raise SpecVerifyError(SPEC_ERR_INVALID_ARG, f"{name}: hidden {tuple(hidden.shape)}, "
                              f"W {tuple(W.shape)}, draft_logits {tuple(draft_logits.shape)}")
    _check(fn(_ptr(hidden), _ptr(W), _ptr(draft_logits), _ptr(draft_tokens), _ptr(temperature),
              _ptr(u_accept), _ptr(u_resample), B, gamma, V, H, _ptr(out_tokens),
              _ptr(out_num_accepted), _ptr(out_debug), _ptr(workspace), _nbytes(workspace),
              _stream(stream)), name)


def spec_verify_lmhead_sample(hidden, W, draft_logits, draft_tokens, temperature, u_accept,
                              u_resample, out_tokens, out_num_accepted, workspace, out_debug=None,
                              stream=None) -> None:
    """Sampling verification with the target logits computed in the call as
    hidden @ W^T: hidden [B*(gamma+1), H], W [V, H], draft_logits [B, gamma, V]
    (all bfloat16); the other arguments as spec_verify_sample.  The workspace
    comes from make_workspace(B, gamma, V, H)."""
    _lmhead_call(load().spec_verify_lmhead_sample, "spec_verify_lmhead_sample", hidden, W,
                 draft_logits, draft_tokens, temperature, u_accept, u_resample, out_tokens,
                 out_num_accepted, workspace, out_debug, stream)


def spec_verify_lmhead_gemm_only(hidden, W, draft_logits, draft_tokens, temperature, u_accept,
                                 u_resample, out_tokens, out_num_accepted, workspace,
                                 out_debug=None, stream=None) -> None:
    """Enqueue only the lm_head GEMM kernel of spec_verify_lmhead_sample (timing aid)."""
    _lmhead_call(load().spec_verify_lmhead_gemm_only, "spec_verify_lmhead_gemm_only", hidden, W,
                 draft_logits, draft_tokens, temperature, u_accept, u_resample, out_tokens,
                 out_num_accepted, workspace, out_debug, stream)


class SpecRoundState(ctypes.Structure):
    """spec_round_state: per-sequence host bookkeeping of the round driver."""
    _fields_ = [("gamma", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("seq_len", ctypes.c_int64), ("kv_len", ctypes.c_int64)]


def spec_round_update(states, num_accepted, gamma_min: int, gamma_max: int):
    """Host round bookkeeping.  ``states``: a ctypes array of SpecRoundState
    (updated in place); ``num_accepted``: host int sequence.  Returns the
    number of KV entries to keep per sequence.  Raises SpecVerifyError
    (SPEC_ERR_STATE, with the first inconsistent sequence) on bad bookkeeping."""
    B = len(states)
    n = (ctypes.c_int32 * B)(*[int(x) for x in num_accepted])
    keep = (ctypes.c_int64 * B)()
    bad = ctypes.c_int(-1)
    code = load().spec_round_update(ctypes.cast(states, _vp) if B else None, ctypes.cast(n, _vp),
                                    B, gamma_min, gamma_max, ctypes.cast(keep, _vp), ctypes.byref(bad))
    _check(code, f"spec_round_update (first bad sequence {bad.value})" if code == SPEC_ERR_STATE
           else "spec_round_update")
    return list(keep)


def spec_verify_status(workspace, stream=None) -> int:
    """Synchronise and return (and clear) the device-side status code."""
    return load().spec_verify_status(_ptr(workspace), _stream(stream))


def spec_verify_version() -> int:
    return load().spec_verify_version()


def spec_verify_selftest_timeout(workspace, stream=None) -> None:
    _check(load().spec_verify_selftest_timeout(_ptr(workspace), _nbytes(workspace), _stream(stream)),
           "spec_verify_selftest_timeout")


# ---------------------------------------------------------------------------
# centroid-masked sparse draft head and verification against its sparse rows
# ---------------------------------------------------------------------------
def _aligned_zeros(n: int, device):
    import torch
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def spec_centroid_head_workspace_bytes(R: int, n_clusters: int, top_k: int) -> int:
    out = _sz(0)
    _check(load().spec_centroid_head_workspace_bytes(R, n_clusters, top_k, ctypes.byref(out)),
           "spec_centroid_head_workspace_bytes")
    return out.value


def make_centroid_head_workspace(R: int, n_clusters: int, top_k: int, device="cuda"):
    """Allocate (torch) and zero a workspace for spec_centroid_head."""
    return _aligned_zeros(spec_centroid_head_workspace_bytes(R, n_clusters, top_k), device)


def spec_centroid_head(hidden, centroids, W_ord, cluster_off, ord2tok, top_k, out_tok, out_logit,
                       out_count, workspace, stream=None) -> None:
    """hidden [R, H], centroids [n_clusters, H], W_ord [V, H] (bf16); cluster_off
    int32 [n_clusters+1]; ord2tok int32 [V]; out_tok int32 / out_logit f32
    [R, max_cand]; out_count int32 [R]."""
    R, H = hidden.shape
    V = W_ord.shape[0]
    n_clusters = centroids.shape[0]
    max_cand = out_tok.shape[1]
    _check(load().spec_centroid_head(
        _ptr(hidden), _ptr(centroids), _ptr(W_ord), _ptr(cluster_off), _ptr(ord2tok), R, H, V, n_clusters,
        int(top_k), max_cand, _ptr(out_tok), _ptr(out_logit), _ptr(out_count), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "spec_centroid_head")


def spec_verify_sparse_workspace_bytes(B: int, gamma: int, V: int) -> int:
    out = _sz(0)
    _check(load().spec_verify_sparse_workspace_bytes(B, gamma, V, ctypes.byref(out)),
           "spec_verify_sparse_workspace_bytes")
    return out.value


def make_sparse_workspace(B: int, gamma: int, V: int, device="cuda"):
    """Allocate (torch) and zero a workspace for spec_verify_sample_sparse."""
    return _aligned_zeros(spec_verify_sparse_workspace_bytes(B, gamma, V), device)


def spec_verify_sample_sparse(target_logits, cand_tok, cand_logit, cand_count, draft_tokens, temperature,
                              u_accept, u_resample, out_tokens, out_num_accepted, workspace, out_debug=None,
                              stream=None) -> None:
    """target_logits [B, gamma+1, V] (fp32/bf16); cand_tok int32 / cand_logit
    f32 [B*gamma, stride] (tokens ascending per row); cand_count int32
    [B*gamma]; the rest as spec_verify_sample."""
    B, g1, V = target_logits.shape
    _check(load().spec_verify_sample_sparse(
        _ptr(target_logits), _dtype_code(target_logits), _ptr(cand_tok), _ptr(cand_logit), _ptr(cand_count),
        cand_tok.shape[1], _ptr(draft_tokens), _ptr(temperature), _ptr(u_accept), _ptr(u_resample), B, g1 - 1, V,
        _ptr(out_tokens), _ptr(out_num_accepted), _ptr(out_debug), _ptr(workspace), _nbytes(workspace),
        _stream(stream)), "spec_verify_sample_sparse")
