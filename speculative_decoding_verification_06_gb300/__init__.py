"""Python binding of libspecverify, the sm_103a speculative-decoding
verification step.

Argument marshalling only: every step of the verification runs in the CUDA
library (``_lib/libspecverify.so``, built by ``build.py``); this module turns
torch tensors into device pointers and the current CUDA stream, and calls the
C ABI of ``include/specverify.h`` by the same names. There is no fallback:
if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import build as _build

LIB_PATH = _build.LIB_PATH

SV_F32, SV_BF16 = 0, 1
SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_WORKSPACE, SV_ERR_TIMEOUT = range(6)
SV_ERR_SCRATCH_LIMIT = 6
SV_NOALLOC_SCRATCH_BYTES = 8 << 20
SV_PHASE_SLOTS = 10
SV_STATUS_BAD_REQUEST, SV_STATUS_TIMEOUT = 0x1, 0x2
SV_STATUS_TRUNCATED = 0x4
SV_MAX_GAMMA, SV_MAX_V = 64, 1 << 24
SV_PATH_AUTO, SV_PATH_ROWWISE, SV_PATH_STREAMING, SV_PATH_CLUSTER = 0, 1, 2, 3
KIND_INVALID, KIND_GREEDY, KIND_RESIDUAL, KIND_BONUS = -1, 0, 1, 2

EXPORTED = (
    "spec_verify_workspace_size", "spec_verify", "spec_verify_ex",
    "spec_verify_host_staging_size", "spec_verify_host", "spec_verify_last_launch_count",
    "spec_verify_status_string", "spec_verify_version", "spec_verify_noalloc",
    "spec_commit", "spec_ngram_propose", "spec_verify_onehot", "spec_verify_tree",
)


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_string(status)})")
        self.status = status


class _Debug(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "max_target", "lse_target", "argmax_target", "max_draft", "lse_draft", "p_x", "q_x",
        "w_total", "kind", "phase_ns")]


class _Options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("grid_ctas", ctypes.c_int32),
                ("peer_wait_us", ctypes.c_int32), ("early_exit", ctypes.c_int32),
                ("hold_flag", ctypes.c_void_p), ("num_draft", ctypes.c_void_p)]


_lib = None


def _declare(lib):
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    int_ = ctypes.c_int
    lib.spec_verify_workspace_size.argtypes = [int_, int_, int_, i32, ctypes.POINTER(sz)]
    lib.spec_verify_host_staging_size.argtypes = [int_, int_, int_, i32, ctypes.POINTER(sz)]
    common = [vp, vp, i32, int_, int_, int_, vp, vp, vp, vp, vp, vp]
    lib.spec_verify.argtypes = common + [vp, sz, vp]
    lib.spec_verify_ex.argtypes = common + [vp, sz, vp, ctypes.POINTER(_Debug), vp,
                                            ctypes.POINTER(_Options)]
    lib.spec_verify_host.argtypes = common + [vp, sz, vp]
    lib.spec_verify_noalloc.argtypes = common + [vp]
    lib.spec_commit.argtypes = [vp, vp, int_, int_, vp, int_, vp, vp, vp, vp]
    lib.spec_ngram_propose.argtypes = [vp, int_, int_, vp, int_, int_, int_, vp, vp, vp, vp]
    lib.spec_verify_onehot.argtypes = [vp, i32, int_, int_, int_, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.spec_verify_tree.argtypes = [vp, i32, int_, int_, int_, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp,
                                     ctypes.POINTER(_Debug), vp, ctypes.POINTER(_Options)]
    for name in ("spec_verify_workspace_size", "spec_verify_host_staging_size", "spec_verify",
                 "spec_verify_ex", "spec_verify_host", "spec_verify_noalloc", "spec_commit",
                 "spec_ngram_propose", "spec_verify_onehot", "spec_verify_tree"):
        getattr(lib, name).restype = i32
    lib.spec_verify_status_string.argtypes = [i32]
    lib.spec_verify_status_string.restype = ctypes.c_char_p
    lib.spec_verify_version.restype = int_
    lib.spec_verify_last_launch_count.restype = int_
    return lib


def load():
    """Load the built library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libspecverify is not built ({LIB_PATH} missing): "
                               "run __graft_entry__.build() or python -m "
                               "speculative_decoding_verification_06_gb300.build")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(status: int) -> str:
    return load().spec_verify_status_string(status).decode()


def version() -> int:
    return load().spec_verify_version()


def last_launch_count() -> int:
    return load().spec_verify_last_launch_count()


def _check(status: int, where: str):
    if status != SV_OK:
        raise SpecVerifyError(status, where)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16 (or 16-bit raw bits), got {t.dtype}")


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def workspace_size(B: int, gamma: int, V: int, dtype: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().spec_verify_workspace_size(B, gamma, V, dtype, ctypes.byref(n)),
           "spec_verify_workspace_size")
    return n.value


def host_staging_size(B: int, gamma: int, V: int, dtype: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().spec_verify_host_staging_size(B, gamma, V, dtype, ctypes.byref(n)),
           "spec_verify_host_staging_size")
    return n.value


@dataclass
class Outputs:
    out_tokens: object        # [B, gamma+1] int32
    out_num_accepted: object  # [B] int32
    debug: dict | None = None
    status: object = None     # [1] int32 device status word (spec_verify_ex)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def spec_verify(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature,
                out_tokens=None, out_num_accepted=None, workspace=None, stream=None,
                debug: bool = False, path: int = SV_PATH_AUTO, grid_ctas: int = 0,
                status=None, peer_wait_us: int = 0, hold_flag=None, num_draft=None,
                early_exit: bool = False) -> Outputs:
    """Verify one batch of CUDA tensors (see include/specverify.h).

    ``target_logits`` [B, gamma+1, V] and ``draft_logits`` [B, gamma, V]
    float32 or bfloat16, ``draft_tokens`` [B, gamma] int32, ``u_accept``
    [B, gamma] float32, ``u_sample`` [B] float32, ``temperature`` [B] float32,
    all contiguous on the current CUDA device. Outputs and workspace are
    allocated with torch when not given. With ``debug``, ``path``,
    ``grid_ctas``, ``status``, ``peer_wait_us`` or ``hold_flag`` (a CUDA int32
    tensor, checking only) the call goes through ``spec_verify_ex``.
    ``draft_logits`` None selects one-hot proposals (``spec_verify_onehot``)
    with ``num_draft`` [B] int32 proposals per request (None: gamma each).
    """
    import torch
    lib = load()
    B, G1, V = target_logits.shape
    G = G1 - 1
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    for t in (target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature, num_draft):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("every input must be a contiguous CUDA tensor")
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_size(B, G, V, dt)), dtype=torch.uint8, device=dev)
    s = _stream_handle(stream)
    args = (_ptr(target_logits), _ptr(draft_logits), dt, B, G, V, _ptr(draft_tokens),
            _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens),
            _ptr(out_num_accepted), _ptr(workspace), workspace.numel() * workspace.element_size(), s)
    dbg = None
    if (debug or path != SV_PATH_AUTO or grid_ctas or status is not None or peer_wait_us or hold_flag is not None
            or draft_logits is None or early_exit):
        d = _Debug()
        if debug:
            f64, f32, i32 = torch.float64, torch.float32, torch.int32
            dbg = {
                "max_target": torch.empty((B, G1), dtype=f32, device=dev),
                "lse_target": torch.empty((B, G1), dtype=f64, device=dev),
                "argmax_target": torch.empty((B, G1), dtype=i32, device=dev),
                "max_draft": torch.empty((B, G), dtype=f32, device=dev),
                "lse_draft": torch.empty((B, G), dtype=f64, device=dev),
                "p_x": torch.empty((B, G), dtype=f64, device=dev),
                "q_x": torch.empty((B, G), dtype=f64, device=dev),
                "w_total": torch.empty((B,), dtype=f64, device=dev),
                "kind": torch.empty((B,), dtype=i32, device=dev),
                "phase_ns": torch.zeros((SV_PHASE_SLOTS,), dtype=torch.int64, device=dev),
            }
            dbg["phase_ns"][0] = -1  # UINT64_MAX
            for k, v in dbg.items():
                setattr(d, k, v.data_ptr())
        o = _Options(path, grid_ctas, peer_wait_us, 1 if early_exit else 0, _ptr(hold_flag) or None,
                     _ptr(num_draft) or None)
        rc = lib.spec_verify_ex(*args, ctypes.byref(d), _ptr(status), ctypes.byref(o))
        _check(rc, "spec_verify_ex")
    else:
        _check(lib.spec_verify(*args), "spec_verify")
    return Outputs(out_tokens, out_num_accepted, dbg, status)


def spec_verify_host(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature,
                     out_tokens, out_num_accepted, staging, stream=None) -> None:
    """``spec_verify_host``: every array a CPU tensor (pinned for asynchronous
    copies), ``staging`` a CUDA uint8 tensor of ``host_staging_size`` bytes.
    Enqueues copies and kernels on ``stream``; the outputs are written when the
    stream reaches them."""
    lib = load()
    B, G1, V = target_logits.shape
    dt = _dtype_code(target_logits)
    for t in (target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature,
              out_tokens, out_num_accepted):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("spec_verify_host takes contiguous host tensors")
    rc = lib.spec_verify_host(
        _ptr(target_logits), _ptr(draft_logits), dt, B, G1 - 1, V, _ptr(draft_tokens),
        _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens),
        _ptr(out_num_accepted), _ptr(staging), staging.numel() * staging.element_size(),
        _stream_handle(stream))
    _check(rc, "spec_verify_host")


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature,
                        out_tokens, out_num_accepted, stream=None) -> None:
    """``spec_verify_noalloc``: the verification with the library's own static
    scratch, for callers that cannot allocate device memory. Every argument is
    a contiguous CUDA tensor the caller already owns (outputs included); this
    wrapper allocates nothing either. Calls that overlap on the GPU share the
    scratch and must not overlap."""
    lib = load()
    B, G1, V = target_logits.shape
    dt = _dtype_code(target_logits)
    for t in (target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature,
              out_tokens, out_num_accepted):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("every argument must be a contiguous CUDA tensor")
    rc = lib.spec_verify_noalloc(
        _ptr(target_logits), _ptr(draft_logits), dt, B, G1 - 1, V, _ptr(draft_tokens),
        _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens),
        _ptr(out_num_accepted), _stream_handle(stream))
    _check(rc, "spec_verify_noalloc")


def spec_commit(out_tokens, out_num_accepted, token_buf, seq_lens, next_input=None, status=None,
                stream=None) -> None:
    """``spec_commit``: append each request's emitted tokens to ``token_buf``
    [B, max_len] int32 at ``seq_lens`` [B] int32 (both updated in place on the
    GPU); ``next_input`` [B] int32 and ``status`` [1] int32 are optional CUDA
    tensors. Enqueued on ``stream``; nothing is copied to the host."""
    lib = load()
    B, G1 = out_tokens.shape
    for t in (out_tokens, out_num_accepted, token_buf, seq_lens):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("every array must be a contiguous CUDA tensor")
    rc = lib.spec_commit(_ptr(out_tokens), _ptr(out_num_accepted), B, G1 - 1, _ptr(token_buf),
                         token_buf.shape[1], _ptr(seq_lens), _ptr(next_input), _ptr(status),
                         _stream_handle(stream))
    _check(rc, "spec_commit")


def spec_ngram_propose(token_buf, seq_lens, gamma, n_min=2, n_max=5, draft_tokens=None, num_draft=None,
                       status=None, stream=None):
    """``spec_ngram_propose``: n-gram lookup drafts from each history
    ``token_buf[b, :seq_lens[b]]`` (CUDA int32 tensors). Returns
    ``(draft_tokens [B, gamma], num_draft [B])`` CUDA int32 tensors."""
    import torch
    lib = load()
    B, max_len = token_buf.shape
    for t in (token_buf, seq_lens):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("token_buf and seq_lens must be contiguous CUDA tensors")
    if draft_tokens is None:
        draft_tokens = torch.empty((B, gamma), dtype=torch.int32, device=token_buf.device)
    if num_draft is None:
        num_draft = torch.empty((B,), dtype=torch.int32, device=token_buf.device)
    rc = lib.spec_ngram_propose(_ptr(token_buf), B, max_len, _ptr(seq_lens), gamma, n_min, n_max,
                                _ptr(draft_tokens), _ptr(num_draft), _ptr(status), _stream_handle(stream))
    _check(rc, "spec_ngram_propose")
    return draft_tokens, num_draft


def spec_verify_onehot(target_logits, draft_tokens, num_draft, u_accept, u_sample, temperature,
                       out_tokens=None, out_num_accepted=None, workspace=None, stream=None) -> Outputs:
    """``spec_verify_onehot``: verification of deterministic proposals (q one-hot
    at each proposed token, no draft logits); ``num_draft`` [B] int32 CUDA
    tensor. Other arguments as ``spec_verify``."""
    import torch
    lib = load()
    B, G1, V = target_logits.shape
    G = G1 - 1
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    for t in (target_logits, draft_tokens, num_draft, u_accept, u_sample, temperature):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("every input must be a contiguous CUDA tensor")
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_size(B, G, V, dt)), dtype=torch.uint8, device=dev)
    rc = lib.spec_verify_onehot(_ptr(target_logits), dt, B, G, V, _ptr(draft_tokens), _ptr(num_draft),
                                _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens),
                                _ptr(out_num_accepted), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "spec_verify_onehot")
    return Outputs(out_tokens, out_num_accepted, None, None)


def spec_verify_tree(target_logits, node_tokens, parents, num_nodes, u_accept, u_sample, temperature,
                     out_tokens=None, out_num_accepted=None, out_nodes=None, workspace=None, debug=False,
                     status=None, stream=None, path: int = SV_PATH_AUTO, grid_ctas: int = 0, peer_wait_us: int = 0,
                     hold_flag=None):
    """``spec_verify_tree``: verification of a candidate tree per request (see
    include/specverify.h). ``target_logits`` [B, G+1, V], ``node_tokens`` /
    ``parents`` / ``u_accept`` [B, G] indexed by node - 1, ``num_nodes`` [B];
    CUDA tensors. The workspace is allocated with torch when not given.
    Returns ``(Outputs, out_nodes)``."""
    import torch
    lib = load()
    B, G1, V = target_logits.shape
    G = G1 - 1
    dt = _dtype_code(target_logits)
    dev = target_logits.device
    for t in (target_logits, node_tokens, parents, num_nodes, u_accept, u_sample, temperature):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("every input must be a contiguous CUDA tensor")
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_nodes is None:
        out_nodes = torch.empty((B, G), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(16, workspace_size(B, G, V, dt)), dtype=torch.uint8, device=dev)
    d = _Debug()
    dbg = None
    if debug:
        f64, f32, i32 = torch.float64, torch.float32, torch.int32
        dbg = {
            "max_target": torch.empty((B, G1), dtype=f32, device=dev),
            "lse_target": torch.empty((B, G1), dtype=f64, device=dev),
            "argmax_target": torch.empty((B, G1), dtype=i32, device=dev),
            "max_draft": torch.empty((B, G), dtype=f32, device=dev),
            "lse_draft": torch.empty((B, G), dtype=f64, device=dev),
            "p_x": torch.empty((B, G), dtype=f64, device=dev),
            "q_x": torch.empty((B, G), dtype=f64, device=dev),
            "w_total": torch.empty((B,), dtype=f64, device=dev),
            "kind": torch.empty((B,), dtype=i32, device=dev),
        }
        for k, v in dbg.items():
            setattr(d, k, v.data_ptr())
    o = _Options(path, grid_ctas, peer_wait_us, 0, _ptr(hold_flag) or None, None)
    rc = lib.spec_verify_tree(_ptr(target_logits), dt, B, G, V, _ptr(node_tokens), _ptr(parents), _ptr(num_nodes),
                              _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens),
                              _ptr(out_num_accepted), _ptr(out_nodes), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream), ctypes.byref(d),
                              _ptr(status), ctypes.byref(o))
    _check(rc, "spec_verify_tree")
    return Outputs(out_tokens, out_num_accepted, dbg, status), out_nodes
