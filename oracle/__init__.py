"""Python access to the CPU oracle of the verification step.

TEST INFRASTRUCTURE ONLY. The oracle (``specverify_oracle.c``) is the plain
fp64 restatement of the method that the CUDA library is checked against.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the CUDA library and its binding never
do, and there is no code path on which the oracle stands in for them.

Logit tensors are numpy arrays: ``float32`` for binary32 logits, ``uint16``
for bfloat16 bit patterns. The call releases the GIL (ctypes), so
``verify_threaded`` runs disjoint request slices on several host threads;
requests are independent, so the result is the same as one call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SOURCES = [os.path.join(_HERE, "specverify_oracle.c"), os.path.join(_HERE, "specverify_oracle.h")]
_LIB_DIR = os.path.join(_HERE, "_lib")
LIB_PATH = os.path.join(_LIB_DIR, "liboracle_specverify.so")

ORACLE_F32 = 0
ORACLE_BF16 = 1
KIND_ERROR, KIND_GREEDY, KIND_RESIDUAL, KIND_BONUS = -1, 0, 1, 2

# No fused multiply-add and no fast-math: the oracle's arithmetic is the plain
# double arithmetic written in the source, identical on x86-64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile the oracle with gcc into ``oracle/_lib`` (or ``out``)."""
    src = src or _SOURCES[0]
    out = out or LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = force or not os.path.exists(out) or any(
        os.path.getmtime(s) > os.path.getmtime(out) for s in _SOURCES if os.path.exists(s))
    if stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-I", _HERE, src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class _Detail(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "max_target", "lse_target", "argmax_target", "max_draft", "lse_draft",
        "p_x", "q_x", "alpha", "accept_margin", "w_total", "sample_margin", "kind", "tie_measure")]


def _bind(lib):
    lib.oracle_spec_verify.restype = ctypes.c_int
    lib.oracle_spec_verify.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Detail)]
    lib.oracle_spec_verify_onehot.restype = ctypes.c_int
    lib.oracle_spec_verify_onehot.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Detail)]
    lib.oracle_spec_verify_early.restype = ctypes.c_int
    lib.oracle_spec_verify_early.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Detail)]
    lib.oracle_spec_verify_tree.restype = ctypes.c_int
    lib.oracle_spec_verify_tree.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(_Detail)]
    lib.oracle_version.restype = ctypes.c_int
    return lib


def load_path(path: str):
    """Load an oracle build from ``path`` (used for rebuilt copies in tests)."""
    return _bind(ctypes.CDLL(path))


def load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_path(build())
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def dtype_code(logits: np.ndarray) -> int:
    if logits.dtype == np.float32:
        return ORACLE_F32
    if logits.dtype == np.uint16:
        return ORACLE_BF16
    raise TypeError(f"logits must be float32 or uint16 (bfloat16 bits), got {logits.dtype}")


def verify(target, draft, tokens, u_accept, u_sample, temperature, detail=False, lib=None):
    """Run the oracle on one batch. Returns ``(out_tokens, num_accepted, det)``.

    ``target`` [B, gamma+1, V], ``draft`` [B, gamma, V], ``tokens`` [B, gamma]
    int32, ``u_accept`` [B, gamma] float32, ``u_sample`` [B] float32,
    ``temperature`` [B] float32. ``det`` is a dict of numpy arrays (see
    ``specverify_oracle.h``) when ``detail`` is true, else None.
    """
    lib = lib or load()
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    B, G1, V = target.shape
    G = G1 - 1
    assert draft.shape == (B, G, V) and draft.dtype == target.dtype
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, G)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, G)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out_tokens = np.full((B, G1), -7, dtype=np.int32)
    num_acc = np.full((B,), -7, dtype=np.int32)
    det = None
    dptr = None
    if detail:
        det = _detail_arrays(B, G)
        d = _Detail(**{k: _ptr(v) for k, v in det.items()})
        dptr = ctypes.byref(d)
    rc = lib.oracle_spec_verify(
        _ptr(target), _ptr(draft), dtype_code(target), B, G, V,
        _ptr(tokens), _ptr(u_accept), _ptr(u_sample), _ptr(temperature),
        _ptr(out_tokens), _ptr(num_acc), dptr)
    if rc != 0:
        raise ValueError("oracle_spec_verify rejected its arguments")
    return out_tokens, num_acc, det


def _detail_arrays(B, G):
    G1 = G + 1
    return {
            "max_target": np.empty((B, G1)), "lse_target": np.empty((B, G1)),
            "argmax_target": np.empty((B, G1), dtype=np.int32),
            "max_draft": np.empty((B, G)), "lse_draft": np.empty((B, G)),
            "p_x": np.empty((B, G)), "q_x": np.empty((B, G)), "alpha": np.empty((B, G)),
            "accept_margin": np.empty((B, G)), "w_total": np.empty((B,)),
            "sample_margin": np.empty((B,)), "kind": np.empty((B,), dtype=np.int32),
            "tie_measure": np.empty((B,)),
    }


def verify_onehot(target, tokens, num_draft, u_accept, u_sample, temperature, detail=False, lib=None):
    """The oracle for deterministic (one-hot) proposals: ``num_draft`` [B]
    int32 proposals per request, no draft logits. Returns
    ``(out_tokens, num_accepted, det)`` like ``verify``."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    B, G1, V = target.shape
    G = G1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, G)
    num_draft = np.ascontiguousarray(num_draft, dtype=np.int32).reshape(B)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, G)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out_tokens = np.full((B, G1), -7, dtype=np.int32)
    num_acc = np.full((B,), -7, dtype=np.int32)
    det = None
    dptr = None
    if detail:
        det = _detail_arrays(B, G)
        d = _Detail(**{k: _ptr(v) for k, v in det.items()})
        dptr = ctypes.byref(d)
    rc = lib.oracle_spec_verify_onehot(
        _ptr(target), dtype_code(target), B, G, V, _ptr(tokens), _ptr(num_draft),
        _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens), _ptr(num_acc), dptr)
    if rc != 0:
        raise ValueError("oracle_spec_verify_onehot rejected its arguments")
    return out_tokens, num_acc, det


def verify_threaded(target, draft, tokens, u_accept, u_sample, temperature,
                    detail=False, threads=None, lib=None):
    """``verify`` over disjoint request slices on host threads, concatenated."""
    B = target.shape[0]
    threads = max(1, min(threads or os.cpu_count() or 1, B))
    if threads == 1:
        return verify(target, draft, tokens, u_accept, u_sample, temperature, detail, lib)
    bounds = np.linspace(0, B, threads + 1).astype(int)
    parts = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(lambda ab: verify(
            target[ab[0]:ab[1]], draft[ab[0]:ab[1]], tokens[ab[0]:ab[1]], u_accept[ab[0]:ab[1]],
            u_sample[ab[0]:ab[1]], temperature[ab[0]:ab[1]], detail, lib), parts))
    out = np.concatenate([r[0] for r in res])
    acc = np.concatenate([r[1] for r in res])
    det = None
    if detail:
        det = {k: np.concatenate([r[2][k] for r in res]) for k in res[0][2]}
    return out, acc, det


def verify_early(target, draft, tokens, u_accept, u_sample, temperature, num_draft=None, detail=False,
                 lib=None):
    """The early-exit oracle: positions in order, nothing read after the first
    rejection. ``draft`` None means one-hot proposals (``num_draft`` [B]
    required). Returns ``(out_tokens, num_accepted, det)`` like ``verify``."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    B, G1, V = target.shape
    G = G1 - 1
    if draft is not None:
        draft = np.ascontiguousarray(draft)
        assert draft.shape == (B, G, V) and draft.dtype == target.dtype
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, G)
    nd = None if num_draft is None else np.ascontiguousarray(num_draft, dtype=np.int32).reshape(B)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, G)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out_tokens = np.full((B, G1), -7, dtype=np.int32)
    num_acc = np.full((B,), -7, dtype=np.int32)
    det = None
    dptr = None
    if detail:
        det = _detail_arrays(B, G)
        d = _Detail(**{k: _ptr(v) for k, v in det.items()})
        dptr = ctypes.byref(d)
    rc = lib.oracle_spec_verify_early(
        _ptr(target), None if draft is None else _ptr(draft), dtype_code(target), B, G, V, _ptr(tokens),
        None if nd is None else _ptr(nd), _ptr(u_accept), _ptr(u_sample), _ptr(temperature),
        _ptr(out_tokens), _ptr(num_acc), dptr)
    if rc != 0:
        raise ValueError("oracle_spec_verify_early rejected its arguments")
    return out_tokens, num_acc, det


def verify_tree(target, tokens, parents, num_nodes, u_accept, u_sample, temperature, detail=False, lib=None):
    """The tree-verification oracle. ``target`` [B, G+1, V] (row j for node j),
    ``tokens``/``parents``/``u_accept`` [B, G] indexed by node - 1,
    ``num_nodes`` [B]. Returns ``(out_tokens, num_accepted, out_nodes, det)``."""
    lib = lib or load()
    target = np.ascontiguousarray(target)
    B, G1, V = target.shape
    G = G1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, G)
    parents = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, G)
    num_nodes = np.ascontiguousarray(num_nodes, dtype=np.int32).reshape(B)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, G)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32).reshape(B)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    out_tokens = np.full((B, G1), -7, dtype=np.int32)
    num_acc = np.full((B,), -7, dtype=np.int32)
    out_nodes = np.full((B, G), -7, dtype=np.int32)
    det = None
    dptr = None
    if detail:
        det = _detail_arrays(B, G)
        d = _Detail(**{k: _ptr(v) for k, v in det.items()})
        dptr = ctypes.byref(d)
    rc = lib.oracle_spec_verify_tree(
        _ptr(target), dtype_code(target), B, G, V, _ptr(tokens), _ptr(parents), _ptr(num_nodes),
        _ptr(u_accept), _ptr(u_sample), _ptr(temperature), _ptr(out_tokens), _ptr(num_acc), _ptr(out_nodes), dptr)
    if rc != 0:
        raise ValueError("oracle_spec_verify_tree rejected its arguments")
    return out_tokens, num_acc, out_nodes, det
