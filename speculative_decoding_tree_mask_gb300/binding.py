"""ctypes binding of ``libspecverify.so`` (C ABI in ``include/spec_verify.h``).

Argument marshalling only: every step runs in the library's CUDA kernels. Tensors are torch
CUDA tensors (torch provides device memory and streams); the functions keep the C names.
Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libspecverify.so")
DEBUG_LIBRARY = os.path.join(HERE, "libspecverify_debug.so")   # checked flavour (SPEC_DEBUG)

SPEC_OK, SPEC_ERR_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA, SPEC_ERR_WORKSPACE = 0, -1, -2, -3, -4
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_DRAFT_POINT, SPEC_DRAFT_PROBS_F32, SPEC_DRAFT_LOGITS = 0, 1, 2
SPEC_REQ_OK, SPEC_REQ_BAD_PARENT, SPEC_REQ_BAD_TOKEN, SPEC_REQ_BAD_ROW, SPEC_REQ_BAD_UNIFORM = \
    0, 1, 2, 3, 4
SPEC_ROW_NAN, SPEC_ROW_POSINF, SPEC_ROW_ALL_NEGINF = 1, 2, 4
KERNEL_CLASSES = ("tree_mask", "row_stats", "draft_stats", "walk_greedy", "walk_sample",
                  "lazy_greedy", "lazy_sample", "kv_commit", "budget")
SPEC_F16 = 2
SPEC_REQ_BAD_SLOT = 5
SPEC_REQ_BAD_BUDGET = 6
SPEC_REQ_INTERNAL = 7   # debug builds: a kernel's own consistency check failed
DBG_INDEX, DBG_ARRIVAL, DBG_WALK = 1, 2, 4
SPEC_KV_NHD, SPEC_KV_HND = 0, 1
SPEC_CACHE_SAME, SPEC_CACHE_FP8_E4M3, SPEC_CACHE_FP8_E5M2 = 0, 1, 2
SPEC_SCALE_TENSOR, SPEC_SCALE_PER_TOKEN = 0, 1



class BudgetParams(ctypes.Structure):
    """spec_budget_params: target ratio, moving-average weight, dead band, limits, step."""
    _fields_ = [("target", ctypes.c_double), ("alpha", ctypes.c_double),
                ("band", ctypes.c_double), ("n_min", ctypes.c_int32),
                ("n_max", ctypes.c_int32), ("step", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code})")


def load() -> ctypes.CDLL:
    """Open the CUDA library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIBRARY)
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every call of this module through another build of the library (for example the
    debug flavour, DEBUG_LIBRARY) inside the `with` block. Handles are tied to the build that
    created them: make them inside the block."""
    global _lib
    lib = _open(path)
    with _lock:
        prev = _lib
        _lib = lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def _open(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first "
            "(python -m speculative_decoding_tree_mask_gb300.build)")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.spec_verify_init.argtypes = [ctypes.POINTER(P), i32, i32, i64, i32]
    lib.spec_verify_destroy.argtypes = [P]
    lib.spec_build_tree_mask.argtypes = [P, P, i32, i32, P, P, P, P]
    lib.spec_verify_greedy.argtypes = [P, P, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
    lib.spec_verify_sample.argtypes = [P, P, i32, i32, i32, i64, P, P, P, i32, i32, f32,
                                       P, P, P, P, P, P, P]
    lib.spec_row_stats.argtypes = [P, P, i32, i32, i32, i64, f32, P, P, P, P, P, P, P, P]
    lib.spec_verify_greedy_lazy.argtypes = lib.spec_verify_greedy.argtypes
    lib.spec_kv_commit.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, i32,
                                   i32, i32, i64, P, i32, P, P, P, i32, P, P]
    lib.spec_verify_sample_lazy.argtypes = lib.spec_verify_sample.argtypes
    lib.spec_set_node_budget.argtypes = [P, P]
    lib.spec_budget_update.argtypes = [P, ctypes.POINTER(BudgetParams), P, P, P, i32,
                                       i32, P, P, P]
    lib.spec_profile_begin.argtypes = [P]
    lib.spec_profile_end.argtypes = [P, P, P]
    lib.spec_error_string.argtypes = [i32]
    lib.spec_error_string.restype = ctypes.c_char_p
    lib.spec_debug_build.argtypes = []
    lib.spec_debug_inject_arrival.argtypes = [P, i32, i32]
    lib.spec_debug_words.argtypes = [P, P, i32, P]
    return lib


def error_string(code: int) -> str:
    return load().spec_error_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != SPEC_OK:
        raise SpecError(rc, where)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _ptr_dev_or_pinned(t):
    """Logits of the lazy calls: a CUDA tensor, or a page-locked host tensor (the library
    checks that the device maps it at the same address)."""
    if t is None:
        return None
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("logits must be a CUDA tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _hdev(h) -> str:
    return f"cuda:{h.device}"


def _same_device(tensors, device, where):
    """Every CUDA tensor of a call must live on `device` (the handle's GPU, or for the
    handle-free call the logits' GPU): the kernels run there and take raw addresses."""
    dev = torch.device(device)
    for t in tensors:
        if t is not None and t.is_cuda and t.device != dev:
            raise ValueError(f"{where}: a tensor is on {t.device}, the call runs on {dev}")


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _i32(t, name):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return t


class Handle:
    """Owner of a ``spec_handle`` (workspace for B <= max_B, N <= max_N, V <= max_V)."""

    def __init__(self, max_B: int, max_N: int, max_V: int, device: int = 0):
        h = ctypes.c_void_p()
        _check(load().spec_verify_init(ctypes.byref(h), int(max_B), int(max_N), int(max_V),
                                       int(device)), "spec_verify_init")
        self.ptr = h
        self.device = int(device)
        self.max_B, self.max_N, self.max_V = int(max_B), int(max_N), int(max_V)

    def close(self):
        if self.ptr is not None and self.ptr.value:
            load().spec_verify_destroy(self.ptr)
        self.ptr = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spec_verify_init(max_B: int, max_N: int, max_V: int, device: int = 0) -> Handle:
    return Handle(max_B, max_N, max_V, device)


def spec_verify_destroy(h: Handle):
    h.close()


def spec_build_tree_mask(h: Handle, parent, anc_mask, depth, status, stream=None):
    """parent int32 [B, N] -> anc_mask int64 [B, N] (uint64 bit patterns), depth int32 [B, N],
    status int32 [B]."""
    B, N = parent.shape
    _same_device((parent, anc_mask, depth, status), _hdev(h), "spec_build_tree_mask")
    if anc_mask.dtype not in (torch.int64, getattr(torch, "uint64", torch.int64)):
        raise TypeError("anc_mask must be a 64-bit integer tensor")
    _check(load().spec_build_tree_mask(h.ptr, _ptr(_i32(parent, "parent")), B, N, _ptr(anc_mask),
                                       _ptr(_i32(depth, "depth")), _ptr(_i32(status, "status")),
                                       _stream(stream, parent.device)), "spec_build_tree_mask")


def spec_verify_greedy(h: Handle, logits, draft_token, parent, accept_len, out_tokens, kv_commit,
                       bonus, status, stream=None):
    B, N, V = logits.shape
    _same_device((logits, draft_token, parent, accept_len, out_tokens, kv_commit, bonus, status),
                 _hdev(h), "spec_verify_greedy")
    _check(load().spec_verify_greedy(
        h.ptr, _ptr(logits), _dtype_code(logits), B, N, V,
        _ptr(_i32(draft_token, "draft_token")), _ptr(_i32(parent, "parent")),
        _ptr(accept_len), _ptr(out_tokens), _ptr(kv_commit), _ptr(bonus), _ptr(status),
        _stream(stream, logits.device)), "spec_verify_greedy")


def spec_verify_sample(h: Handle, logits, draft_token, parent, temperature: float, uniforms,
                       accept_len, out_tokens, kv_commit, bonus, status, draft=None,
                       draft_kind: int = SPEC_DRAFT_POINT, stream=None):
    B, N, V = logits.shape
    _same_device((logits, draft_token, parent, uniforms, accept_len, out_tokens, kv_commit,
                  bonus, status, draft), _hdev(h), "spec_verify_sample")
    ddt = 0
    if draft is not None and draft_kind == SPEC_DRAFT_LOGITS:
        ddt = _dtype_code(draft)
    if draft is not None and draft_kind == SPEC_DRAFT_PROBS_F32 and draft.dtype != torch.float32:
        raise TypeError("draft probabilities must be float32")
    _check(load().spec_verify_sample(
        h.ptr, _ptr(logits), _dtype_code(logits), B, N, V,
        _ptr(_i32(draft_token, "draft_token")), _ptr(_i32(parent, "parent")), _ptr(draft),
        int(draft_kind), ddt, float(temperature), _ptr(uniforms), _ptr(accept_len),
        _ptr(out_tokens), _ptr(kv_commit), _ptr(bonus), _ptr(status),
        _stream(stream, logits.device)), "spec_verify_sample")


def spec_verify_greedy_lazy(h: Handle, logits, draft_token, parent, accept_len, out_tokens,
                            kv_commit, bonus, status, stream=None):
    """Greedy verification reading only the rows on the accepted path."""
    B, N, V = logits.shape
    _same_device((logits, draft_token, parent, accept_len, out_tokens, kv_commit, bonus, status),
                 _hdev(h), "spec_verify_greedy_lazy")
    _check(load().spec_verify_greedy_lazy(
        h.ptr, _ptr_dev_or_pinned(logits), _dtype_code(logits), B, N, V,
        _ptr(_i32(draft_token, "draft_token")), _ptr(_i32(parent, "parent")),
        _ptr(accept_len), _ptr(out_tokens), _ptr(kv_commit), _ptr(bonus), _ptr(status),
        _stream(stream, draft_token.device)), "spec_verify_greedy_lazy")


def spec_verify_sample_lazy(h: Handle, logits, draft_token, parent, temperature: float, uniforms,
                            accept_len, out_tokens, kv_commit, bonus, status, draft=None,
                            draft_kind: int = SPEC_DRAFT_POINT, stream=None):
    """Sampling verification reading only the rows the walk visits."""
    B, N, V = logits.shape
    _same_device((logits, draft_token, parent, uniforms, accept_len, out_tokens, kv_commit,
                  bonus, status, draft), _hdev(h), "spec_verify_sample_lazy")
    ddt = 0
    if draft is not None and draft_kind == SPEC_DRAFT_LOGITS:
        ddt = _dtype_code(draft)
    if draft is not None and draft_kind == SPEC_DRAFT_PROBS_F32 and draft.dtype != torch.float32:
        raise TypeError("draft probabilities must be float32")
    _check(load().spec_verify_sample_lazy(
        h.ptr, _ptr_dev_or_pinned(logits), _dtype_code(logits), B, N, V,
        _ptr(_i32(draft_token, "draft_token")), _ptr(_i32(parent, "parent")),
        _ptr_dev_or_pinned(draft), int(draft_kind), ddt, float(temperature), _ptr(uniforms),
        _ptr(accept_len), _ptr(out_tokens), _ptr(kv_commit), _ptr(bonus), _ptr(status),
        _stream(stream, draft_token.device)), "spec_verify_sample_lazy")


def spec_row_stats(h: Handle, logits, N: int, temperature: float, row_max, row_sum, row_argmax,
                   row_flags, draft_token=None, parent=None, child_prob=None, stream=None):
    """logits [rows, V] (or [B, N, V]) -> per-row max, sum, argmax, flags; optional gather of
    p_parent(token) at every child into child_prob [B, N]."""
    V = logits.shape[-1]
    rows = logits.numel() // V
    _same_device((logits, row_max, row_sum, row_argmax, row_flags, draft_token, parent,
                  child_prob), _hdev(h), "spec_row_stats")
    _check(load().spec_row_stats(
        h.ptr, _ptr(logits), _dtype_code(logits), rows, int(N), V, float(temperature),
        _ptr(draft_token), _ptr(parent), _ptr(row_max), _ptr(row_sum), _ptr(row_argmax),
        _ptr(row_flags), _ptr(child_prob), _stream(stream, logits.device)), "spec_row_stats")


def _kv_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return SPEC_F16
    return _dtype_code(t)


def spec_kv_commit(h: Handle, src_k, src_v, kv_commit, accept_len, cache_k, cache_v, layout: int,
                   block_table, seq_pos, cache_kind: int = SPEC_CACHE_SAME, k_scale=None,
                   v_scale=None, commit_status=None, stream=None):
    """Copy the K/V of the root and the accepted nodes ([B, N, H, D]) into a paged cache
    (NHD [blocks, block_size, H, D] or HND [blocks, H, block_size, D]); fp8 caches are uint8.
    Scales: float32 tensors of one element, or [B, N] (one per source token)."""
    B, N, H, D = src_k.shape
    _same_device((src_k, src_v, kv_commit, accept_len, cache_k, cache_v, block_table, seq_pos,
                  k_scale, v_scale, commit_status), _hdev(h), "spec_kv_commit")
    if layout == SPEC_KV_NHD:
        num_blocks, block_size = cache_k.shape[0], cache_k.shape[1]
    else:
        num_blocks, block_size = cache_k.shape[0], cache_k.shape[2]
    scale_mode = SPEC_SCALE_TENSOR
    given = [sc for sc in (k_scale, v_scale) if sc is not None]
    if any(sc.dtype != torch.float32 for sc in given):
        raise TypeError("scales must be float32")
    if any(sc.numel() != 1 for sc in given):
        if not all(tuple(sc.shape) == (B, N) for sc in given):
            raise ValueError("scales must all be single values or all [B, N]")
        scale_mode = SPEC_SCALE_PER_TOKEN
    _check(load().spec_kv_commit(
        h.ptr, _ptr(src_k), _ptr(src_v), _kv_dtype(src_k), B, N, H, D,
        _ptr(_i32(kv_commit, "kv_commit")), _ptr(_i32(accept_len, "accept_len")), _ptr(cache_k),
        _ptr(cache_v), int(cache_kind), int(layout), int(block_size), int(num_blocks),
        _ptr(_i32(block_table, "block_table")), int(block_table.shape[1]),
        _ptr(_i32(seq_pos, "seq_pos")), _ptr(k_scale), _ptr(v_scale), scale_mode,
        _ptr(commit_status),
        _stream(stream, src_k.device)), "spec_kv_commit")


def spec_set_node_budget(h: Handle, n_active):
    """Later verify calls on ``h`` verify request b as its first n_active[b] nodes (device
    int32 [>= B], read when the kernels run); None verifies every node."""
    if n_active is not None:
        _i32(n_active, "n_active")
    _check(load().spec_set_node_budget(h.ptr, _ptr(n_active)), "spec_set_node_budget")
    h.n_active = n_active   # keep the array alive while the handle reads it


def spec_budget_update(h: Handle, params: BudgetParams, accept_len, status, parent, state,
                       n_active, stream=None):
    """One controller update on the device; ``state`` is a tensor from budget_state()."""
    B, N = parent.shape
    _same_device((accept_len, status, parent, state, n_active), _hdev(h), "spec_budget_update")
    if state.dtype != torch.float64 or state.numel() != 2:
        raise TypeError("state must be the float64 [2] tensor made by budget_state()")
    _check(load().spec_budget_update(
        h.ptr, ctypes.byref(params), _ptr(_i32(accept_len, "accept_len")),
        _ptr(_i32(status, "status")), _ptr(_i32(parent, "parent")), B, N, _ptr(state),
        _ptr(_i32(n_active, "n_active")), _stream(stream, parent.device)), "spec_budget_update")


def budget_state(ema: float, budget: int, device, steps: int = 0) -> torch.Tensor:
    """A device spec_budget_state {double ema; int32 budget; int32 steps} in a float64 [2]."""
    t = torch.zeros(2, dtype=torch.float64)
    t[0] = float(ema)
    t[1:].view(torch.int32)[0] = int(budget)
    t[1:].view(torch.int32)[1] = int(steps)
    return t.to(device)


def read_budget_state(state: torch.Tensor):
    """-> (ema, budget, steps) of a state tensor (synchronises with the device)."""
    t = state.cpu()
    iv = t[1:].view(torch.int32)
    return float(t[0]), int(iv[0]), int(iv[1])


def spec_profile_begin(h: Handle):
    _check(load().spec_profile_begin(h.ptr), "spec_profile_begin")


def spec_profile_end(h: Handle):
    """-> {kernel class: (total ms, launches)} for the launches since spec_profile_begin."""
    ms = (ctypes.c_float * len(KERNEL_CLASSES))()
    n = (ctypes.c_int32 * len(KERNEL_CLASSES))()
    _check(load().spec_profile_end(h.ptr, ms, n), "spec_profile_end")
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KERNEL_CLASSES)}


# ---- convenience: allocate outputs -----------------------------------------------------------

def alloc_outputs(B: int, N: int, device) -> dict:
    opts = dict(dtype=torch.int32, device=device)
    return dict(accept_len=torch.empty(B, **opts), out_tokens=torch.empty((B, N), **opts),
                kv_commit=torch.empty((B, N), **opts), bonus=torch.empty(B, **opts),
                status=torch.empty(B, **opts))


def verify_greedy(h: Handle, logits, draft_token, parent, out: dict | None = None,
                  stream=None) -> dict:
    B, N, _ = logits.shape
    out = out or alloc_outputs(B, N, logits.device)
    spec_verify_greedy(h, logits, draft_token, parent, out["accept_len"], out["out_tokens"],
                       out["kv_commit"], out["bonus"], out["status"], stream)
    return out


def verify_sample(h: Handle, logits, draft_token, parent, temperature, uniforms, draft=None,
                  draft_kind=SPEC_DRAFT_POINT, out: dict | None = None, stream=None) -> dict:
    B, N, _ = logits.shape
    out = out or alloc_outputs(B, N, logits.device)
    spec_verify_sample(h, logits, draft_token, parent, temperature, uniforms, out["accept_len"],
                       out["out_tokens"], out["kv_commit"], out["bonus"], out["status"], draft,
                       draft_kind, stream)
    return out


def verify_greedy_lazy(h: Handle, logits, draft_token, parent, out: dict | None = None,
                       stream=None) -> dict:
    B, N, _ = logits.shape
    out = out or alloc_outputs(B, N, draft_token.device)
    spec_verify_greedy_lazy(h, logits, draft_token, parent, out["accept_len"], out["out_tokens"],
                            out["kv_commit"], out["bonus"], out["status"], stream)
    return out


def verify_sample_lazy(h: Handle, logits, draft_token, parent, temperature, uniforms, draft=None,
                       draft_kind=SPEC_DRAFT_POINT, out: dict | None = None, stream=None) -> dict:
    B, N, _ = logits.shape
    out = out or alloc_outputs(B, N, draft_token.device)
    spec_verify_sample_lazy(h, logits, draft_token, parent, temperature, uniforms,
                            out["accept_len"], out["out_tokens"], out["kv_commit"], out["bonus"],
                            out["status"], draft, draft_kind, stream)
    return out


def build_tree_mask(h: Handle, parent, stream=None) -> dict:
    B, N = parent.shape
    dev = parent.device
    out = dict(anc_mask=torch.empty((B, N), dtype=torch.int64, device=dev),
               depth=torch.empty((B, N), dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    spec_build_tree_mask(h, parent, out["anc_mask"], out["depth"], out["status"], stream)
    return out


# ---- greedy verification without device allocation --------------------------------------------

SPEC_NOALLOC_MAX_ROWS = 16384


def spec_verify_greedy_noalloc(logits, draft_token, parent, accept_len, out_tokens, kv_commit,
                               bonus, status, stream=None):
    """Greedy verification whose scratch is a static device array (no cudaMalloc anywhere),
    for callers that must not allocate device memory. Runs on the tensors' device, which must
    be the current device; B*N <= SPEC_NOALLOC_MAX_ROWS. Calls share the scratch, so calls
    that overlap on the GPU race."""
    lib = load()
    fn = lib.spec_verify_greedy_noalloc
    if fn.argtypes is None:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        fn.argtypes = [P, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
    B, N, V = logits.shape
    tensors = (logits, draft_token, parent, accept_len, out_tokens, kv_commit, bonus, status)
    _same_device(tensors, logits.device, "spec_verify_greedy_noalloc")
    # the library runs on the current device: make it the tensors' device for the call
    with torch.cuda.device(logits.device):
        _check(fn(_ptr(logits), _dtype_code(logits), B, N, V,
                  _ptr(_i32(draft_token, "draft_token")), _ptr(_i32(parent, "parent")),
                  _ptr(accept_len), _ptr(out_tokens), _ptr(kv_commit), _ptr(bonus),
                  _ptr(status), _stream(stream, logits.device)),
               "spec_verify_greedy_noalloc")


# ---- debug flavour -------------------------------------------------------------------------

def spec_debug_build() -> bool:
    """True when the loaded library is the checked (SPEC_DEBUG) build."""
    return bool(load().spec_debug_build())


def spec_debug_inject_arrival(h: Handle, row: int, value: int):
    """Debug builds: the next split row-statistics launch on ``h`` finds ``value`` in the
    arrival counter of ``row`` (a test of the counter check)."""
    _check(load().spec_debug_inject_arrival(h.ptr, int(row), int(value)),
           "spec_debug_inject_arrival")


def spec_debug_words(h: Handle, B: int, stream=None) -> torch.Tensor:
    """Debug builds: the violation bits (DBG_*) of requests 0..B-1 in the handle's last call."""
    words = torch.empty(B, dtype=torch.int32, device=_hdev(h))
    _check(load().spec_debug_words(h.ptr, _ptr(words), int(B), _stream(stream, words.device)),
           "spec_debug_words")
    return words
