"""Python binding of libcpa.so, the cascade paged-attention library for sm_103a.

Argument marshalling only: every function here checks tensor dtypes, shapes
and devices, allocates outputs / workspace with PyTorch when the caller does
not pass them, and calls the C entry point of the same name on PyTorch's
current CUDA stream.  All arithmetic runs in the library's CUDA kernels; there
is no fallback path, and a missing library raises ``RuntimeError``.

Every call that takes a workspace (and the static-scratch call) accepts
``check=True``: after the launch it reads the device status word
(synchronising the stream) and raises ``CpaError`` when the GPU recorded a bad
page id, a bad prefix length, a bad tree parent or a pipeline timeout.  The
outputs of such a call are undefined.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

__all__ = [
    "CpaError",
    "lib",
    "build_library",
    "cpa_status_string",
    "cpa_version",
    "cpa_cascade_verify_workspace_size",
    "cpa_prefill_hit_workspace_size",
    "cpa_status_workspace_size",
    "cpa_cascade_verify",
    "cpa_cascade_verify_noalloc",
    "cpa_cascade_verify_fp8",
    "cpa_cascade_pass_a_fp8",
    "cpa_naive_expand_verify",
    "cpa_cascade_pass_a",
    "cpa_cascade_pass_b",
    "cpa_merge_state",
    "cpa_prefill_hit",
    "cpa_cascade_verify_shared_workspace_size",
    "cpa_cascade_verify_shared",
    "cpa_tree_verify_workspace_size",
    "cpa_tree_verify",
    "cpa_tree_pass_b",
    "cpa_get_device_status",
    "cpa_noalloc_device_status",
    "cpa_debug_wait_timeout",
    "cpa_plan_partition",
    "declared_functions",
    "PREFILL_FULL",
    "PREFILL_RECT",
    "PREFILL_TRI",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "cpa.h")

PREFILL_FULL, PREFILL_RECT, PREFILL_TRI = 0, 1, 2
_STATUS = {0: "CPA_OK", 1: "CPA_ERR_INVALID_ARG", 2: "CPA_ERR_UNSUPPORTED",
           3: "CPA_ERR_WORKSPACE", 4: "CPA_ERR_LAUNCH", 5: "CPA_ERR_BAD_PAGE",
           6: "CPA_ERR_TIMEOUT", 7: "CPA_ERR_CUDA", 8: "CPA_ERR_BAD_LENGTH",
           9: "CPA_ERR_BAD_TREE"}


class CpaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}: "
                         f"{cpa_status_string(status)}")


_lib: Optional[ctypes.CDLL] = None


def build_library(force: bool = False) -> str:
    """Compile libcpa.so in-tree (nvcc, sm_103a)."""
    import importlib
    return importlib.import_module(__name__ + ".build").build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library: libcpa.so, or the build that $CPA_LIBRARY names (the
    diagnostic trace build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("CPA_LIBRARY") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m cascade_paged_attention_gb300.build`")
    L = ctypes.CDLL(path)
    P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                        ctypes.c_size_t)
    verify_args = [P, P, P, P, I, P, I, P, I, I, I, I, I, I, I, I, I, F, P, P, P, SZ, P]
    sig = {
        "cpa_status_string": (ctypes.c_char_p, [I]),
        "cpa_version": (I, []),
        "cpa_status_workspace_size": (SZ, []),
        "cpa_cascade_verify_workspace_size": (SZ, [I, I, I, I, I, I, I]),
        "cpa_prefill_hit_workspace_size": (SZ, [I, I, I, I, I, I, I]),
        "cpa_cascade_verify": (I, verify_args),
        "cpa_naive_expand_verify": (I, verify_args),
        "cpa_cascade_verify_noalloc": (I, verify_args[:20] + [P]),
        "cpa_cascade_verify_fp8": (I, verify_args[:3] + [P, P, I] + verify_args[3:]),
        "cpa_cascade_pass_a_fp8": (I, [P, P, P, P, P, I, P, I, P, I, I, I, I, I, I, I, I, I, F, P,
                                       P, P, SZ, P]),
        "cpa_cascade_pass_a": (I, [P, P, P, P, I, P, I, I, I, I, I, I, I, I, I, F, P, P, P, SZ,
                                   P]),
        "cpa_cascade_pass_b": (I, [P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P, P, SZ, P]),
        "cpa_merge_state": (I, [P, P, P, P, I, I, I, P, P, P]),
        "cpa_prefill_hit": (I, [P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P, P, P, SZ, P]),
        "cpa_cascade_verify_shared_workspace_size": (SZ, [I, I, I, I, I, I, I, I]),
        "cpa_cascade_verify_shared": (I, [P, P, P, P, I, I, I, P, I, P, I, P, I, I, I, I, I, I,
                                          I, I, I, F, P, P, P, SZ, P]),
        "cpa_tree_verify_workspace_size": (SZ, [I, I, I, I, I, I]),
        "cpa_tree_verify": (I, [P, P, P, P, I, P, I, P, P, I, I, I, I, I, I, I, I, F, P, P, P, SZ,
                                P]),
        "cpa_tree_pass_b": (I, [P, P, P, P, I, P, I, I, I, I, I, I, I, F, P, P, P, SZ, P]),
        "cpa_get_device_status": (I, [P, ctypes.POINTER(ctypes.c_uint32), P]),
        "cpa_noalloc_device_status": (I, [ctypes.POINTER(ctypes.c_uint32), P]),
        "cpa_debug_wait_timeout": (I, [P, SZ, I, P]),
        "cpa_plan_partition": (I, [I64, I, I, I64, ctypes.POINTER(ctypes.c_int64),
                                   ctypes.POINTER(ctypes.c_int64)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def declared_functions() -> list[str]:
    """Names of the functions include/cpa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpa_[a-z0-9_]+)\s*\(", text)))


def cpa_status_string(status: int) -> str:
    return lib().cpa_status_string(int(status)).decode()


def cpa_version() -> int:
    return lib().cpa_version()


def cpa_status_workspace_size() -> int:
    return lib().cpa_status_workspace_size()


def cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, head_dim, page_size) -> int:
    return lib().cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, head_dim, page_size)


def cpa_prefill_hit_workspace_size(B, N, H_hit, H_q, H_kv, head_dim, page_size) -> int:
    return lib().cpa_prefill_hit_workspace_size(B, N, H_hit, H_q, H_kv, head_dim, page_size)


# ---------------------------------------------------------------- marshalling helpers
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")


_ws_cache: dict = {}


def _workspace(nbytes: int, device: torch.device, workspace: Optional[torch.Tensor]):
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8)
        return workspace
    key = (device.index, nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache.clear()
        _ws_cache[key] = ws
    return ws


def _check(fn: str, status: int):
    if status != 0:
        raise CpaError(fn, status)


def _check_device(fn: str, workspace: torch.Tensor, stream):
    """Raise if the device status word of `workspace` has any bit set (synchronises)."""
    st, word = cpa_get_device_status(workspace, stream)
    if st != 0:
        raise CpaError(f"{fn} (device status word {word:#x})", st)


def _verify_shapes(q, k_pages, v_pages, prefix_page_table, prefix_lens, topk, S):
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(prefix_page_table, "prefix_page_table", torch.int32, 2)
    _need(prefix_lens, "prefix_lens", torch.int32, 1)
    if k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape")
    num_pages, page_size, H_kv, d = k_pages.shape
    B = prefix_lens.numel()
    T, H_q, dq = q.shape
    if dq != d or T != B * topk * S or prefix_page_table.shape[0] != B:
        raise ValueError("inconsistent verify shapes")
    return B, H_q, H_kv, d, page_size, num_pages


def _verify_call(name, q, k_pages, v_pages, prefix_page_table, draft_page_table, prefix_lens,
                 topk, S, max_prefix_len, sm_scale, o, lse, workspace, stream, check=False):
    B, H_q, H_kv, d, P, num_pages = _verify_shapes(q, k_pages, v_pages, prefix_page_table,
                                                    prefix_lens, topk, S)
    _need(draft_page_table, "draft_page_table", torch.int32, 2)
    if draft_page_table.shape[0] != B * topk:
        raise ValueError("draft_page_table must have B*topk rows")
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o, "o", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    nbytes = cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, d, P)
    ws = _workspace(nbytes, q.device, workspace)
    st = getattr(lib(), name)(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(prefix_page_table),
        prefix_page_table.shape[1], _ptr(draft_page_table), draft_page_table.shape[1],
        _ptr(prefix_lens), B, topk, S, H_q, H_kv, d, P, num_pages, int(max_prefix_len),
        float(sm_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(name, st)
    if check:
        _check_device(name, ws, stream)
    return o, lse


# ---------------------------------------------------------------- entry points
def cpa_cascade_verify(q, k_pages, v_pages, prefix_page_table, draft_page_table, prefix_lens,
                       topk: int, S: int, max_prefix_len: Optional[int] = None,
                       sm_scale: Optional[float] = None, o=None, lse=None, workspace=None,
                       stream=None, check: bool = False):
    """Cascade verify attention (Pass A + Pass B + merge).  Returns (o bf16, lse fp32)."""
    return _verify_call("cpa_cascade_verify", q, k_pages, v_pages, prefix_page_table,
                        draft_page_table, prefix_lens, topk, S, max_prefix_len, sm_scale, o, lse,
                        workspace, stream, check)


def cpa_cascade_verify_noalloc(q, k_pages, v_pages, prefix_page_table, draft_page_table,
                               prefix_lens, topk: int, S: int, o, lse,
                               max_prefix_len: Optional[int] = None,
                               sm_scale: Optional[float] = None, stream=None,
                               check: bool = False):
    """Cascade verify without a workspace, for callers that cannot allocate device memory.

    The library keeps its scratch in a fixed-size array it owns on every GPU,
    and this path allocates nothing: the caller passes preallocated `o`
    (bf16, shaped like q) and `lse` (fp32 [T, H_q]).  Returns (o, lse).
    """
    B, H_q, H_kv, d, P, num_pages = _verify_shapes(q, k_pages, v_pages, prefix_page_table,
                                                    prefix_lens, topk, S)
    _need(draft_page_table, "draft_page_table", torch.int32, 2)
    _need(o, "o", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    if draft_page_table.shape[0] != B * topk or o.shape != q.shape or \
            lse.shape != (q.shape[0], H_q):
        raise ValueError("inconsistent verify shapes")
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    st = lib().cpa_cascade_verify_noalloc(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(prefix_page_table),
        prefix_page_table.shape[1], _ptr(draft_page_table), draft_page_table.shape[1],
        _ptr(prefix_lens), B, topk, S, H_q, H_kv, d, P, num_pages, int(max_prefix_len),
        float(sm_scale), _ptr(o), _ptr(lse), _stream(stream))
    _check("cpa_cascade_verify_noalloc", st)
    if check:
        st, word = cpa_noalloc_device_status(stream)
        if st != 0:
            raise CpaError(f"cpa_cascade_verify_noalloc (device status word {word:#x})", st)
    return o, lse


def _fp8_pools(q, k_pages, v_pages, k_scale, v_scale, prefix_page_table, prefix_lens, topk, S):
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.uint8, 4)
    _need(v_pages, "v_pages", torch.uint8, 4)
    _need(k_scale, "k_scale", torch.float32)
    _need(v_scale, "v_scale", torch.float32)
    _need(prefix_page_table, "prefix_page_table", torch.int32, 2)
    _need(prefix_lens, "prefix_lens", torch.int32, 1)
    if k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape")
    num_pages, P, H_kv, d = k_pages.shape
    B = prefix_lens.numel()
    T, H_q, dq = q.shape
    if dq != d or T != B * topk * S or prefix_page_table.shape[0] != B:
        raise ValueError("inconsistent verify shapes")
    n = k_scale.numel()
    if v_scale.numel() != n or n not in (1, H_kv * d):
        raise ValueError("k_scale / v_scale must hold 1 or H_kv * head_dim values each")
    return B, H_q, H_kv, d, P, num_pages, int(n > 1)


def cpa_cascade_verify_fp8(q, k_pages, v_pages, k_scale, v_scale, prefix_page_table,
                           draft_page_table, prefix_lens, topk: int, S: int,
                           max_prefix_len: Optional[int] = None, sm_scale: Optional[float] = None,
                           o=None, lse=None, workspace=None, stream=None, check: bool = False):
    """Cascade verify over FP8 E4M3 KV pages.  Returns (o bf16, lse fp32).

    ``k_pages`` / ``v_pages`` are uint8 E4M3 codes; ``k_scale`` / ``v_scale``
    fp32 with one value each (per tensor) or ``[H_kv, head_dim]`` (per channel).
    """
    B, H_q, H_kv, d, P, num_pages, per_ch = _fp8_pools(q, k_pages, v_pages, k_scale, v_scale,
                                                       prefix_page_table, prefix_lens, topk, S)
    _need(draft_page_table, "draft_page_table", torch.int32, 2)
    if draft_page_table.shape[0] != B * topk:
        raise ValueError("draft_page_table must have B*topk rows")
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o, "o", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    ws = _workspace(cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, d, P), q.device,
                    workspace)
    st = lib().cpa_cascade_verify_fp8(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale), _ptr(v_scale), per_ch,
        _ptr(prefix_page_table), prefix_page_table.shape[1], _ptr(draft_page_table),
        draft_page_table.shape[1], _ptr(prefix_lens), B, topk, S, H_q, H_kv, d, P, num_pages,
        int(max_prefix_len), float(sm_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("cpa_cascade_verify_fp8", st)
    if check:
        _check_device("cpa_cascade_verify_fp8", ws, stream)
    return o, lse


def cpa_cascade_pass_a_fp8(q, k_pages, v_pages, k_scale, v_scale, prefix_page_table,
                           prefix_lens, topk: int, S: int, max_prefix_len: Optional[int] = None,
                           sm_scale: Optional[float] = None, o_a=None, lse_a=None,
                           workspace=None, stream=None, check: bool = False):
    """Pass A alone over FP8 E4M3 KV pages.  Returns (o_a fp32, lse_a fp32)."""
    B, H_q, H_kv, d, P, num_pages, per_ch = _fp8_pools(q, k_pages, v_pages, k_scale, v_scale,
                                                       prefix_page_table, prefix_lens, topk, S)
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o_a is None:
        o_a = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse_a is None:
        lse_a = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o_a, "o_a", torch.float32)
    _need(lse_a, "lse_a", torch.float32)
    ws = _workspace(cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, d, P), q.device,
                    workspace)
    st = lib().cpa_cascade_pass_a_fp8(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale), _ptr(v_scale), per_ch,
        _ptr(prefix_page_table), prefix_page_table.shape[1], _ptr(prefix_lens), B, topk, S, H_q,
        H_kv, d, P, num_pages, int(max_prefix_len), float(sm_scale), _ptr(o_a), _ptr(lse_a),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("cpa_cascade_pass_a_fp8", st)
    if check:
        _check_device("cpa_cascade_pass_a_fp8", ws, stream)
    return o_a, lse_a


def cpa_naive_expand_verify(q, k_pages, v_pages, prefix_page_table, draft_page_table,
                            prefix_lens, topk: int, S: int, max_prefix_len: Optional[int] = None,
                            sm_scale: Optional[float] = None, o=None, lse=None, workspace=None,
                            stream=None, check: bool = False):
    """Naive-expand verify (the baseline).  Returns (o bf16, lse fp32)."""
    return _verify_call("cpa_naive_expand_verify", q, k_pages, v_pages, prefix_page_table,
                        draft_page_table, prefix_lens, topk, S, max_prefix_len, sm_scale, o, lse,
                        workspace, stream, check)


def cpa_cascade_pass_a(q, k_pages, v_pages, prefix_page_table, prefix_lens, topk: int, S: int,
                       max_prefix_len: Optional[int] = None, sm_scale: Optional[float] = None,
                       o_a=None, lse_a=None, workspace=None, stream=None, check: bool = False):
    """Pass A alone.  Returns (o_a fp32, lse_a fp32)."""
    B, H_q, H_kv, d, P, num_pages = _verify_shapes(q, k_pages, v_pages, prefix_page_table,
                                                    prefix_lens, topk, S)
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o_a is None:
        o_a = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse_a is None:
        lse_a = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o_a, "o_a", torch.float32)
    _need(lse_a, "lse_a", torch.float32)
    nbytes = cpa_cascade_verify_workspace_size(B, topk, S, H_q, H_kv, d, P)
    ws = _workspace(nbytes, q.device, workspace)
    st = lib().cpa_cascade_pass_a(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(prefix_page_table),
        prefix_page_table.shape[1], _ptr(prefix_lens), B, topk, S, H_q, H_kv, d, P, num_pages,
        int(max_prefix_len), float(sm_scale), _ptr(o_a), _ptr(lse_a), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("cpa_cascade_pass_a", st)
    if check:
        _check_device("cpa_cascade_pass_a", ws, stream)
    return o_a, lse_a


def cpa_cascade_pass_b(q, k_pages, v_pages, draft_page_table, B: int, topk: int, S: int,
                       sm_scale: Optional[float] = None, o_b=None, lse_b=None, workspace=None,
                       stream=None, check: bool = False):
    """Pass B alone (warp-level draft kernel).  Returns (o_b fp32, lse_b fp32)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(draft_page_table, "draft_page_table", torch.int32, 2)
    num_pages, P, H_kv, d = k_pages.shape
    T, H_q, _ = q.shape
    if T != B * topk * S or draft_page_table.shape[0] != B * topk:
        raise ValueError("inconsistent Pass B shapes")
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o_b is None:
        o_b = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse_b is None:
        lse_b = torch.empty(T, H_q, dtype=torch.float32, device=q.device)
    ws = _workspace(cpa_status_workspace_size(), q.device, workspace)
    st = lib().cpa_cascade_pass_b(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(draft_page_table), draft_page_table.shape[1],
        B, topk, S, H_q, H_kv, d, P, num_pages, float(sm_scale), _ptr(o_b), _ptr(lse_b),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("cpa_cascade_pass_b", st)
    if check:
        _check_device("cpa_cascade_pass_b", ws, stream)
    return o_b, lse_b


def cpa_merge_state(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """merge_state of two fp32 partial attentions -> (o bf16, lse fp32)."""
    for t, n in ((o_a, "o_a"), (o_b, "o_b")):
        _need(t, n, torch.float32, 3)
    for t, n in ((lse_a, "lse_a"), (lse_b, "lse_b")):
        _need(t, n, torch.float32, 2)
    n_tokens, H, d = o_a.shape
    if o_b.shape != o_a.shape or lse_a.shape != (n_tokens, H) or lse_b.shape != (n_tokens, H):
        raise ValueError("inconsistent merge_state shapes")
    if o_out is None:
        o_out = torch.empty(o_a.shape, dtype=torch.bfloat16, device=o_a.device)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    st = lib().cpa_merge_state(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), n_tokens, H, d,
                               _ptr(o_out), _ptr(lse_out), _stream(stream))
    _check("cpa_merge_state", st)
    return o_out, lse_out


def cpa_prefill_hit(q, k_pages, v_pages, page_table, B: int, N: int, H_hit: int,
                    part: int = PREFILL_FULL, sm_scale: Optional[float] = None, o=None, lse=None,
                    workspace=None, stream=None, check: bool = False):
    """Prefix-hit prefill.  Returns (o, lse); o is bf16 for PREFILL_FULL, fp32 otherwise."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    num_pages, P, H_kv, d = k_pages.shape
    T, H_q, _ = q.shape
    if T != B * (N - H_hit) or page_table.shape[0] != B:
        raise ValueError("inconsistent prefill shapes")
    if sm_scale is None:
        sm_scale = d ** -0.5
    odt = torch.bfloat16 if part == PREFILL_FULL else torch.float32
    if o is None:
        o = torch.empty(q.shape, dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty(T, H_q, dtype=torch.float32, device=q.device)
    _need(o, "o", odt)
    nbytes = cpa_prefill_hit_workspace_size(B, N, H_hit, H_q, H_kv, d, P)
    ws = _workspace(nbytes, q.device, workspace)
    st = lib().cpa_prefill_hit(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), page_table.shape[1], B, N,
        H_hit, H_q, H_kv, d, P, num_pages, float(sm_scale), int(part), _ptr(o), _ptr(lse),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("cpa_prefill_hit", st)
    if check:
        _check_device("cpa_prefill_hit", ws, stream)
    return o, lse


def cpa_cascade_verify_shared_workspace_size(B, n_groups, topk, S, H_q, H_kv, head_dim,
                                            page_size) -> int:
    return lib().cpa_cascade_verify_shared_workspace_size(B, n_groups, topk, S, H_q, H_kv,
                                                          head_dim, page_size)


def cpa_cascade_verify_shared(q, k_pages, v_pages, shared_page_table, shared_len: int,
                              prefix_page_table, draft_page_table, prefix_lens, topk: int, S: int,
                              max_prefix_len: Optional[int] = None,
                              sm_scale: Optional[float] = None, o=None, lse=None, workspace=None,
                              stream=None, check: bool = False):
    """Multi-level cascade verify.  Returns (o bf16, lse fp32).

    ``shared_page_table`` int32 [n_groups, stride]: one shared prefix of
    ``shared_len`` tokens per group of ``B // n_groups`` consecutive requests;
    ``prefix_page_table`` / ``prefix_lens`` describe each request's own prefix.
    """
    B, H_q, H_kv, d, P, num_pages = _verify_shapes(q, k_pages, v_pages, prefix_page_table,
                                                    prefix_lens, topk, S)
    _need(shared_page_table, "shared_page_table", torch.int32, 2)
    _need(draft_page_table, "draft_page_table", torch.int32, 2)
    n_groups = shared_page_table.shape[0]
    if draft_page_table.shape[0] != B * topk or n_groups < 1 or B % n_groups:
        raise ValueError("inconsistent multi-level verify shapes")
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o, "o", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    nbytes = cpa_cascade_verify_shared_workspace_size(B, n_groups, topk, S, H_q, H_kv, d, P)
    ws = _workspace(nbytes, q.device, workspace)
    st = lib().cpa_cascade_verify_shared(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(shared_page_table),
        shared_page_table.shape[1], n_groups, int(shared_len), _ptr(prefix_page_table),
        prefix_page_table.shape[1], _ptr(draft_page_table), draft_page_table.shape[1],
        _ptr(prefix_lens), B, topk, S, H_q, H_kv, d, P, num_pages, int(max_prefix_len),
        float(sm_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check("cpa_cascade_verify_shared", st)
    if check:
        _check_device("cpa_cascade_verify_shared", ws, stream)
    return o, lse


def cpa_tree_verify_workspace_size(B, N, H_q, H_kv, head_dim, page_size) -> int:
    return lib().cpa_tree_verify_workspace_size(B, N, H_q, H_kv, head_dim, page_size)


def _tree_shapes(q, k_pages, v_pages, tree_page_table, tree_parents):
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(tree_page_table, "tree_page_table", torch.int32, 2)
    _need(tree_parents, "tree_parents", torch.int32, 2)
    if k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape")
    num_pages, P, H_kv, d = k_pages.shape
    B, N = tree_parents.shape
    T, H_q, dq = q.shape
    if dq != d or T != B * N or tree_page_table.shape[0] != B:
        raise ValueError("inconsistent tree verify shapes")
    return B, N, H_q, H_kv, d, P, num_pages


def cpa_tree_verify(q, k_pages, v_pages, prefix_page_table, tree_page_table, prefix_lens,
                    tree_parents, max_prefix_len: Optional[int] = None,
                    sm_scale: Optional[float] = None, o=None, lse=None, workspace=None,
                    stream=None, check: bool = False):
    """Verify over draft trees (prefix pass + tree pass + merge).  Returns (o bf16, lse fp32).

    ``tree_parents`` int32 [B, N]: parent BFS index of each node, -1 for a root.
    """
    B, N, H_q, H_kv, d, P, num_pages = _tree_shapes(q, k_pages, v_pages, tree_page_table,
                                                     tree_parents)
    _need(prefix_page_table, "prefix_page_table", torch.int32, 2)
    _need(prefix_lens, "prefix_lens", torch.int32, 1)
    if prefix_lens.numel() != B or prefix_page_table.shape[0] != B:
        raise ValueError("inconsistent tree verify shapes")
    if max_prefix_len is None:
        max_prefix_len = prefix_page_table.shape[1] * P
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o, "o", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    nbytes = cpa_tree_verify_workspace_size(B, N, H_q, H_kv, d, P)
    ws = _workspace(nbytes, q.device, workspace)
    st = lib().cpa_tree_verify(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(prefix_page_table),
        prefix_page_table.shape[1], _ptr(tree_page_table), tree_page_table.shape[1],
        _ptr(prefix_lens), _ptr(tree_parents), B, N, H_q, H_kv, d, P, num_pages,
        int(max_prefix_len), float(sm_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("cpa_tree_verify", st)
    if check:
        _check_device("cpa_tree_verify", ws, stream)
    return o, lse


def cpa_tree_pass_b(q, k_pages, v_pages, tree_page_table, tree_parents,
                    sm_scale: Optional[float] = None, o_b=None, lse_b=None, workspace=None,
                    stream=None, check: bool = False):
    """The tree part alone (each node against its ancestor-or-self nodes).  Returns fp32 (o_b, lse_b)."""
    B, N, H_q, H_kv, d, P, num_pages = _tree_shapes(q, k_pages, v_pages, tree_page_table,
                                                     tree_parents)
    if sm_scale is None:
        sm_scale = d ** -0.5
    if o_b is None:
        o_b = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if lse_b is None:
        lse_b = torch.empty(q.shape[0], H_q, dtype=torch.float32, device=q.device)
    _need(o_b, "o_b", torch.float32)
    _need(lse_b, "lse_b", torch.float32)
    ws = _workspace(cpa_status_workspace_size(), q.device, workspace)
    st = lib().cpa_tree_pass_b(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(tree_page_table), tree_page_table.shape[1],
        _ptr(tree_parents), B, N, H_q, H_kv, d, P, num_pages, float(sm_scale), _ptr(o_b),
        _ptr(lse_b), _ptr(ws), ws.numel(), _stream(stream))
    _check("cpa_tree_pass_b", st)
    if check:
        _check_device("cpa_tree_pass_b", ws, stream)
    return o_b, lse_b


def cpa_get_device_status(workspace: torch.Tensor, stream=None) -> tuple[int, int]:
    """(status code, raw device status word) of the last call on `workspace` (synchronises)."""
    word = ctypes.c_uint32(0)
    st = lib().cpa_get_device_status(_ptr(workspace), ctypes.byref(word), _stream(stream))
    return st, word.value


def cpa_noalloc_device_status(stream=None) -> tuple[int, int]:
    """(status code, raw word) of the static scratch of the current device (synchronises)."""
    word = ctypes.c_uint32(0)
    st = lib().cpa_noalloc_device_status(ctypes.byref(word), _stream(stream))
    return st, word.value


def cpa_debug_wait_timeout(workspace: torch.Tensor, limit_us: int, stream=None) -> None:
    st = lib().cpa_debug_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_us),
                                      _stream(stream))
    _check("cpa_debug_wait_timeout", st)


def cpa_plan_partition(total: int, n_ctas: int, cta: int, tile: int):
    """(owner of `tile`, begin, end of `cta`) of the kernels' work partition (host-side)."""
    b = ctypes.c_int64(0)
    e = ctypes.c_int64(0)
    owner = lib().cpa_plan_partition(total, n_ctas, cta, tile, ctypes.byref(b), ctypes.byref(e))
    return owner, b.value, e.value
