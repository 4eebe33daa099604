"""Python binding of libpf.so -- paged-KV decode attention on GB300 (sm_103a).

A thin ctypes layer over the C ABI in include/pf.h: it checks shapes, dtypes
and devices of torch tensors, passes their device pointers and the current
CUDA stream, and raises PFError on a non-OK status.  Every step of the
computation runs in the library's CUDA kernels; there is no Python or CPU
fallback -- if libpf.so is missing, every call raises.

Entry points (same names as the C ABI without the pf_ prefix):
    reshape_and_cache              KV append through slot_mapping (-1 = skip)
    paged_attention_decode         single-pass decode attention, fp32 out
    partition_workspace_layout     sizes/offsets of the split-K workspace
    paged_attention_decode_partition   partition pass (flash-decoding)
    paged_attention_merge          log-sum-exp merge of the partitions
    paged_attention_split          partition + merge with a torch-allocated workspace
    get_device_error / check_device_error / debug_bounded_wait / version
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpf.so")

PF_OK, PF_ERR_INVALID_ARG, PF_ERR_UNSUPPORTED, PF_ERR_CUDA, PF_ERR_DEVICE_BOUNDS, PF_ERR_DEVICE_TIMEOUT = range(6)
STATUS_NAMES = {0: "PF_OK", 1: "PF_ERR_INVALID_ARG", 2: "PF_ERR_UNSUPPORTED", 3: "PF_ERR_CUDA",
                4: "PF_ERR_DEVICE_BOUNDS", 5: "PF_ERR_DEVICE_TIMEOUT"}


class PFError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded libpf.so (built in-tree by paged_kv_decode_pf_gb300._build)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m paged_kv_decode_pf_gb300._build` "
                               "(nvcc, sm_103a); this package has no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        st = ctypes.c_int
        L.pf_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64, P]
        L.pf_reshape_and_cache.restype = st
        L.pf_paged_attention_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, P, P]
        L.pf_paged_attention_decode.restype = st
        L.pf_paged_attention_decode_bf16.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, P, P]
        L.pf_paged_attention_decode_bf16.restype = st
        L.pf_paged_attention_partition_workspace_layout.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(sz),
                                                                    ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.pf_paged_attention_partition_workspace_layout.restype = sz
        L.pf_paged_attention_partition_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.pf_paged_attention_partition_workspace_size.restype = sz
        L.pf_paged_attention_decode_partition.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32,
                                                          i32, i32, P, sz, P]
        L.pf_paged_attention_decode_partition.restype = st
        L.pf_paged_attention_merge.argtypes = [P, P, i32, i32, i32, i32, i32, P, P]
        L.pf_paged_attention_merge.restype = st
        L.pf_get_device_error.argtypes = [P]
        L.pf_get_device_error.restype = st
        L.pf_status_string.argtypes = [st]
        L.pf_status_string.restype = ctypes.c_char_p
        L.pf_debug_bounded_wait.argtypes = [i64, P]
        L.pf_debug_bounded_wait.restype = st
        L.pf_version.argtypes = []
        L.pf_version.restype = ctypes.c_char_p
        L.pf_copy_blocks.argtypes = [P, P, P, i64, i32, i32, i32, i64, P]
        L.pf_copy_blocks.restype = st
        L.pf_paged_attention_decode_append.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                                       f32, P, P]
        L.pf_paged_attention_decode_append.restype = st
        L.pf_paged_attention_decode_auto_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
        L.pf_paged_attention_decode_auto_plan.restype = i32
        L.pf_paged_attention_decode_auto.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, f32, i32, P,
                                                     sz, P, P]
        L.pf_paged_attention_decode_auto.restype = st
        L.pf_paged_attention_multi_query.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, f32, P,
                                                     P]
        L.pf_paged_attention_multi_query.restype = st
        L.pf_paged_attention_multi_query_tcgen05.argtypes = L.pf_paged_attention_multi_query.argtypes
        L.pf_paged_attention_multi_query_tcgen05.restype = st
        _LIB = L
    return _LIB


def version() -> str:
    return lib().pf_version().decode()


def _check(status: int, where: str) -> None:
    if status != PF_OK:
        raise PFError(status, where)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _cuda(t: torch.Tensor, name: str, dtypes, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_BF16 = (torch.bfloat16, torch.int16)   # int16 views carry raw bf16 bits


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor) -> None:
    """Scatter k/v [T, Hkv, D] into the caches [NB, Hkv, bs, D] at slot_mapping [T] (int64, -1 = skip)."""
    _cuda(k, "k", _BF16, 3)
    _cuda(v, "v", _BF16, 3)
    _cuda(slot_mapping, "slot_mapping", (torch.int64,), 1)
    _cuda(k_cache, "k_cache", _BF16, 4)
    _cuda(v_cache, "v_cache", _BF16, 4)
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D) or slot_mapping.shape[0] != T:
        raise ValueError("reshape_and_cache: inconsistent shapes")
    with torch.cuda.device(k.device):
        _check(lib().pf_reshape_and_cache(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
                                          v_cache.data_ptr(), T, Hkv, D, bs, NB, _stream(k.device)),
               "pf_reshape_and_cache")


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_mapping: torch.Tensor) -> None:
    """Copy whole physical blocks: block_mapping [n, 2] int64 of (src, dst) pairs."""
    _cuda(k_cache, "k_cache", _BF16, 4)
    _cuda(v_cache, "v_cache", _BF16, 4)
    _cuda(block_mapping, "block_mapping", (torch.int64,), 2)
    if v_cache.shape != k_cache.shape or block_mapping.shape[1] != 2:
        raise ValueError("copy_blocks: inconsistent shapes")
    NB, Hkv, bs, D = k_cache.shape
    with torch.cuda.device(k_cache.device):
        _check(lib().pf_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), block_mapping.data_ptr(),
                                    block_mapping.shape[0], Hkv, D, bs, NB, _stream(k_cache.device)),
               "pf_copy_blocks")


def _attn_shapes(q, k_cache, v_cache, block_tables, context_lens):
    _cuda(q, "q", _BF16, 3)
    _cuda(k_cache, "k_cache", _BF16, 4)
    _cuda(v_cache, "v_cache", _BF16, 4)
    _cuda(block_tables, "block_tables", (torch.int32,), 2)
    _cuda(context_lens, "context_lens", (torch.int32,), 1)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("paged attention: inconsistent shapes")
    return S, Hq, Hkv, D, bs, NB, block_tables.shape[1]


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: Optional[float] = None,
                           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Single-pass decode attention; returns out [S, Hq, D] fp32."""
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
    _cuda(out, "out", (torch.float32,), 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        _check(lib().pf_paged_attention_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                               block_tables.data_ptr(), context_lens.data_ptr(), S, Hq, Hkv, D, bs,
                                               MB, NB, scale, out.data_ptr(), _stream(q.device)),
               "pf_paged_attention_decode")
    return out


def paged_attention_decode_bf16(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor, scale: Optional[float] = None,
                                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Single-pass decode attention with a bf16 output [S, Hq, D]: the fp32 result rounded once (to
    nearest, ties to even)."""
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=q.device)
    _cuda(out, "out", _BF16, 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        _check(lib().pf_paged_attention_decode_bf16(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                                    block_tables.data_ptr(), context_lens.data_ptr(), S, Hq, Hkv, D,
                                                    bs, MB, NB, scale, out.data_ptr(), _stream(q.device)),
               "pf_paged_attention_decode_bf16")
    return out


def paged_attention_decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                  slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  scale: Optional[float] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step in one launch: write k_new/v_new [S, Hkv, D] of each sequence's newest token to
    slot_mapping [S] (int64; -1 = nothing to append), then attend.  Returns out [S, Hq, D] fp32."""
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    _cuda(k_new, "k_new", _BF16, 3)
    _cuda(v_new, "v_new", _BF16, 3)
    _cuda(slot_mapping, "slot_mapping", (torch.int64,), 1)
    if k_new.shape != (S, Hkv, D) or v_new.shape != k_new.shape or slot_mapping.shape[0] != S:
        raise ValueError("paged_attention_decode_append: inconsistent shapes")
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
    _cuda(out, "out", (torch.float32,), 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        _check(lib().pf_paged_attention_decode_append(
            q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
            v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(), S, Hq, Hkv, D, bs, MB, NB, scale,
            out.data_ptr(), _stream(q.device)), "pf_paged_attention_decode_append")
    return out


def paged_attention_multi_query(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                                kernel: str = "auto") -> torch.Tensor:
    """q [S, q_len, Hq, D]: the last q_len tokens of each sequence, already in the cache, attend causally.
    Returns out [S, q_len, Hq, D] fp32.  Needs (Hq / Hkv) * q_len <= 65536.  kernel="auto" calls
    pf_paged_attention_multi_query (which picks its kernel by row count: past 64 rows per kv head
    the prompt-chunk kernel); kernel="tcgen05" calls pf_paged_attention_multi_query_tcgen05
    (D = 128 only)."""
    if kernel not in ("auto", "tcgen05"):
        raise ValueError(f"paged_attention_multi_query: unknown kernel {kernel!r}")
    _cuda(q, "q", _BF16, 4)
    _cuda(k_cache, "k_cache", _BF16, 4)
    _cuda(v_cache, "v_cache", _BF16, 4)
    _cuda(block_tables, "block_tables", (torch.int32,), 2)
    _cuda(context_lens, "context_lens", (torch.int32,), 1)
    S, Q, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("paged_attention_multi_query: inconsistent shapes")
    MB = block_tables.shape[1]
    if out is None:
        out = torch.empty((S, Q, Hq, D), dtype=torch.float32, device=q.device)
    _cuda(out, "out", (torch.float32,), 4)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        name = "pf_paged_attention_multi_query" + ("_tcgen05" if kernel == "tcgen05" else "")
        _check(getattr(lib(), name)(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                    context_lens.data_ptr(), S, Q, Hq, Hkv, D, bs, MB, NB, scale, out.data_ptr(),
                                    _stream(q.device)), name)
    return out


def decode_auto_plan(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     max_context_len: int, device=None) -> Tuple[int, int]:
    """(partition size the auto decode will use, workspace bytes it needs): (0, 0) for the single
    pass, (chunk per CTA, 0) for the cluster split (few items: one launch, no workspace),
    (partition size, bytes) for the split over context partitions + merge."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws = ctypes.c_size_t()
    with torch.cuda.device(device):
        P = lib().pf_paged_attention_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                      max_context_len, ctypes.byref(ws))
    return int(P), ws.value


def paged_attention_decode_auto(q, k_cache, v_cache, block_tables, context_lens, max_context_len: Optional[int] = None,
                                scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode attention with the decomposition chosen by the library (single pass, cluster split, or
    split + merge).  max_context_len defaults to the table's capacity; a workspace is allocated when the
    plan needs one."""
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    if max_context_len is None:
        max_context_len = MB * bs
    P, need = decode_auto_plan(S, Hq, Hkv, D, max_context_len, q.device)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
    _cuda(out, "out", (torch.float32,), 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    with torch.cuda.device(q.device):
        _check(lib().pf_paged_attention_decode_auto(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
            S, Hq, Hkv, D, bs, MB, NB, scale, max_context_len, ws_ptr, ws_bytes, out.data_ptr(),
            _stream(q.device)), "pf_paged_attention_decode_auto")
    return out


def partition_workspace_layout(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                               partition_size: int) -> Tuple[int, int, int, int]:
    """(total_bytes, tmp_out_offset, tmp_m_offset, tmp_l_offset) of the split-K workspace."""
    o, m, l = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    total = lib().pf_paged_attention_partition_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len,
                                                                partition_size, ctypes.byref(o), ctypes.byref(m),
                                                                ctypes.byref(l))
    return int(total), o.value, m.value, l.value


def num_partitions(max_context_len: int, partition_size: int) -> int:
    return max(1, -(-max_context_len // partition_size))


def alloc_workspace(num_seqs, num_q_heads, head_dim, max_context_len, partition_size, device) -> torch.Tensor:
    total = partition_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len, partition_size)[0]
    if total == 0:
        raise PFError(PF_ERR_INVALID_ARG, "partition_workspace_layout")
    return torch.empty(total, dtype=torch.uint8, device=device)   # the caching allocator aligns to 512 B


def workspace_views(workspace: torch.Tensor, num_seqs, num_q_heads, head_dim, max_context_len, partition_size):
    """(tmp_out [S,Hq,NP,D], tmp_m [S,Hq,NP], tmp_l [S,Hq,NP]) fp32 views of a workspace."""
    total, oo, om, ol = partition_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len, partition_size)
    NP = num_partitions(max_context_len, partition_size)
    n = num_seqs * num_q_heads * NP
    f = lambda off, cnt: workspace[off:off + 4 * cnt].view(torch.float32)
    return (f(oo, n * head_dim).view(num_seqs, num_q_heads, NP, head_dim),
            f(om, n).view(num_seqs, num_q_heads, NP), f(ol, n).view(num_seqs, num_q_heads, NP))


def paged_attention_decode_partition(q, k_cache, v_cache, block_tables, context_lens, partition_size: int,
                                     max_context_len: int, workspace: torch.Tensor,
                                     scale: Optional[float] = None) -> None:
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    _cuda(workspace, "workspace", (torch.uint8,), 1)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        _check(lib().pf_paged_attention_decode_partition(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
            S, Hq, Hkv, D, bs, MB, NB, scale, partition_size, max_context_len, workspace.data_ptr(),
            workspace.numel(), _stream(q.device)), "pf_paged_attention_decode_partition")


def paged_attention_merge(workspace: torch.Tensor, context_lens: torch.Tensor, num_q_heads: int, head_dim: int,
                          partition_size: int, max_context_len: int,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(workspace, "workspace", (torch.uint8,), 1)
    _cuda(context_lens, "context_lens", (torch.int32,), 1)
    S = context_lens.shape[0]
    if out is None:
        out = torch.empty((S, num_q_heads, head_dim), dtype=torch.float32, device=context_lens.device)
    _cuda(out, "out", (torch.float32,), 3)
    with torch.cuda.device(context_lens.device):
        _check(lib().pf_paged_attention_merge(workspace.data_ptr(), context_lens.data_ptr(), S, num_q_heads,
                                              head_dim, partition_size, max_context_len, out.data_ptr(),
                                              _stream(context_lens.device)), "pf_paged_attention_merge")
    return out


def paged_attention_split(q, k_cache, v_cache, block_tables, context_lens, partition_size: int = 512,
                          max_context_len: Optional[int] = None, scale: Optional[float] = None,
                          workspace: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Partition pass + log-sum-exp merge.  max_context_len defaults to the table's capacity
    (max_blocks_per_seq * block_size), which needs no read of device memory."""
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    if max_context_len is None:
        max_context_len = MB * bs
    if workspace is None:
        workspace = alloc_workspace(S, Hq, D, max_context_len, partition_size, q.device)
    paged_attention_decode_partition(q, k_cache, v_cache, block_tables, context_lens, partition_size,
                                     max_context_len, workspace, scale)
    return paged_attention_merge(workspace, context_lens, Hq, D, partition_size, max_context_len, out)


SPLIT_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024   # PF_SPLIT_NOALLOC_SCRATCH_BYTES in pf.h


def _split_noalloc_fn():
    f = lib().pf_paged_attention_split_noalloc
    if f.argtypes is None:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        f.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, ctypes.c_float, i32, i32, P, P]
        f.restype = ctypes.c_int
    return f


def paged_attention_split_noalloc(q, k_cache, v_cache, block_tables, context_lens, partition_size: int,
                                  max_context_len: int, scale: Optional[float] = None,
                                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Split-K decode whose partials live in the library's fixed scratch array instead of a
    caller workspace, for callers that cannot allocate device memory on the decode path.
    Calls that overlap on one device race on that array; `out` is still the caller's."""
    S, Hq, Hkv, D, bs, NB, MB = _attn_shapes(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
    _cuda(out, "out", (torch.float32,), 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        _check(_split_noalloc_fn()(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                   context_lens.data_ptr(), S, Hq, Hkv, D, bs, MB, NB, scale, partition_size,
                                   max_context_len, out.data_ptr(), _stream(q.device)),
               "pf_paged_attention_split_noalloc")
    return out


def get_device_error(device=None) -> int:
    """Synchronise the current stream, read and clear the device error word; returns the status code."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return int(lib().pf_get_device_error(_stream(device)))


def check_device_error(device=None) -> None:
    _check(get_device_error(device), "device error word")


def debug_bounded_wait(limit_ns: int, device=None) -> None:
    """Launch the failure-detection check: a wait nothing completes, bounded by limit_ns."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        _check(lib().pf_debug_bounded_wait(int(limit_ns), _stream(device)), "pf_debug_bounded_wait")


__all__ = ["PFError", "lib", "version", "reshape_and_cache", "copy_blocks", "paged_attention_decode", "partition_workspace_layout",
           "alloc_workspace", "workspace_views", "paged_attention_decode_partition", "paged_attention_merge",
           "paged_attention_split", "get_device_error", "check_device_error", "debug_bounded_wait",
           "num_partitions", "STATUS_NAMES"]
