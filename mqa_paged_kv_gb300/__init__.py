"""Python binding of libpaged_attn.so (paged-KV GQA/MQA attention, sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.
The functions carry the C ABI's names (include/paged_attn.h) and take
torch tensors for device memory and the current torch CUDA stream.  If the
compiled library is missing this module raises at import; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpaged_attn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python mqa_paged_kv_gb300/build.py` "
        "(nvcc, sm_103a); there is no CPU or library fallback")

_lib = ctypes.CDLL(LIB_PATH)

PA_F16 = 0
PA_BF16 = 1
PA_DEV_BAD_BLOCK_ID = 0x1
PA_DEV_BAD_SLOT = 0x2
PA_DEV_WAIT_TIMEOUT = 0x4
PA_DEV_BAD_LENGTHS = 0x8

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_lib.pa_status_string.argtypes = [_I]
_lib.pa_status_string.restype = ctypes.c_char_p
_lib.pa_version.argtypes = []
_lib.pa_version.restype = _I
_lib.pa_last_launch_count.argtypes = []
_lib.pa_last_launch_count.restype = _I
_lib.pa_limit_next_call_ctas.argtypes = [_I]
_lib.pa_limit_next_call_ctas.restype = None
_lib.pa_last_cuda_error.argtypes = []
_lib.pa_last_cuda_error.restype = _I
_lib.pa_last_cuda_error_string.argtypes = []
_lib.pa_last_cuda_error_string.restype = ctypes.c_char_p
_lib.reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]
_lib.reshape_and_cache.restype = _I
_lib.paged_attn_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I, _I]
_lib.paged_attn_workspace_bytes.restype = _SZ
_lib.paged_attn_decode.argtypes = [_P, _P, _P, _P, _I, _P, _F, _I, _I, _I, _I, _I, _I, _I,
                                   _I, _P, _P, _SZ, _P]
_lib.paged_attn_decode.restype = _I
_lib.paged_attn_chunked_prefill_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I]
_lib.paged_attn_chunked_prefill_workspace_bytes.restype = _SZ
_lib.paged_attn_chunked_prefill.argtypes = [_P, _P, _P, _P, _I, _P, _P, _I, _I, _F, _I, _I,
                                            _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]
_lib.paged_attn_chunked_prefill.restype = _I
_lib.paged_attn_cross_attention.argtypes = _lib.paged_attn_chunked_prefill.argtypes
_lib.paged_attn_cross_attention.restype = _I
_lib.gqa_varlen_prefill_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
_lib.gqa_varlen_prefill_workspace_bytes.restype = _SZ
_lib.gqa_varlen_prefill.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _F, _I, _I, _I, _I, _I,
                                    _P, _P, _SZ, _P]
_lib.gqa_varlen_prefill.restype = _I
_lib.pa_read_device_status.argtypes = [_P, _I, ctypes.POINTER(ctypes.c_uint32), _P]
_lib.pa_read_device_status.restype = _I

_lib.paged_attn_decode_noalloc.argtypes = [_P, _P, _P, _P, _I, _P, _F, _I, _I, _I, _I, _I,
                                           _I, _I, _I, _P, _P]
_lib.paged_attn_decode_noalloc.restype = _I
_lib.pa_profile_next_call.argtypes = [_P, _P]
_lib.pa_profile_next_call.restype = None
_lib.pa_set_pipeline_wait_limit.argtypes = [ctypes.c_uint64]
_lib.pa_set_pipeline_wait_limit.restype = None

EXPORTED = ["pa_profile_next_call", "pa_status_string", "pa_version", "pa_last_launch_count",
            "pa_last_cuda_error", "pa_last_cuda_error_string", "pa_limit_next_call_ctas",
            "reshape_and_cache",
            "paged_attn_workspace_bytes", "paged_attn_decode",
            "paged_attn_chunked_prefill_workspace_bytes", "paged_attn_chunked_prefill",
            "pa_read_device_status", "paged_attn_decode_noalloc",
            "paged_attn_cross_attention", "gqa_varlen_prefill_workspace_bytes",
            "gqa_varlen_prefill", "pa_set_pipeline_wait_limit"]


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        if status == -7:  # PA_ERR_CUDA: name the runtime error behind it
            msg += f": {_lib.pa_last_cuda_error_string().decode()} ({_lib.pa_last_cuda_error()})"
        super().__init__(msg)


def status_string(status: int) -> str:
    return _lib.pa_status_string(int(status)).decode()


def last_launch_count() -> int:
    return int(_lib.pa_last_launch_count())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    return -1


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise PagedAttnError(rc, where)


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


# The C ABI sees raw pointers and sizes only, so the binding checks what a
# pointer cannot carry -- device, integer width, matching shapes -- before any
# allocation or launch: a host tensor, an int64 table or a short lengths
# array would otherwise reach the kernels as a bad address or a misread.
def _expect(ok: bool, msg: str) -> None:
    if not ok:
        raise ValueError(msg)


def _same_device(ref: torch.Tensor, **named) -> None:
    _expect(ref.device.type == "cuda", f"tensors must be CUDA tensors (got {ref.device})")
    for name, t in named.items():
        if t is not None:
            _expect(t.device == ref.device, f"{name} is on {t.device}, expected {ref.device}")


def _int32(**named) -> None:
    for name, t in named.items():
        _expect(t.dtype == torch.int32, f"{name} must be int32 (got {t.dtype})")


def _check_paged(q, k_cache, v_cache, block_tables, context_lens, out, workspace,
                 cu_query_lens=None) -> None:
    """Shapes and types shared by the paged attention calls: q [T, Hq, D],
    caches [NB, Hkv, bs, D] of q's type, block_tables [B, MBS] and
    context_lens [B] int32, cu_query_lens [B + 1] int32, out like q."""
    _expect(q.dim() == 3 and k_cache.dim() == 4, "q must be [T, Hq, D], caches [NB, Hkv, bs, D]")
    _expect(v_cache.shape == k_cache.shape and k_cache.shape[3] == q.shape[2],
            "k_cache and v_cache must have one shape whose last dim is q's head_dim")
    _expect(k_cache.dtype == q.dtype and v_cache.dtype == q.dtype, "caches must have q's dtype")
    _int32(block_tables=block_tables, context_lens=context_lens)
    B = context_lens.shape[0]
    _expect(context_lens.dim() == 1 and block_tables.dim() == 2 and block_tables.shape[0] == B,
            "block_tables must be [B, max_blocks] and context_lens [B]")
    if cu_query_lens is None:
        _expect(q.shape[0] == B, "decode takes one query row per sequence")
    else:
        _int32(cu_query_lens=cu_query_lens)
        _expect(cu_query_lens.shape == (B + 1,), "cu_query_lens must be [B + 1]")
    if out is not None:
        _expect(out.shape == q.shape and out.dtype == q.dtype, "out must match q")
    _same_device(q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                 context_lens=context_lens, cu_query_lens=cu_query_lens, out=out,
                 workspace=workspace)


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      status_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v [T, Hkv, D] -> k_cache, v_cache [NB, Hkv, bs, D] at slot_mapping
    (int64, -1 skips)."""
    _contig(k, v, k_cache, v_cache, slot_mapping)
    _expect(status_word is None
            or status_word.dtype in (torch.int32, getattr(torch, "uint32", None)),
            "status_word must be a 32-bit integer tensor")
    _expect(k.dim() == 3 and k_cache.dim() == 4 and slot_mapping.shape == (k.shape[0],),
            "k, v must be [T, Hkv, D], caches [NB, Hkv, bs, D], slot_mapping [T]")
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = k_cache.shape
    if Hkv2 != Hkv or D2 != D or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if slot_mapping.dtype != torch.int64 or not (k.dtype == v.dtype == k_cache.dtype
                                                 == v_cache.dtype):
        raise ValueError("slot_mapping must be int64 and caches match k's dtype")
    _same_device(k, v=v, k_cache=k_cache, v_cache=v_cache, slot_mapping=slot_mapping,
                 status_word=status_word)
    rc = _lib.reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                _ptr(slot_mapping), T, Hkv, D, bs, NB, _dtype_code(k),
                                _ptr(status_word), _stream(stream))
    _check(rc, "reshape_and_cache")


def paged_attn_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int,
                               head_dim: int, max_blocks_per_seq: int, block_size: int,
                               num_splits: int = 0) -> int:
    return int(_lib.paged_attn_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                               max_blocks_per_seq, block_size, num_splits))


def paged_attn_chunked_prefill_workspace_bytes(num_seqs: int, total_query_tokens: int,
                                               num_heads: int, num_kv_heads: int,
                                               head_dim: int, max_blocks_per_seq: int,
                                               block_size: int, num_splits: int = 0) -> int:
    return int(_lib.paged_attn_chunked_prefill_workspace_bytes(
        num_seqs, total_query_tokens, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
        block_size, num_splits))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned workspace (torch's allocator aligns to 512 B)."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, num_splits: int = 0,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q [B, Hq, D]; caches [NB, Hkv, bs, D]; block_tables [B, MBS] int32;
    context_lens [B] int32 -> out [B, Hq, D]."""
    _contig(q, k_cache, v_cache, block_tables, context_lens, out)
    _check_paged(q, k_cache, v_cache, block_tables, context_lens, out, workspace)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    mbs = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(
            paged_attn_workspace_bytes(B, Hq, Hkv, D, mbs, bs, num_splits), q.device)
    rc = _lib.paged_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mbs,
                                _ptr(context_lens), float(scale), B, Hq, Hkv, D, bs, NB,
                                _dtype_code(q), num_splits, _ptr(out), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "paged_attn_decode")
    return out


def paged_attn_chunked_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, cu_query_lens: torch.Tensor,
                               context_lens: torch.Tensor, max_query_len: int, scale: float,
                               out: Optional[torch.Tensor] = None, num_splits: int = 0,
                               workspace: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """q [T, Hq, D] in the cu_query_lens layout -> out [T, Hq, D]."""
    _contig(q, k_cache, v_cache, block_tables, cu_query_lens, context_lens, out)
    _check_paged(q, k_cache, v_cache, block_tables, context_lens, out, workspace,
                 cu_query_lens=cu_query_lens)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    B = context_lens.shape[0]
    mbs = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(paged_attn_chunked_prefill_workspace_bytes(
            B, T, Hq, Hkv, D, mbs, bs, num_splits), q.device)
    rc = _lib.paged_attn_chunked_prefill(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mbs, _ptr(cu_query_lens),
        _ptr(context_lens), T, int(max_query_len), float(scale), B, Hq, Hkv, D, bs, NB,
        _dtype_code(q), num_splits, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "paged_attn_chunked_prefill")
    return out


def paged_attn_cross_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, cu_query_lens: torch.Tensor,
                               context_lens: torch.Tensor, max_query_len: int, scale: float,
                               out: Optional[torch.Tensor] = None, num_splits: int = 0,
                               workspace: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """Decoder rows q [T, Hq, D] (cu_query_lens layout) over a static encoder
    cache; context_lens = encoder tokens per sequence; no causal mask."""
    _contig(q, k_cache, v_cache, block_tables, cu_query_lens, context_lens, out)
    _check_paged(q, k_cache, v_cache, block_tables, context_lens, out, workspace,
                 cu_query_lens=cu_query_lens)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    B = context_lens.shape[0]
    mbs = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(paged_attn_chunked_prefill_workspace_bytes(
            B, T, Hq, Hkv, D, mbs, bs, num_splits), q.device)
    rc = _lib.paged_attn_cross_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mbs, _ptr(cu_query_lens),
        _ptr(context_lens), T, int(max_query_len), float(scale), B, Hq, Hkv, D, bs, NB,
        _dtype_code(q), num_splits, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "paged_attn_cross_attention")
    return out


def gqa_varlen_prefill_workspace_bytes(num_seqs: int, total_query_tokens: int, num_heads: int,
                                       num_kv_heads: int, head_dim: int) -> int:
    return int(_lib.gqa_varlen_prefill_workspace_bytes(num_seqs, total_query_tokens, num_heads,
                                                       num_kv_heads, head_dim))


def gqa_varlen_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                       max_seqlen_q: int, scale: float, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q [Tq, Hq, D], k, v [Tk, Hkv, D] contiguous; cu_seqlens int32 [B+1]
    -> out [Tq, Hq, D] (bottom-right causal per sequence, no cache)."""
    _contig(q, k, v, cu_seqlens_q, cu_seqlens_k, out)
    _expect(q.dim() == 3 and k.dim() == 3 and v.shape == k.shape and k.shape[2] == q.shape[2],
            "q must be [Tq, Hq, D], k and v [Tk, Hkv, D]")
    _expect(k.dtype == q.dtype and v.dtype == q.dtype, "k and v must have q's dtype")
    _int32(cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k)
    _expect(cu_seqlens_q.dim() == 1 and cu_seqlens_k.shape == cu_seqlens_q.shape,
            "cu_seqlens_q and cu_seqlens_k must both be [B + 1]")
    _expect(out is None or (out.shape == q.shape and out.dtype == q.dtype), "out must match q")
    _same_device(q, k=k, v=v, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, out=out,
                 workspace=workspace)
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    B = cu_seqlens_q.shape[0] - 1
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(gqa_varlen_prefill_workspace_bytes(B, Tq, Hq, Hkv, D),
                                    q.device)
    rc = _lib.gqa_varlen_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), Tq, Tk, int(max_seqlen_q), float(scale), B,
                                 Hq, Hkv, D, _dtype_code(q), _ptr(out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gqa_varlen_prefill")
    return out


def pa_read_device_status(workspace: torch.Tensor, clear: bool = False, stream=None) -> int:
    _same_device(workspace)
    flags = ctypes.c_uint32(0)
    rc = _lib.pa_read_device_status(_ptr(workspace), int(bool(clear)), ctypes.byref(flags),
                                    _stream(stream))
    _check(rc, "pa_read_device_status")
    return int(flags.value)


def pa_set_pipeline_wait_limit(limit_ns: int) -> None:
    """Limit of each pipeline wait of the decode kernels enqueued from now
    on (0 = the default 2 s); see include/paged_attn.h."""
    _lib.pa_set_pipeline_wait_limit(int(limit_ns))


def pa_limit_next_call_ctas(max_ctas: int) -> None:
    """Run the next attention call's persistent kernels on at most max_ctas
    SMs (see include/paged_attn.h)."""
    _lib.pa_limit_next_call_ctas(int(max_ctas))


def pa_profile_next_call(start_event, stop_event) -> None:
    """Record two torch.cuda.Event objects around the attention kernels of
    the next call on this thread (see include/paged_attn.h)."""
    for ev in (start_event, stop_event):
        if not ev.cuda_event:  # torch creates the CUDA event on first record
            ev.record()
    _lib.pa_profile_next_call(ctypes.c_void_p(start_event.cuda_event),
                              ctypes.c_void_p(stop_event.cuda_event))
