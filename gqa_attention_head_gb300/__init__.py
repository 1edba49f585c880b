"""GB300 (sm_103a) sink attention: grouped-query attention with a per-head sink logit.

Thin ctypes binding of ``libsink_attn.so`` (declared in ``include/sink_attn.h``).
The functions below keep the C names and only marshal arguments: they check
torch tensors (device, dtype, contiguity), allocate the output (and decode
workspace) when the caller passes none, and hand raw device pointers plus the
current CUDA stream to the library. Every step of the computation runs in the
library's CUDA kernels. There is no fallback: if the library is missing or a call
fails, an exception says so. One function goes beyond marshalling:
``sink_attn_prefill_from_host`` orders host<->device copies and per-group
``sink_attn_prefill`` launches on three streams. It moves data; it computes nothing.

Operation ("GPT-OSS am Day 0", §Kernel für GPT-OSS › Sink-Attention): for query
head h, key/value head g = h // G and the visible keys of row i,

    out_i = sum_j exp(s_ij - m) v_j / (exp(sink_h - m) + sum_j exp(s_ij - m)),
    s_ij = scale * <q_i, k_j>,  m = max(sink_h, max_j s_ij).
"""
import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "SinkAttnError", "load_library", "library_path", "sink_attn_prefill", "sink_attn_decode",
    "sink_attn_decode_workspace_bytes", "sink_attn_read_device_error", "sink_attn_status_string",
    "sink_attn_num_sms", "sink_attn_prefill_lse", "sink_attn_decode_lse", "sink_attn_merge_states",
    "sink_attn_append_kv", "sink_attn_prefill_paged", "sink_attn_quantize_fp8",
    "sink_attn_append_kv_fp8", "sink_attn_decode_fp8", "sink_attn_prefill_from_host",
    "sink_attn_prefill_varlen", "STATUS",
]

STATUS = {0: "SINK_ATTN_OK", 1: "SINK_ATTN_ERR_INVALID_ARG", 2: "SINK_ATTN_ERR_UNSUPPORTED",
          3: "SINK_ATTN_ERR_WORKSPACE", 4: "SINK_ATTN_ERR_CUDA", 5: "SINK_ATTN_ERR_DEVICE"}


class SinkAttnError(RuntimeError):
    """A library call returned a status other than SINK_ATTN_OK."""

    def __init__(self, func, status, detail=""):
        self.status = int(status)
        name = STATUS.get(self.status, str(status))
        super().__init__(f"{func} failed: {name} ({sink_attn_status_string(status)}){detail}")


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libsink_attn.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first (python -c "
            "'import __graft_entry__ as g; g.build()'). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    p, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.sink_attn_prefill.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, f32, p, p]
    lib.sink_attn_prefill.restype = ctypes.c_int
    lib.sink_attn_prefill_varlen.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32,
                                             i32, i32, f32, p, p, p]
    lib.sink_attn_prefill_varlen.restype = ctypes.c_int
    lib.sink_attn_decode.argtypes = [p, p, p, i32, i32, p, i32, p, i32, i32, i32, i32, i32, p, i32,
                                     f32, i32, p, sz, p, p]
    lib.sink_attn_decode.restype = ctypes.c_int
    lib.sink_attn_prefill_lse.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, f32, p,
                                          p, p]
    lib.sink_attn_prefill_lse.restype = ctypes.c_int
    lib.sink_attn_decode_lse.argtypes = [p, p, p, i32, i32, p, i32, p, i32, i32, i32, i32, i32, p,
                                         i32, f32, i32, p, sz, p, p, p]
    lib.sink_attn_decode_lse.restype = ctypes.c_int
    lib.sink_attn_append_kv.argtypes = [p, p, p, p, i32, i32, p, i32, p, p, i32, i32, i32, i32, p]
    lib.sink_attn_append_kv.restype = ctypes.c_int
    lib.sink_attn_prefill_paged.argtypes = [p, p, p, p, p, i32, i32, p, i32, p, p, i32, i32, i32,
                                            i32, i32, i32, i32, p, i32, f32, p, p, p]
    lib.sink_attn_prefill_paged.restype = ctypes.c_int
    lib.sink_attn_merge_states.argtypes = [p, p, p, p, i32, i32, i32, p, p, p]
    lib.sink_attn_merge_states.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.sink_attn_quantize_fp8.argtypes = [p, i64, i32, p, p, p]
    lib.sink_attn_quantize_fp8.restype = ctypes.c_int
    lib.sink_attn_append_kv_fp8.argtypes = [p, p, p, p, p, p, i32, i32, p, i32, p, p, i32, i32, i32,
                                            i32, p]
    lib.sink_attn_append_kv_fp8.restype = ctypes.c_int
    lib.sink_attn_decode_fp8.argtypes = [p, p, p, p, p, i32, i32, p, i32, p, i32, i32, i32, i32, i32,
                                         p, i32, f32, i32, p, sz, p, p, p]
    lib.sink_attn_decode_fp8.restype = ctypes.c_int
    lib.sink_attn_prefill_from_host.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, f32,
                                                p, p, p, p, p, p, sz, i32, p, p, p]
    lib.sink_attn_prefill_from_host.restype = ctypes.c_int
    lib.sink_attn_prefill_from_host_scratch_bytes.argtypes = [i32, i32, i32]
    lib.sink_attn_prefill_from_host_scratch_bytes.restype = sz
    lib.sink_attn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.sink_attn_decode_workspace_bytes.restype = sz
    lib.sink_attn_status_string.argtypes = [ctypes.c_int]
    lib.sink_attn_status_string.restype = ctypes.c_char_p
    lib.sink_attn_read_device_error.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    lib.sink_attn_read_device_error.restype = ctypes.c_int
    lib.sink_attn_num_sms.argtypes = []
    lib.sink_attn_num_sms.restype = i32
    _lib = lib
    return lib


def sink_attn_status_string(status) -> str:
    return load_library().sink_attn_status_string(int(status)).decode()


def sink_attn_num_sms() -> int:
    return int(load_library().sink_attn_num_sms())


def sink_attn_decode_workspace_bytes(batch, num_q_heads, head_dim, max_seq_len, kv_chunk=1024):
    return int(load_library().sink_attn_decode_workspace_bytes(batch, num_q_heads, head_dim,
                                                               max_seq_len, kv_chunk))


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _expect(t, name, dtype, device, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")


def sink_attn_prefill(q, k, v, sinks, cu_seqlens, max_seqlen, window=0, scale=None, out=None,
                      stream=None):
    """Ragged causal prefill; returns ``out`` [T, Hq, D] bf16 (allocated if None).

    q [T, Hq, D], k/v [T, Hkv, D] bf16 CUDA; sinks [Hq] fp32 CUDA or None;
    cu_seqlens [S+1] int32 CUDA; max_seqlen a host int bounding every length.
    """
    return _prefill(q, k, v, sinks, cu_seqlens, max_seqlen, window, scale, out, None, stream,
                    False)[0]


def sink_attn_prefill_lse(q, k, v, sinks, cu_seqlens, max_seqlen, window=0, scale=None, out=None,
                          lse=None, stream=None):
    """As sink_attn_prefill, also returning the rows' log-sum-exp: (out, lse [T, Hq] fp32).

    lse = ln(exp(sink) + sum_j exp(s_ij)) (natural log), the state's second half; see
    sink_attn_merge_states.
    """
    return _prefill(q, k, v, sinks, cu_seqlens, max_seqlen, window, scale, out, lse, stream,
                    True)


def sink_attn_prefill_varlen(q, k, v, sinks, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                             max_seqlen_k, window=0, scale=None, out=None, lse=None,
                             want_lse=False, stream=None):
    """Ragged causal prefill with keys of their own: sequence s's queries are the last
    n_s = cu_q[s+1]-cu_q[s] positions of its m_s = cu_k[s+1]-cu_k[s] keys. Returns (out, lse)
    (lse None unless ``want_lse`` or given). q [Tq, Hq, D], k/v [Tk, Hkv, D] bf16 CUDA;
    cu_seqlens_q/k [S+1] int32 CUDA; max_seqlen_q/k host bounds."""
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _expect(q, "q", torch.bfloat16, dev, 3)
    _expect(k, "k", torch.bfloat16, dev, 3)
    _expect(v, "v", torch.bfloat16, dev, 3)
    _expect(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev, 1)
    _expect(cu_seqlens_k, "cu_seqlens_k", torch.int32, dev, 1)
    if cu_seqlens_k.numel() != cu_seqlens_q.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if sinks is not None:
        _expect(sinks, "sinks", torch.float32, dev, 1)
    Tq, hq, d = q.shape
    Tk, hkv, d2 = k.shape
    if d2 != d or v.shape != k.shape:
        raise ValueError("k and v must be [Tk, Hkv, D] with q's D")
    if out is None:
        out = torch.empty_like(q)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((Tq, hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _expect(lse, "lse", torch.float32, dev, 2)
        if lse.shape != (Tq, hq):
            raise ValueError("lse must be [Tq, Hq]")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(dev):
        st = load_library().sink_attn_prefill_varlen(
            _ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            cu_seqlens_q.numel() - 1, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
            int(window), float(scale), _ptr(out), _ptr(lse), _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_prefill_varlen", st)
    return out, lse


_side_streams = {}


def _streams(dev):
    """Two side streams per device (host->device copies, device->host copies), reused."""
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    if key not in _side_streams:
        _side_streams[key] = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    return _side_streams[key]


def sink_attn_prefill_from_host(q, k, v, sinks, cu_seqlens, max_seqlen=None, window=0, scale=None,
                                out=None, device=None, q_dev=None, k_dev=None, v_dev=None,
                                out_dev=None, n_ranges=8):
    """Ragged causal prefill from host tensors, result back in host memory
    (sink_attn_prefill_from_host of the C ABI: copies and kernels overlapped in row ranges).

    q [T, Hq, D], k/v [T, Hkv, D] bf16 on the host (pinned memory lets the copies overlap);
    sinks [Hq] fp32 host or None; cu_seqlens [S+1] int32 host. The rows are cut into
    `n_ranges` equal ranges, in order, regardless of sequence boundaries. Per range a copy
    stream brings in its Q, K and V rows, the varlen prefill runs on the current stream with
    the range's rows as queries and each range-sequence's rows from its start as keys, and a
    second copy stream takes the range's output back. Outputs equal those of one
    sink_attn_prefill over the whole batch up to rounding (a cut moves q-tile boundaries,
    and with them the per-warp O-rescale points). q_dev/k_dev/v_dev/out_dev: optional device
    buffers of the inputs' shapes (allocated when None). `max_seqlen` is not needed (the
    row offsets are on the host) and is accepted for symmetry with sink_attn_prefill.
    Returns `out` (a host tensor, pinned when allocated here). The current stream waits for
    the last copy; synchronise it before reading `out`, and keep the host tensors unchanged
    until then.
    """
    del max_seqlen
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 host tensor")
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape or k.shape[0] != q.shape[0]:
        raise ValueError("q must be [T, Hq, D] and k, v [T, Hkv, D]")
    T, hq, d = q.shape
    hkv = k.shape[1]
    cu = cu_seqlens.to(torch.int32).contiguous()
    if cu.device.type != "cpu" or cu.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D host tensor")
    sk = None
    if sinks is not None:
        sk = sinks.to(torch.float32).contiguous()
        if sk.device.type != "cpu" or sk.shape != (hq,):
            raise ValueError("sinks must be a [Hq] host tensor")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    elif out.device.type != "cpu" or out.dtype != torch.bfloat16 or out.shape != q.shape \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 host tensor of q's shape")
    bufs = []
    for src, given in ((q, q_dev), (k, k_dev), (v, v_dev), (q, out_dev)):
        b = torch.empty(src.shape, dtype=torch.bfloat16, device=dev) if given is None else given
        _expect(b, "device buffer", torch.bfloat16, dev, 3)
        if b.shape != src.shape:
            raise ValueError("device buffers must have the shapes of q, k, v and q")
        bufs.append(b)
    S = cu.numel() - 1
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(dev):
        lib = load_library()
        nbytes = int(lib.sink_attn_prefill_from_host_scratch_bytes(max(S, 0), hq, int(n_ranges)))
        scratch = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        main = torch.cuda.current_stream(dev)
        s_in, s_out = _streams(dev)
        for t in bufs + [scratch]:  # in use on the copy streams until they pass this call
            t.record_stream(s_in)
            t.record_stream(s_out)
        st = lib.sink_attn_prefill_from_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(sk), _ptr(cu), S, T, hq, hkv, d, int(window),
            float(scale), _ptr(out), *(_ptr(b) for b in bufs), _ptr(scratch), nbytes,
            int(n_ranges), ctypes.c_void_p(main.cuda_stream), ctypes.c_void_p(s_in.cuda_stream),
            ctypes.c_void_p(s_out.cuda_stream))
    if st != 0:
        raise SinkAttnError("sink_attn_prefill_from_host", st)
    return out


def _prefill(q, k, v, sinks, cu_seqlens, max_seqlen, window, scale, out, lse, stream, with_lse):
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _expect(q, "q", torch.bfloat16, dev, 3)
    _expect(k, "k", torch.bfloat16, dev, 3)
    _expect(v, "v", torch.bfloat16, dev, 3)
    _expect(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    if sinks is not None:
        _expect(sinks, "sinks", torch.float32, dev, 1)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if k.shape != (T, hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [T, Hkv, D] with q's T and D")
    if out is None:
        out = torch.empty_like(q)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if scale is None:
        scale = d ** -0.5
    if with_lse:
        if lse is None:
            lse = torch.empty((T, hq), dtype=torch.float32, device=dev)
        else:
            _expect(lse, "lse", torch.float32, dev, 2)
            if lse.shape != (T, hq):
                raise ValueError("lse must be [T, Hq]")
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
            int(max_seqlen), hq, hkv, d, int(window), float(scale), _ptr(out))
    with torch.cuda.device(dev):
        lib = load_library()
        if with_lse:
            st = lib.sink_attn_prefill_lse(*args, _ptr(lse), _stream_handle(stream, dev))
        else:
            st = lib.sink_attn_prefill(*args, _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_prefill_lse" if with_lse else "sink_attn_prefill", st)
    return out, lse


def sink_attn_decode(q, k_cache, v_cache, page_table, seq_lens, sinks, max_seq_len, window=0,
                     scale=None, kv_chunk=1024, workspace=None, out=None, stream=None):
    """Paged split-KV decode; returns ``out`` [B, Hq, D] bf16 (allocated if None).

    q [B, Hq, D] bf16; k_cache/v_cache [pages, Hkv, 16, D] bf16 (HND); page_table
    [B, max_pages] int32; seq_lens [B] int32 (all CUDA); max_seq_len a host int.
    ``workspace`` is a uint8 CUDA tensor of at least
    ``sink_attn_decode_workspace_bytes(...)`` bytes (allocated if None).
    """
    return _decode(q, k_cache, v_cache, page_table, seq_lens, sinks, max_seq_len, window, scale,
                   kv_chunk, workspace, out, None, stream, False)[0]


def sink_attn_decode_lse(q, k_cache, v_cache, page_table, seq_lens, sinks, max_seq_len, window=0,
                         scale=None, kv_chunk=1024, workspace=None, out=None, lse=None,
                         stream=None):
    """As sink_attn_decode, also returning the log-sum-exp: (out, lse [B, Hq] fp32)."""
    return _decode(q, k_cache, v_cache, page_table, seq_lens, sinks, max_seq_len, window, scale,
                   kv_chunk, workspace, out, lse, stream, True)


def _decode(q, k_cache, v_cache, page_table, seq_lens, sinks, max_seq_len, window, scale, kv_chunk,
            workspace, out, lse, stream, with_lse):
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _expect(q, "q", torch.bfloat16, dev, 3)
    _expect(k_cache, "k_cache", torch.bfloat16, dev, 4)
    _expect(v_cache, "v_cache", torch.bfloat16, dev, 4)
    _expect(page_table, "page_table", torch.int32, dev, 2)
    _expect(seq_lens, "seq_lens", torch.int32, dev, 1)
    if sinks is not None:
        _expect(sinks, "sinks", torch.float32, dev, 1)
    B, hq, d = q.shape
    npages, hkv, psz, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [pages, Hkv, page_size, D] with q's D")
    if page_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("page_table and seq_lens must have q's batch size")
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    need = int(lib.sink_attn_decode_workspace_bytes(B, hq, d, int(max_seq_len), int(kv_chunk)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _expect(workspace, "workspace", torch.uint8, dev, 1)
    if out is None:
        out = torch.empty_like(q)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if with_lse:
        if lse is None:
            lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
        else:
            _expect(lse, "lse", torch.float32, dev, 2)
            if lse.shape != (B, hq):
                raise ValueError("lse must be [B, Hq]")
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), npages, psz, _ptr(page_table),
            page_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), hq, hkv, d, _ptr(sinks),
            int(window), float(scale), int(kv_chunk), _ptr(workspace),
            0 if workspace is None else workspace.numel(), _ptr(out))
    with torch.cuda.device(dev):
        if with_lse:
            st = lib.sink_attn_decode_lse(*args, _ptr(lse), _stream_handle(stream, dev))
        else:
            st = lib.sink_attn_decode(*args, _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_decode_lse" if with_lse else "sink_attn_decode", st)
    return out, lse


def sink_attn_merge_states(o_a, lse_a, o_b, lse_b, out=None, lse_out=None, want_lse=True,
                           stream=None):
    """Merge two attention states over disjoint key sets; returns (out, lse_out).

    o_a/o_b [R, H, D] bf16, lse_a/lse_b [R, H] fp32 (natural log), all CUDA and on one
    device. out is allocated if None; lse_out too when ``want_lse`` (else None is passed
    and returned). See include/sink_attn.h for the formula.
    """
    dev = o_a.device
    if dev.type != "cuda":
        raise ValueError("o_a must be a CUDA tensor")
    _expect(o_a, "o_a", torch.bfloat16, dev, 3)
    _expect(o_b, "o_b", torch.bfloat16, dev, 3)
    _expect(lse_a, "lse_a", torch.float32, dev, 2)
    _expect(lse_b, "lse_b", torch.float32, dev, 2)
    R, H, d = o_a.shape
    if o_b.shape != o_a.shape or lse_a.shape != (R, H) or lse_b.shape != (R, H):
        raise ValueError("o_a/o_b must be [R, H, D] and lse_a/lse_b [R, H]")
    if out is None:
        out = torch.empty_like(o_a)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
        if out.shape != o_a.shape:
            raise ValueError("out must have o_a's shape")
    if want_lse and lse_out is None:
        lse_out = torch.empty_like(lse_a)
    elif lse_out is not None:
        _expect(lse_out, "lse_out", torch.float32, dev, 2)
        if lse_out.shape != (R, H):
            raise ValueError("lse_out must be [R, H]")
    with torch.cuda.device(dev):
        st = load_library().sink_attn_merge_states(
            _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), R, H, d, _ptr(out), _ptr(lse_out),
            _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_merge_states", st)
    return out, lse_out


def _paged_args(k_new, v_new, k_cache, v_cache, page_table, cu_seqlens, seq_lens, dev,
                cache_dtype=torch.bfloat16):
    _expect(k_new, "k_new", torch.bfloat16, dev, 3)
    _expect(v_new, "v_new", torch.bfloat16, dev, 3)
    _expect(k_cache, "k_cache", cache_dtype, dev, 4)
    _expect(v_cache, "v_cache", cache_dtype, dev, 4)
    _expect(page_table, "page_table", torch.int32, dev, 2)
    _expect(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    _expect(seq_lens, "seq_lens", torch.int32, dev, 1)
    T, hkv, d = k_new.shape
    npages, hkv2, psz, d2 = k_cache.shape
    if v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or hkv2 != hkv or d2 != d:
        raise ValueError("k_new/v_new [T, Hkv, D] and k_cache/v_cache [pages, Hkv, P, D] disagree")
    S = cu_seqlens.numel() - 1
    if seq_lens.numel() != S or page_table.shape[0] != S:
        raise ValueError("seq_lens and page_table must have one entry/row per sequence")
    return T, hkv, d, npages, psz, S


def sink_attn_append_kv(k_new, v_new, k_cache, v_cache, page_table, cu_seqlens, seq_lens,
                        stream=None):
    """Write the new rows' K/V into the paged cache in place (see include/sink_attn.h).

    k_new/v_new [T, Hkv, D] bf16; k_cache/v_cache [pages, Hkv, 16, D] bf16; page_table
    [S, max_pages] int32; cu_seqlens [S+1] int32 (new rows); seq_lens [S] int32 (tokens
    after the append). All CUDA.
    """
    dev = k_new.device
    if dev.type != "cuda":
        raise ValueError("k_new must be a CUDA tensor")
    T, hkv, d, npages, psz, S = _paged_args(k_new, v_new, k_cache, v_cache, page_table,
                                            cu_seqlens, seq_lens, dev)
    with torch.cuda.device(dev):
        st = load_library().sink_attn_append_kv(
            _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), npages, psz, _ptr(page_table),
            page_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens), S, T, hkv, d,
            _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_append_kv", st)


def sink_attn_prefill_paged(q, k_new, v_new, k_cache, v_cache, page_table, cu_seqlens, seq_lens,
                            sinks, max_q_len, max_seq_len, window=0, scale=None, out=None,
                            lse=None, want_lse=False, stream=None):
    """Chunked prefill over the paged cache: append the new rows' K/V, then attend the new
    queries to all cached keys of their sequence. Returns (out, lse) (lse None unless
    ``want_lse`` or given). q [T, Hq, D] bf16 (new rows); see sink_attn_append_kv for the rest.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _expect(q, "q", torch.bfloat16, dev, 3)
    T, hkv, d, npages, psz, S = _paged_args(k_new, v_new, k_cache, v_cache, page_table,
                                            cu_seqlens, seq_lens, dev)
    if q.shape[0] != T or q.shape[2] != d:
        raise ValueError("q must be [T, Hq, D] with k_new's T and D")
    hq = q.shape[1]
    if sinks is not None:
        _expect(sinks, "sinks", torch.float32, dev, 1)
    if out is None:
        out = torch.empty_like(q)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((T, hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _expect(lse, "lse", torch.float32, dev, 2)
        if lse.shape != (T, hq):
            raise ValueError("lse must be [T, Hq]")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(dev):
        st = load_library().sink_attn_prefill_paged(
            _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), npages, psz,
            _ptr(page_table), page_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens), S, T,
            int(max_q_len), int(max_seq_len), hq, hkv, d, _ptr(sinks), int(window), float(scale),
            _ptr(out), _ptr(lse), _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_prefill_paged", st)
    return out, lse


# ---------------------------------------------------------------------------
# FP8 KV cache: e4m3 codes (uint8) [pages, Hkv, 16, D] + fp32 row scales [pages, Hkv, 16].
# ---------------------------------------------------------------------------

def _expect_scales(t, name, codes, dev):
    _expect(t, name, torch.float32, dev, codes.dim() - 1)
    if tuple(t.shape) != tuple(codes.shape[:-1]):
        raise ValueError(f"{name} must have shape {tuple(codes.shape[:-1])}")


def sink_attn_quantize_fp8(x, codes=None, scales=None, stream=None):
    """Quantise bf16 rows x [..., D] to the FP8 cache format; returns (codes uint8 [..., D],
    scales fp32 [...]). A whole bf16 cache [pages, Hkv, 16, D] converts in one call."""
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    _expect(x, "x", torch.bfloat16, dev)
    d = x.shape[-1]
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=dev)
    _expect(codes, "codes", torch.uint8, dev, x.dim())
    if codes.shape != x.shape:
        raise ValueError("codes must have x's shape")
    _expect_scales(scales, "scales", codes, dev)
    rows = x.numel() // d if d else 0
    with torch.cuda.device(dev):
        st = load_library().sink_attn_quantize_fp8(_ptr(x), rows, d, _ptr(codes), _ptr(scales),
                                                   _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_quantize_fp8", st)
    return codes, scales


def sink_attn_append_kv_fp8(k_new, v_new, k_codes, v_codes, k_scale, v_scale, page_table,
                            cu_seqlens, seq_lens, stream=None):
    """sink_attn_append_kv into the FP8 cache: the new rows are quantised into their slots."""
    dev = k_new.device
    if dev.type != "cuda":
        raise ValueError("k_new must be a CUDA tensor")
    T, hkv, d, npages, psz, S = _paged_args(k_new, v_new, k_codes, v_codes, page_table,
                                            cu_seqlens, seq_lens, dev, torch.uint8)
    _expect_scales(k_scale, "k_scale", k_codes, dev)
    _expect_scales(v_scale, "v_scale", v_codes, dev)
    with torch.cuda.device(dev):
        st = load_library().sink_attn_append_kv_fp8(
            _ptr(k_new), _ptr(v_new), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
            npages, psz, _ptr(page_table), page_table.shape[1], _ptr(cu_seqlens), _ptr(seq_lens),
            S, T, hkv, d, _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_append_kv_fp8", st)


def sink_attn_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, page_table, seq_lens, sinks,
                         max_seq_len, window=0, scale=None, kv_chunk=1024, workspace=None,
                         out=None, lse=None, want_lse=False, stream=None):
    """Paged split-KV decode over the FP8 cache; returns (out, lse) (lse None unless
    ``want_lse`` or given). q [B, Hq, D] bf16; codes uint8 [pages, Hkv, 16, D]; scales fp32
    [pages, Hkv, 16]; the rest as sink_attn_decode."""
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _expect(q, "q", torch.bfloat16, dev, 3)
    _expect(k_codes, "k_codes", torch.uint8, dev, 4)
    _expect(v_codes, "v_codes", torch.uint8, dev, 4)
    _expect_scales(k_scale, "k_scale", k_codes, dev)
    _expect_scales(v_scale, "v_scale", v_codes, dev)
    _expect(page_table, "page_table", torch.int32, dev, 2)
    _expect(seq_lens, "seq_lens", torch.int32, dev, 1)
    if sinks is not None:
        _expect(sinks, "sinks", torch.float32, dev, 1)
    B, hq, d = q.shape
    npages, hkv, psz, d2 = k_codes.shape
    if d2 != d or v_codes.shape != k_codes.shape:
        raise ValueError("k_codes/v_codes must be [pages, Hkv, page_size, D] with q's D")
    if page_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("page_table and seq_lens must have q's batch size")
    if scale is None:
        scale = d ** -0.5
    lib = load_library()
    need = int(lib.sink_attn_decode_workspace_bytes(B, hq, d, int(max_seq_len), int(kv_chunk)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _expect(workspace, "workspace", torch.uint8, dev, 1)
    if out is None:
        out = torch.empty_like(q)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _expect(lse, "lse", torch.float32, dev, 2)
        if lse.shape != (B, hq):
            raise ValueError("lse must be [B, Hq]")
    with torch.cuda.device(dev):
        st = lib.sink_attn_decode_fp8(
            _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), npages, psz,
            _ptr(page_table), page_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), hq, hkv, d,
            _ptr(sinks), int(window), float(scale), int(kv_chunk), _ptr(workspace),
            0 if workspace is None else workspace.numel(), _ptr(out), _ptr(lse),
            _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_decode_fp8", st)
    return out, lse


def sink_attn_read_device_error(stream=None, device=None):
    """Synchronise the stream, return (status, bits) of the device error word and clear it."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    bits = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        st = load_library().sink_attn_read_device_error(_stream_handle(stream, dev),
                                                        ctypes.byref(bits))
    return int(st), int(bits.value)


def sink_attn_debug_decode_withhold_page(enable, wait_limit_ns=1_000_000_000):
    """Test switch for the decode's failure path (process-wide; see include/sink_attn.h).

    With ``enable``, later decode launches never copy the first page of (chunk 0, kv head 0,
    sequence 0), so the wait for it runs out after ``wait_limit_ns`` and the device error
    word gets SINK_ATTN_DEVERR_WAIT_TIMEOUT; ``enable=False`` restores normal launches.
    """
    lib = load_library()
    fn = lib.sink_attn_debug_decode_withhold_page
    fn.argtypes = [ctypes.c_int32, ctypes.c_uint64]
    fn.restype = None
    fn(1 if enable else 0, int(wait_limit_ns))


def sink_attn_decode_static_workspace(q, k_cache, v_cache, page_table, seq_lens, sinks,
                                      max_seq_len, window=0, scale=None, kv_chunk=1024,
                                      out=None, stream=None):
    """Paged split-KV decode that allocates no device memory for its scratch.

    For callers that cannot allocate device memory (a plugin handed only its input and
    output buffers by a framework that owns all allocations, or a decode loop that must
    not call cudaMalloc because it can synchronise the device). The split-KV scratch is
    a fixed 16 MiB array inside the library; sizes that need more are rejected with
    SINK_ATTN_ERR_WORKSPACE. Calls that overlap on the GPU share that array and race:
    serialise them. Arguments and results are those of ``sink_attn_decode``; pass
    ``out`` to keep the call itself free of torch allocations too. The first call on a
    device looks up the array there; with CUDA's default lazy module loading that lookup
    also loads the module and reserves the array (it may allocate and synchronise), so
    make one warm-up call per device before a latency-critical loop or a stream capture.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _expect(q, "q", torch.bfloat16, dev, 3)
    _expect(k_cache, "k_cache", torch.bfloat16, dev, 4)
    _expect(v_cache, "v_cache", torch.bfloat16, dev, 4)
    _expect(page_table, "page_table", torch.int32, dev, 2)
    _expect(seq_lens, "seq_lens", torch.int32, dev, 1)
    if sinks is not None:
        _expect(sinks, "sinks", torch.float32, dev, 1)
    B, hq, d = q.shape
    npages, hkv, psz, _ = k_cache.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    else:
        _expect(out, "out", torch.bfloat16, dev, 3)
    lib = load_library()
    fn = lib.sink_attn_decode_static_workspace
    p, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [p, p, p, i32, i32, p, i32, p, i32, i32, i32, i32, i32, p, i32, ctypes.c_float,
                   i32, p, p]
    fn.restype = ctypes.c_int
    with torch.cuda.device(dev):
        st = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), npages, psz, _ptr(page_table),
                page_table.shape[1], _ptr(seq_lens), B, int(max_seq_len), hq, hkv, d,
                _ptr(sinks), int(window), float(scale), int(kv_chunk), _ptr(out),
                _stream_handle(stream, dev))
    if st != 0:
        raise SinkAttnError("sink_attn_decode_static_workspace", st)
    return out
