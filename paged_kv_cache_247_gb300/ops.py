"""torch-facing binding of the device calls (marshalling only).

Each function checks tensor placement, dtype and layout, then hands raw
device pointers and the current CUDA stream to the C ABI.  All arithmetic
happens in the library's kernels; nothing here computes a result.
"""

import ctypes

import numpy as np
import torch

from . import _lib

_DTYPE_CODE = {torch.float16: _lib.PKV_F16, torch.bfloat16: _lib.PKV_BF16}
_SIZE_T_MAX = ctypes.c_size_t(-1).value


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def decode_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len):
    """Tokens per partition the library picks on the current device."""
    return _lib.load().pkv_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_context_len)


def decode_uses_tensor_cores(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                             partition_size=0):
    """Whether a decode call of these sizes runs the tensor-core kernel."""
    r = _lib.load().pkv_decode_uses_tensor_cores(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_context_len, partition_size)
    if r < 0:
        raise ValueError("invalid decode sizes")
    return bool(r)


def set_decode_path(path):
    """Process-wide decode kernel choice: 0 = library's choice, 1 = CUDA cores,
    2 = tensor cores where supported."""
    _lib.check(_lib.load().pkv_set_decode_path(int(path)), "pkv_set_decode_path")


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                          partition_size=0):
    """Bytes of scratch :func:`paged_attn_decode` needs (0 when it does not split)."""
    n = _lib.load().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              max_context_len, partition_size)
    if n == _SIZE_T_MAX:
        raise ValueError("invalid decode sizes")
    return n


def paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                      max_context_len, partition_size=0, workspace=None):
    """softmax(scale * q.K) V for every sequence and query head, K/V read
    through the block table.  Writes ``out`` ([S, Hq, D]) and returns it.

    ``workspace`` (uint8 CUDA tensor) is used when the context is split into
    partitions; if omitted and needed, one is allocated here with torch.
    """
    _cuda(q, "q", ndim=3)
    dtype = q.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError("q must be float16 or bfloat16")
    _cuda(out, "out", dtype, 3)
    _cuda(k_cache, "k_cache", dtype, 4)
    _cuda(v_cache, "v_cache", dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables / context_lens must have one row per sequence")
    lib = _lib.load()
    ws_bytes = decode_workspace_size(S, Hq, Hkv, D, max_context_len, partition_size)
    ws_ptr, ws_len = None, 0
    if ws_bytes:
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
        _cuda(workspace, "workspace")
        ws_ptr, ws_len = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.pkv_paged_attn_decode(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(),
        int(max_context_len), S, Hq, Hkv, D, B, NB, float(scale), _DTYPE_CODE[dtype],
        int(partition_size), ws_ptr, ws_len, _stream_handle(q.device))
    _lib.check(st, "pkv_paged_attn_decode")
    return out


def paged_attn_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                             context_lens, scale, max_context_len, partition_size=0,
                             workspace=None):
    """One fused decode step: write each sequence's new token (``k_new``,
    ``v_new`` [S, Hkv, D], position ``context_lens[s] - 1``) into its slot and
    attend over the whole context in the same launch."""
    _cuda(q, "q", ndim=3)
    dtype = q.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError("q must be float16 or bfloat16")
    for t, name in ((out, "out"), (k_new, "k_new"), (v_new, "v_new")):
        _cuda(t, name, dtype, 3)
    _cuda(k_cache, "k_cache", dtype, 4)
    _cuda(v_cache, "v_cache", dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if (v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape
            or k_new.shape != (S, Hkv, D) or v_new.shape != (S, Hkv, D)):
        raise ValueError("shape mismatch between q, out, new rows and the caches")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables / context_lens must have one row per sequence")
    lib = _lib.load()
    ws_bytes = decode_workspace_size(S, Hq, Hkv, D, max_context_len, partition_size)
    ws_ptr, ws_len = None, 0
    if ws_bytes:
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
        _cuda(workspace, "workspace")
        ws_ptr, ws_len = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.pkv_paged_attn_decode_append(
        out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
        context_lens.data_ptr(), int(max_context_len), S, Hq, Hkv, D, B, NB, float(scale),
        _DTYPE_CODE[dtype], int(partition_size), ws_ptr, ws_len, _stream_handle(q.device))
    _lib.check(st, "pkv_paged_attn_decode_append")
    return out


def paged_attn_prefill(out, q, query_start, k_cache, v_cache, block_tables, context_lens, scale,
                       max_context_len, max_query_len):
    """Causal multi-query attention of each sequence's last L_s positions
    (``q[query_start[s]:query_start[s+1]]``) over its paged context, on the
    tensor cores.  Writes ``out`` ([total_queries, Hq, D]) and returns it."""
    _cuda(q, "q", ndim=3)
    dtype = q.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError("q must be float16 or bfloat16")
    _cuda(out, "out", dtype, 3)
    _cuda(k_cache, "k_cache", dtype, 4)
    _cuda(v_cache, "v_cache", dtype, 4)
    _cuda(block_tables, "block_tables", torch.int32, 2)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    _cuda(query_start, "query_start", torch.int32, 1)
    T, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    S = context_lens.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    if block_tables.shape[0] != S or query_start.shape[0] != S + 1:
        raise ValueError("block_tables / query_start must match context_lens")
    st = _lib.load().pkv_paged_attn_prefill(
        out.data_ptr(), q.data_ptr(), T, query_start.data_ptr(), int(max_query_len),
        k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
        context_lens.data_ptr(), int(max_context_len), S, Hq, Hkv, D, B, NB, float(scale),
        _DTYPE_CODE[dtype], _stream_handle(q.device))
    _lib.check(st, "pkv_paged_attn_prefill")
    return out


def contiguous_attn_decode(out, q, k_cache, v_cache, context_lens, scale, partition_size=0,
                           workspace=None):
    """Decode over a contiguous cache ``[S, Hkv, capacity, D]`` (no block
    table): the baseline the paged layout is compared with.  It runs the
    CUDA-core decode kernel, whatever the decode-path setting."""
    _cuda(q, "q", ndim=3)
    dtype = q.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError("q must be float16 or bfloat16")
    _cuda(out, "out", dtype, 3)
    _cuda(k_cache, "k_cache", dtype, 4)
    _cuda(v_cache, "v_cache", dtype, 4)
    _cuda(context_lens, "context_lens", torch.int32, 1)
    S, Hq, D = q.shape
    S2, Hkv, cap, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or S2 != S or out.shape != q.shape:
        raise ValueError("shape mismatch between q, out and the caches")
    lib = _lib.load()
    ws_bytes = lib.pkv_contiguous_workspace_size(S, Hq, Hkv, D, cap, partition_size)
    if ws_bytes == _SIZE_T_MAX:
        raise ValueError("invalid decode sizes")
    ws_ptr, ws_len = None, 0
    if ws_bytes:
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
        _cuda(workspace, "workspace")
        ws_ptr, ws_len = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.pkv_contiguous_attn_decode(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        context_lens.data_ptr(), cap, S, Hq, Hkv, D, float(scale), _DTYPE_CODE[dtype],
        int(partition_size), ws_ptr, ws_len, _stream_handle(q.device))
    _lib.check(st, "pkv_contiguous_attn_decode")
    return out


def kv_append(k, v, k_cache, v_cache, slot_mapping):
    """Scatter token t's K/V ([T, Hkv, D]) into slot ``slot_mapping[t]`` (int64;
    negative = skip) of both caches."""
    _cuda(k, "k", ndim=3)
    dtype = k.dtype
    if dtype not in _DTYPE_CODE:
        raise ValueError("k must be float16 or bfloat16")
    _cuda(v, "v", dtype, 3)
    _cuda(k_cache, "k_cache", dtype, 4)
    _cuda(v_cache, "v_cache", dtype, 4)
    _cuda(slot_mapping, "slot_mapping", torch.int64, 1)
    T, Hkv, D = k.shape
    NB, Hkv2, B, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or Hkv2 != Hkv or D2 != D:
        raise ValueError("shape mismatch between new tokens and the caches")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    st = _lib.load().pkv_kv_append(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slot_mapping.data_ptr(), T, Hkv, D, B, NB, _DTYPE_CODE[dtype], _stream_handle(k.device))
    _lib.check(st, "pkv_kv_append")


def check_copy_pairs(pairs, num_blocks):
    """Raise ValueError unless ``pairs`` ([P, 2] ids, host data) is a valid
    block_copy batch: ids in [0, num_blocks), destinations distinct, and no
    destination also a source (the pairs are copied in parallel)."""
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    if pairs.size and (pairs.min() < 0 or pairs.max() >= num_blocks):
        raise ValueError("block id outside [0, num_blocks)")
    dst = pairs[:, 1]
    if len(np.unique(dst)) != len(dst):
        raise ValueError("destinations must be distinct")
    if np.intersect1d(dst, pairs[:, 0]).size:
        raise ValueError("a destination is also a source")


def block_copy(k_cache, v_cache, src_dst_pairs, validate=False):
    """Copy whole physical blocks ``src -> dst`` (int64 [P, 2] CUDA tensor) in
    both caches.  ``validate=True`` reads the pairs back to the host and
    checks them first (see check_copy_pairs; this synchronises)."""
    _cuda(k_cache, "k_cache", ndim=4)
    _cuda(v_cache, "v_cache", k_cache.dtype, 4)
    _cuda(src_dst_pairs, "src_dst_pairs", torch.int64)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    if src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [P, 2]")
    NB = k_cache.shape[0]
    if validate:
        check_copy_pairs(src_dst_pairs.cpu().numpy(), NB)
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    st = _lib.load().pkv_block_copy(
        k_cache.data_ptr(), v_cache.data_ptr(), src_dst_pairs.data_ptr(),
        src_dst_pairs.shape[0], NB, block_bytes, _stream_handle(k_cache.device))
    _lib.check(st, "pkv_block_copy")


def debug_wait_timeout(device=None):
    """Enqueue one kernel whose bounded wait cannot complete: after the wait
    limit (2 s) it raises PKV_DEV_WAIT_TIMEOUT and ends (a check of the
    kernels' timeout path; the context stays usable)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _lib.check(_lib.load().pkv_debug_wait_timeout(_stream_handle(dev)), "pkv_debug_wait_timeout")


def device_status(clear=False, device=None):
    """Synchronise the current stream and return the device status flags."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    flags = ctypes.c_uint32(0)
    st = _lib.load().pkv_device_status(ctypes.byref(flags), 1 if clear else 0,
                                       _stream_handle(dev))
    _lib.check(st, "pkv_device_status")
    return flags.value
