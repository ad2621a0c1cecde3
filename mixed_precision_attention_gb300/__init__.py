"""Adaptive-precision causal attention prefill with GQA packing for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libapa.so`` (``include/apa.h``): it
checks and marshals arguments; every step of the computation runs in the
library's CUDA kernels.  PyTorch is used for device memory and the current
stream only.  There is no CPU fallback: without the built library (see
``mixed_precision_attention_gb300.build``) every compute call raises.

Method: "APA: sloppy attention, exact where it counts" (rfriedmann.de blog).
Pass 1 computes every 64-key tile in block-scaled NVFP4 and flags the tiles
whose FP4 softmax mass exceeds eps times a row's running sum; pass 2 recomputes
those exactly in BF16; the two states are merged exactly by log-sum-exp.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import ApaError, status_string

__all__ = ["attention", "attention_paged", "attention_host", "quantize", "quantize_noalloc", "workspace_bytes",
           "workspace_operands", "check_error", "ApaError",
           "status_string", "hot_mask_shape", "TILE", "GROUP_ROWS", "BLOCK_ROWS", "FLAG_Q_RESIDUAL",
           "FLAG_LSE_SCALES", "FLAG_VALUE_WEIGHTED", "FLAG_ROWSUM_MMA"]

FLAG_Q_RESIDUAL = 1  # APA_FLAG_Q_RESIDUAL: Q as two FP4 terms in pass 1
FLAG_LSE_SCALES = 2  # APA_FLAG_LSE_SCALES: least-squared-error block scales for Q, K, V
FLAG_VALUE_WEIGHTED = 4  # APA_FLAG_VALUE_WEIGHTED: hot test weighted by value norm
FLAG_ROWSUM_MMA = 8  # APA_FLAG_ROWSUM_MMA: pass-1 row sums from an MMA against an E2M1 ones tile
TILE = 64          # keys per tile
GROUP_ROWS = 16    # rows per hot-test group
BLOCK_ROWS = 128   # GQA-packed rows per CTA


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(device):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def hot_mask_shape(B, Hq, Hkv, Nq, Nkv):
    G = Hq // Hkv
    ng = (G * Nq + GROUP_ROWS - 1) // GROUP_ROWS
    T = (Nkv + TILE - 1) // TILE
    return (B, Hkv, ng, (T + 31) // 32)


def _check_qkv(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4:
            raise TypeError(f"{name} must be a 4-D torch.bfloat16 tensor (BHSD)")
        if not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Hq, Nq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, Nkv, d] with q's B and d")
    return B, Hq, k.shape[1], Nq, k.shape[2], d


def _flags(q_residual=False, lse_scales=False, value_weighted=False, rowsum_mma=False):
    return ((FLAG_Q_RESIDUAL if q_residual else 0) | (FLAG_LSE_SCALES if lse_scales else 0)
            | (FLAG_VALUE_WEIGHTED if value_weighted else 0) | (FLAG_ROWSUM_MMA if rowsum_mma else 0))


def workspace_bytes(B, Hq, Hkv, Nq, Nkv, d, eps, q_residual: bool = False, value_weighted: bool = False):
    flags = _flags(q_residual, value_weighted=value_weighted)
    return int(_lib.load().apa_workspace_bytes_ex(B, Hq, Hkv, Nq, Nkv, d, float(eps), flags))


def workspace_operands(B, Hq, Hkv, Nq, Nkv, d, eps, q_residual: bool = False, value_weighted: bool = False,
                       rowsum_mma: bool = False):
    """apa_workspace_operands: byte offsets, inside the workspace of an eps > 0
    call with these options, of the pass-1 operands the call leaves there.
    Returns dict(kv_blob, q_blob, mu, s_q, s_k, s_v) of offsets."""
    lib = _lib.load()
    offs = [ctypes.c_size_t() for _ in range(6)]
    st = lib.apa_workspace_operands(B, Hq, Hkv, Nq, Nkv, d, float(eps),
                                    _flags(q_residual, value_weighted=value_weighted, rowsum_mma=rowsum_mma),
                                    *[ctypes.byref(o) for o in offs])
    _lib.check(st, "apa_workspace_operands")
    return dict(zip(("kv_blob", "q_blob", "mu", "s_q", "s_k", "s_v"), (o.value for o in offs)))


def attention(q, k, v, causal: bool = True, eps: float = 0.005, return_hot_mask: bool = False,
              return_lse: bool = True, workspace=None, q_residual: bool = False, lse_scales: bool = False,
              value_weighted: bool = False, rowsum_mma: bool = False):
    """Adaptive-precision attention.

    q: [B, Hq, Nq, d] bf16; k, v: [B, Hkv, Nkv, d] bf16 (CUDA, contiguous).
    causal: tail-aligned causal mask (query row i sees keys j <= i + Nkv - Nq).
    eps: hot-test threshold; 0 = every visible tile exact (BF16), inf = all FP4.
    Returns (out fp32 [B,Hq,Nq,d], lse fp32 [B,Hq,Nq] or None, hot_mask or None);
    hot_mask is int32 [B, Hkv, ceil(G*Nq/16), ceil(T/32)] holding uint32 bit
    words (bit t%32 of word t/32: tile t hot for that 16-row group).
    workspace: optional uint8 CUDA tensor of at least workspace_bytes(...) bytes.
    q_residual: Q as two FP4 terms in pass 1 (apa_attention_ex, APA_FLAG_Q_RESIDUAL).
    lse_scales: least-squared-error block scales for Q, K, V (APA_FLAG_LSE_SCALES).
    value_weighted: hot test weighted by the tile's value norm (APA_FLAG_VALUE_WEIGHTED).
    rowsum_mma: pass-1 tile row sums from an MMA against an E2M1 ones tile (APA_FLAG_ROWSUM_MMA).
    """
    import torch
    lib = _lib.load()
    B, Hq, Hkv, Nq, Nkv, d = _check_qkv(q, k, v)
    dev = q.device
    out = torch.empty((B, Hq, Nq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev) if return_lse else None
    mask = torch.empty(hot_mask_shape(B, Hq, Hkv, Nq, Nkv), dtype=torch.int32, device=dev) if return_hot_mask else None
    need = workspace_bytes(B, Hq, Hkv, Nq, Nkv, d, eps, q_residual, value_weighted)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    nbytes = 0 if workspace is None else workspace.numel()
    flags = _flags(q_residual, lse_scales, value_weighted, rowsum_mma)
    if flags:
        st = lib.apa_attention_ex(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)), float(eps),
                                  flags, _ptr(out), _ptr(lse), _ptr(mask), _ptr(workspace),
                                  nbytes, _stream(dev))
        _lib.check(st, "apa_attention_ex")
    else:
        st = lib.apa_attention_ws(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)), float(eps),
                                  _ptr(out), _ptr(lse), _ptr(mask), _ptr(workspace), nbytes, _stream(dev))
        _lib.check(st, "apa_attention_ws")
    return out, lse, mask


def attention_paged(q, k_pages, v_pages, block_table, Nkv: int, causal: bool = True, eps: float = 0.005,
                    return_hot_mask: bool = False, return_lse: bool = True):
    """apa_attention_paged: attention over a paged K/V cache.

    q: [B, Hq, Nq, d] bf16; k_pages, v_pages: [num_pages, Hkv, 64, d] bf16 (one page
    = one 64-key tile of one sequence, all KV heads); block_table: int32 CUDA tensor
    [B, max_pages], entry t of sequence b = the page holding its keys 64t..64t+63;
    Nkv: keys per sequence.  Returns (out, lse or None, hot_mask or None) as attention()."""
    import torch
    lib = _lib.load()
    for name, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_cuda \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    if k_pages.shape != v_pages.shape or k_pages.shape[2] != TILE or k_pages.shape[3] != q.shape[3]:
        raise ValueError("k_pages and v_pages must be [num_pages, Hkv, 64, d] with q's d")
    if (not isinstance(block_table, torch.Tensor) or block_table.dtype != torch.int32 or block_table.dim() != 2
            or not block_table.is_cuda or not block_table.is_contiguous() or block_table.shape[0] != q.shape[0]):
        raise ValueError("block_table must be a contiguous int32 CUDA tensor [B, max_pages]")
    B, Hq, Nq, d = q.shape
    num_pages, Hkv = k_pages.shape[0], k_pages.shape[1]
    dev = q.device
    out = torch.empty((B, Hq, Nq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev) if return_lse else None
    mask = torch.empty(hot_mask_shape(B, Hq, Hkv, Nq, Nkv), dtype=torch.int32, device=dev) if return_hot_mask else None
    st = lib.apa_attention_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), num_pages, _ptr(block_table),
                                 block_table.shape[1], B, Hq, Hkv, Nq, int(Nkv), d, int(bool(causal)), float(eps),
                                 _ptr(out), _ptr(lse), _ptr(mask), _stream(dev))
    _lib.check(st, "apa_attention_paged")
    return out, lse, mask


def attention_host(q, k, v, causal: bool = True, eps: float = 0.005, return_hot_mask: bool = False, stream=None,
                   out=None, lse=None):
    """apa_attention_host: the same computation on HOST tensors (torch CPU, bf16,
    contiguous; pinned memory recommended).  Copies in, runs, copies out and
    synchronizes the stream.  `out` [B,Hq,Nq,d] and `lse` [B,Hq,Nq] (fp32 CPU,
    contiguous) may be passed in to reuse them; by default they are allocated in
    pinned memory.  Returns CPU tensors (out, lse, hot_mask or None)."""
    import torch
    lib = _lib.load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CPU tensor")
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    for name, t, shape in (("out", out, (B, Hq, Nq, d)), ("lse", lse, (B, Hq, Nq))):
        if t is not None and (t.dtype != torch.float32 or t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape):
            raise ValueError(f"{name} must be a contiguous fp32 CPU tensor of shape {shape}")
    if out is None:
        out = torch.empty((B, Hq, Nq, d), dtype=torch.float32, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=True)
    mask = torch.empty(hot_mask_shape(B, Hq, Hkv, Nq, Nkv), dtype=torch.int32) if return_hot_mask else None
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(None)
    st = lib.apa_attention_host(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)), float(eps),
                                _ptr(out), _ptr(lse), _ptr(mask), s)
    _lib.check(st, "apa_attention_host")
    return out, lse, mask


def quantize(q, k, v, q_residual: bool = False, lse_scales: bool = False):
    """The pass-1 NVFP4 operands (apa_quantize_ex): dict of CUDA tensors
    kv_blob, q_blob (uint8), mu [B,Hkv,d], s_q [B,Hq], s_k, s_v [B,Hkv] (fp32);
    with q_residual also q2_blob (uint8, q_blob's layout), the FP4 residual of Q;
    lse_scales: least-squared-error block scales."""
    import torch
    lib = _lib.load()
    B, Hq, Hkv, Nq, Nkv, d = _check_qkv(q, k, v)
    dev = q.device
    r = dict(kv_blob=torch.empty(lib.apa_kv_blob_bytes(B, Hkv, Nkv, d), dtype=torch.uint8, device=dev),
             q_blob=torch.empty(lib.apa_q_blob_bytes(B, Hq, Hkv, Nq, d), dtype=torch.uint8, device=dev),
             mu=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev),
             s_q=torch.empty((B, Hq), dtype=torch.float32, device=dev),
             s_k=torch.empty((B, Hkv), dtype=torch.float32, device=dev),
             s_v=torch.empty((B, Hkv), dtype=torch.float32, device=dev))
    if q_residual:
        r["q2_blob"] = torch.empty_like(r["q_blob"])
    st = lib.apa_quantize_ex(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, _flags(q_residual, lse_scales),
                             _ptr(r["kv_blob"]),
                             _ptr(r["q_blob"]), _ptr(r.get("q2_blob")), _ptr(r["mu"]), _ptr(r["s_q"]), _ptr(r["s_k"]),
                             _ptr(r["s_v"]), _stream(dev))
    _lib.check(st, "apa_quantize_ex")
    return r


def quantize_noalloc(q, k, v, out=None):
    """quantize() through apa_quantize_noalloc, for callers that cannot allocate
    device memory during the call: the library keeps the temporary statistics in
    a fixed 16 MiB device array.  Pass `out` (a dict shaped like quantize()'s
    result) to write into existing buffers; without it the outputs are allocated
    here, before the call.  Raises ApaError(APA_ERR_SCRATCH) when the problem's
    statistics do not fit the fixed array."""
    lib = _lib.load()
    B, Hq, Hkv, Nq, Nkv, d = _check_qkv(q, k, v)
    r = out
    if r is None:
        import torch
        dev = q.device
        r = dict(kv_blob=torch.empty(lib.apa_kv_blob_bytes(B, Hkv, Nkv, d), dtype=torch.uint8, device=dev),
                 q_blob=torch.empty(lib.apa_q_blob_bytes(B, Hq, Hkv, Nq, d), dtype=torch.uint8, device=dev),
                 mu=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev),
                 s_q=torch.empty((B, Hq), dtype=torch.float32, device=dev),
                 s_k=torch.empty((B, Hkv), dtype=torch.float32, device=dev),
                 s_v=torch.empty((B, Hkv), dtype=torch.float32, device=dev))
    st = lib.apa_quantize_noalloc(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, _ptr(r["kv_blob"]),
                                  _ptr(r["q_blob"]), _ptr(r["mu"]), _ptr(r["s_q"]), _ptr(r["s_k"]),
                                  _ptr(r["s_v"]), _stream(q.device))
    _lib.check(st, "apa_quantize_noalloc")
    return r


def check_error(device=None):
    """Synchronizes the current stream and raises if a kernel recorded a device-side timeout."""
    _lib.check(_lib.load().apa_check_error(_stream(device)), "apa_check_error")
