"""Fused FP16 attention for one GB300 (sm_103a): Python binding of libgbattn.

The CUDA library (``libgbattn.so``, built in-tree from ``csrc/`` by
``build.py``) does all the work; this module only marshals arguments.  PyTorch
supplies device memory and the current CUDA stream.  Every function has the
name of the C entry point it calls (see ``include/gbattn.h``) and raises
``GbattnError`` when that call returns a non-zero status.  There is no CPU
path: if the library is missing, the first call raises.

The library is loaded lazily, so the seeded input generators in ``inputs``
can be imported on a machine without a GPU.
"""

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgbattn.so")

_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "gbattn_version": (_i, []),
    "gbattn_status_string": (ctypes.c_char_p, [_i]),
    "gbattn_device_status": (_i, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "gbattn_set_wait_limit_ns": (_i, [ctypes.c_uint64]),
    "gbattn_launch_count": (ctypes.c_uint64, []),
    "gbattn_test_inject_fault": (_i, [_i]),
    "attn_dense_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _f, _vp]),
    "attn_dense_mask_fwd": (_i, [_vp, _vp, _vp, _vp, ctypes.c_longlong, ctypes.c_longlong, _vp, _vp,
                                 _i, _i, _i, _i, _i, _f, _vp]),
    "attn_causal_prefill_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "attn_causal_prefill_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                     _vp, _f, _i, _vp, _sz, _vp]),
    "e4m3_paged_to_fp16": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _vp, _vp, _vp]),
    "attn_causal_prefill_paged_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                           _i, _i, _i, _i, _f, _f, _f, _i, _vp, _sz, _vp]),
    "attn_paged_decode_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "attn_paged_decode_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                   _i, _i, _f, _f, _f, _vp, _sz, _vp]),
    "vsa_select_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "vsa_select_blocks": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "vsa_sparse_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                            _i, _i, _f, _vp, _sz, _vp]),
    "vsa_sparse_workspace_size": (_sz, []),
    "vsa_select_coarse_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "vsa_select_blocks_coarse": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _f, _vp, _vp,
                                      _vp, _sz, _vp]),
    "vsa_pair_workspace_size": (_sz, [_i, _i, _i]),
    "vsa_pair_query_cubes": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
}

PROB_SPLIT = 1          # flags of the causal prefill calls (GBATTN_PROB_SPLIT)

DEV_WAIT_TIMEOUT = 1
DEV_BAD_PAGE = 2
DEV_BAD_INDEX = 4
DEV_BAD_LENGTH = 8


class GbattnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def load():
    """Load libgbattn.so (once) and declare its C signatures."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status):
    return load().gbattn_status_string(int(status)).decode()


def _check(fn, rc):
    if rc != 0:
        raise GbattnError(fn, rc)


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _need_view(t, name, dtype):
    """A [B, H, S, D] CUDA view whose last dimension is contiguous (any other strides)."""
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError(f"{name} must be a 4-D view with a contiguous last dimension")


def _strides(t):
    """{batch, head, row} element strides of a [B, H, S, D] view, or None when dense."""
    if t.is_contiguous():
        return None
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def _scale(scale, D):
    return float(1.0 / D ** 0.5) if scale is None else float(scale)


def version():
    return load().gbattn_version()


def launch_count():
    """Kernels launched by the library since it was loaded."""
    return int(load().gbattn_launch_count())


def set_wait_limit_ns(ns):
    _check("gbattn_set_wait_limit_ns", load().gbattn_set_wait_limit_ns(int(ns)))


def test_inject_fault(mode):
    """Test hook: 1 makes attention launches skip their query load, 2 stops their K/V loads
    after two rounds of the ring (timeout paths, mid-stream for 2); 0 restores."""
    _check("gbattn_test_inject_fault", load().gbattn_test_inject_fault(int(mode)))


def device_status(stream=None):
    """Read and clear the device status word (gbattn_device_flag bits)."""
    out = ctypes.c_uint32(0)
    _check("gbattn_device_status", load().gbattn_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def attn_dense_fwd(q, k, v, o=None, lse=None, scale=None, stream=None):
    """Dense non-causal attention. q [B,H,Sq,D], k/v [B,H,Skv,D] FP16 -> o [B,H,Sq,D].

    q, k, v and o may be strided views with a contiguous last dimension (e.g. the
    slices of a packed [B,S,3,H,D] QKV tensor, permuted to [B,H,S,D]); k and v
    must share their strides."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_view(t, n, torch.float16)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if tuple(k.shape) != (B, H, Skv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, H, Skv, D] matching q")
    if k.stride() != v.stride():
        raise ValueError("k and v must have the same strides")
    o = torch.empty((B, H, Sq, D), dtype=torch.float16, device=q.device) if o is None else o
    _need_view(o, "o", torch.float16)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    rc = load().attn_dense_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Sq, Skv, D,
                               _strides(q), _strides(k), _strides(o), _scale(scale, D),
                               _stream(stream))
    _check("attn_dense_fwd", rc)
    return o


def attn_dense_mask_fwd(q, k, v, mask, o=None, lse=None, scale=None, stream=None):
    """Dense attention with an additive FP16 mask broadcastable to [B,H,Sq,Skv]
    (rows of Skv contiguous; a size-1 batch or head dimension is shared)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.float16, 4)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if tuple(k.shape) != (B, H, Skv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, H, Skv, D] matching q")
    if not isinstance(mask, torch.Tensor) or not mask.is_cuda or mask.dtype != torch.float16:
        raise ValueError("mask must be a CUDA float16 tensor")
    m4 = mask.reshape((1, 1) + tuple(mask.shape)) if mask.dim() == 2 else mask
    if m4.dim() != 4 or tuple(m4.shape[2:]) != (Sq, Skv) or m4.shape[0] not in (1, B) \
            or m4.shape[1] not in (1, H):
        raise ValueError("mask must broadcast to [B, H, Sq, Skv]")
    if m4.stride(3) != 1 or m4.stride(2) != Skv:
        raise ValueError("mask rows must be contiguous [Sq][Skv]")
    sb = m4.stride(0) if m4.shape[0] > 1 else 0
    sh = m4.stride(1) if m4.shape[1] > 1 else 0
    o = torch.empty_like(q) if o is None else o
    _need(o, "o", torch.float16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    rc = load().attn_dense_mask_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(m4), sb, sh, _ptr(o), _ptr(lse),
                                    B, H, Sq, Skv, D, _scale(scale, D), _stream(stream))
    _check("attn_dense_mask_fwd", rc)
    return o


def attn_causal_prefill_workspace_size(B, Hq, Q_pad, KV, D):
    return int(load().attn_causal_prefill_workspace_size(B, Hq, Q_pad, KV, D))


def attn_causal_prefill_fwd(q, k, v, q_real=None, o=None, lse=None, scale=None, workspace=None,
                            prob_split=False, stream=None):
    """Causal prefill with shared-KV heads. q [B,Hq,Q_pad,D], k/v [B,Hkv,KV,D] FP16.

    Strided views with a contiguous last dimension are accepted as for
    attn_dense_fwd.  prob_split=True carries the probabilities into the PV
    product as FP16 hi + lo (GBATTN_PROB_SPLIT)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_view(t, n, torch.float16)
    B, Hq, Qp, D = q.shape
    Hkv, KV = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, KV, D] matching q")
    if k.stride() != v.stride():
        raise ValueError("k and v must have the same strides")
    q_real = Qp if q_real is None else int(q_real)
    o = torch.empty((B, Hq, Qp, D), dtype=torch.float16, device=q.device) if o is None else o
    _need_view(o, "o", torch.float16)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    if workspace is None:
        nbytes = attn_causal_prefill_workspace_size(B, Hq, Qp, KV, D)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    rc = load().attn_causal_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                        Qp, q_real, KV, D, _strides(q), _strides(k), _strides(o),
                                        _scale(scale, D), PROB_SPLIT if prob_split else 0,
                                        _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream))
    _check("attn_causal_prefill_fwd", rc)
    return o


def attn_causal_prefill_paged_fwd(q, k_pages, v_pages, page_table, kv_len, k_scale, v_scale,
                                  q_real=None, o=None, lse=None, scale=None, workspace=None,
                                  prob_split=False, stream=None):
    """Causal prefill over paged E4M3 K/V (the bridge fused in).  q [B,Hq,Q_pad,D] FP16;
    pages [P,page,Hkv,D] uint8; page_table int32 [B,max_pages] (or [max_pages] for B=1)."""
    import torch
    _need(q, "q", torch.float16, 4)
    _need(k_pages, "k_pages", torch.uint8, 4)
    _need(v_pages, "v_pages", torch.uint8, 4)
    B, Hq, Qp, D = q.shape
    table = page_table.reshape(1, -1) if page_table.dim() == 1 else page_table
    _need(table, "page_table", torch.int32, 2)
    if table.shape[0] != B:
        raise ValueError("page_table needs one row per batch entry")
    P, ps, Hkv, Dk = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or Dk != D:
        raise ValueError("k_pages and v_pages must be [P, page, Hkv, D] matching q")
    q_real = Qp if q_real is None else int(q_real)
    o = torch.empty_like(q) if o is None else o
    _need(o, "o", torch.float16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    if workspace is None:
        nbytes = attn_causal_prefill_workspace_size(B, Hq, Qp, int(kv_len), D)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    rc = load().attn_causal_prefill_paged_fwd(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(table), _ptr(o), _ptr(lse), B, Hq, Hkv, Qp,
        q_real, int(kv_len), D, P, ps, table.shape[1], float(k_scale), float(v_scale),
        _scale(scale, D), PROB_SPLIT if prob_split else 0, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("attn_causal_prefill_paged_fwd", rc)
    return o


def e4m3_paged_to_fp16(k_pages, v_pages, page_table, kv_len, k_scale, v_scale, k_out=None,
                       v_out=None, stream=None):
    """Paged E4M3 bytes [P, page, Hkv, D] -> FP16 [Hkv, kv_len, D] for K and V."""
    import torch
    _need(k_pages, "k_pages", torch.uint8, 4)
    _need(v_pages, "v_pages", torch.uint8, 4)
    _need(page_table, "page_table", torch.int32, 1)
    P, ps, Hkv, D = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages and v_pages must have the same shape")
    if k_out is None:
        k_out = torch.empty((Hkv, kv_len, D), dtype=torch.float16, device=k_pages.device)
    if v_out is None:
        v_out = torch.empty((Hkv, kv_len, D), dtype=torch.float16, device=k_pages.device)
    _need(k_out, "k_out", torch.float16)
    _need(v_out, "v_out", torch.float16)
    rc = load().e4m3_paged_to_fp16(_ptr(k_pages), _ptr(v_pages), _ptr(page_table), P, ps,
                                   int(kv_len), Hkv, D, float(k_scale), float(v_scale),
                                   _ptr(k_out), _ptr(v_out), _stream(stream))
    _check("e4m3_paged_to_fp16", rc)
    return k_out, v_out


def attn_paged_decode_workspace_size(B, Hq, Hkv, nq, max_kv_len, D):
    return int(load().attn_paged_decode_workspace_size(B, Hq, Hkv, nq, max_kv_len, D))


def attn_paged_decode_fwd(q, k_pages, v_pages, page_table, kv_lens, k_scale, v_scale,
                          max_kv_len=None, o=None, lse=None, scale=None, workspace=None,
                          stream=None):
    """Decode over paged E4M3 caches. q [B,Hq,nq,D] FP16; pages [P,page,Hkv,D] uint8;
    page_table int32 [B,max_pages]; kv_lens int32 [B] (device).  max_kv_len defaults to
    max_pages * page_size (no device read)."""
    import torch
    _need(q, "q", torch.float16, 4)
    _need(k_pages, "k_pages", torch.uint8, 4)
    _need(v_pages, "v_pages", torch.uint8, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    B, Hq, nq, D = q.shape
    P, ps, Hkv, Dk = k_pages.shape
    if tuple(v_pages.shape) != tuple(k_pages.shape) or Dk != D:
        raise ValueError("k_pages and v_pages must be [P, page, Hkv, D] matching q")
    if page_table.shape[0] != B or kv_lens.shape[0] != B:
        raise ValueError("page_table and kv_lens need one row per sequence")
    max_pages = page_table.shape[1]
    max_kv_len = max_pages * ps if max_kv_len is None else int(max_kv_len)
    o = torch.empty_like(q) if o is None else o
    _need(o, "o", torch.float16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    if workspace is None:
        nbytes = attn_paged_decode_workspace_size(B, Hq, Hkv, nq, max_kv_len, D)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    rc = load().attn_paged_decode_fwd(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                      _ptr(kv_lens), _ptr(o), _ptr(lse), B, Hq, Hkv, nq, D, P,
                                      ps, max_pages, max_kv_len, float(k_scale), float(v_scale),
                                      _scale(scale, D), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(stream))
    _check("attn_paged_decode_fwd", rc)
    return o


def vsa_select_workspace_size(B, H, S, D, block):
    return int(load().vsa_select_workspace_size(B, H, S, D, block))


def vsa_select_blocks(q, k, topk, block=64, prefix=0, cube_valid=None, idx=None, workspace=None,
                      stream=None):
    """Top-k key cubes per query cube.  q, k [B,H,S,D] FP16: `prefix` prefix tokens, then
    cube-major video tokens; cube_valid int32 [cubes] real tokens per cube (None: full).
    Returns idx int32 [B,H,(S-prefix)/block,topk]."""
    import torch
    _need(q, "q", torch.float16, 4)
    _need(k, "k", torch.float16, 4)
    B, H, S, D = q.shape
    if tuple(k.shape) != tuple(q.shape):
        raise ValueError("q and k must have the same shape")
    nc = (S - int(prefix)) // block
    if cube_valid is not None:
        _need(cube_valid, "cube_valid", torch.int32, 1)
    if idx is None:
        idx = torch.empty((B, H, nc, topk), dtype=torch.int32, device=q.device)
    _need(idx, "idx", torch.int32)
    if workspace is None:
        workspace = torch.empty(max(vsa_select_workspace_size(B, H, S, D, block), 16),
                                dtype=torch.uint8, device=q.device)
    rc = load().vsa_select_blocks(_ptr(q), _ptr(k), B, H, S, D, block, int(topk), int(prefix),
                                  _ptr(cube_valid), _ptr(idx), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check("vsa_select_blocks", rc)
    return idx


def vsa_select_coarse_workspace_size(B, H, S, D, block=64):
    return int(load().vsa_select_coarse_workspace_size(B, H, S, D, block))


def vsa_select_blocks_coarse(q, k, v, topk, block=64, prefix=0, cube_valid=None, scale=None,
                             idx=None, coarse=None, workspace=None, stream=None):
    """The selection plus the coarse branch: returns (idx int32 [B,H,cubes,topk], coarse FP32
    [B,H,cubes,D]), coarse[i] = softmax over all key cubes of scale * pooled q_i . pooled k_j,
    times the pooled values."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.float16, 4)
    B, H, S, D = q.shape
    if tuple(k.shape) != tuple(q.shape) or tuple(v.shape) != tuple(q.shape):
        raise ValueError("q, k and v must have the same shape")
    nc = (S - int(prefix)) // block
    if cube_valid is not None:
        _need(cube_valid, "cube_valid", torch.int32, 1)
    if idx is None:
        idx = torch.empty((B, H, nc, topk), dtype=torch.int32, device=q.device)
    if coarse is None:
        coarse = torch.empty((B, H, nc, D), dtype=torch.float32, device=q.device)
    _need(idx, "idx", torch.int32)
    _need(coarse, "coarse", torch.float32)
    if workspace is None:
        workspace = torch.empty(max(vsa_select_coarse_workspace_size(B, H, S, D, block), 16),
                                dtype=torch.uint8, device=q.device)
    rc = load().vsa_select_blocks_coarse(_ptr(q), _ptr(k), _ptr(v), B, H, S, D, block, int(topk),
                                         int(prefix), _ptr(cube_valid), _scale(scale, D), _ptr(idx),
                                         _ptr(coarse), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream))
    _check("vsa_select_blocks_coarse", rc)
    return idx, coarse


def vsa_pair_query_cubes(idx, pairs=None, workspace=None, stream=None):
    """Query-cube pairs for vsa_sparse_fwd.  idx int32 [B,H,cubes,topk] ->
    pairs int32 [B,H,ceil(cubes/2),2] (second entry -1 for a lone cube), greedy by selection
    overlap, longest union first.  workspace: vsa_pair_workspace_size bytes (allocated here
    when None)."""
    import torch
    _need(idx, "idx", torch.int32, 4)
    B, H, nc, topk = idx.shape
    if pairs is None:
        pairs = torch.empty((B, H, (nc + 1) // 2, 2), dtype=torch.int32, device=idx.device)
    _need(pairs, "pairs", torch.int32)
    if workspace is None:
        workspace = torch.empty(int(load().vsa_pair_workspace_size(B, H, nc)), dtype=torch.uint8,
                                device=idx.device)
    rc = load().vsa_pair_query_cubes(_ptr(idx), B, H, nc, topk, _ptr(pairs), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check("vsa_pair_query_cubes", rc)
    return pairs


_SPARSE_COUNTERS = {}


def sparse_counter(stream=None):
    """The item counter vsa_sparse_fwd uses on `stream` (default: the current stream) when
    it is given no workspace: zeroed device bytes, one buffer per stream, which every call
    leaves at zero.  Calls on one stream run one after another, so they can share it; a
    caller that replays a captured graph on another stream while that stream is busy
    passes its own workspace instead."""
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    key = (s.device.index if s.device.index is not None else torch.cuda.current_device(),
           s.cuda_stream)
    buf = _SPARSE_COUNTERS.get(key)
    if buf is None:
        n = int(load().vsa_sparse_workspace_size())
        buf = torch.zeros(n, dtype=torch.uint8, device=s.device)
        torch.cuda.synchronize(s.device)
        _SPARSE_COUNTERS[key] = buf
    return buf


def vsa_sparse_fwd(q, k, v, idx, block=64, prefix=0, cube_valid=None, pairs=None, o=None,
                   lse=None, scale=None, coarse=None, gate=None, workspace=None, stream=None):
    """Block-sparse attention over the cubes in idx.  q/k/v [B,H,S,D] FP16: `prefix` dense
    prefix tokens, then cube-major video tokens; cube_valid int32 [cubes] or None; pairs from
    vsa_pair_query_cubes or None (adjacent cubes).  coarse (FP32 [B,H,cubes,D] from
    vsa_select_blocks_coarse) and gate (FP16 [B,H,S,D]) add gate * coarse[cube] to every real
    video token's output.  workspace: the item counter (zeroed, left zero by every call);
    None takes this stream's (sparse_counter), False splits the items statically."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.float16, 4)
    _need(idx, "idx", torch.int32, 4)
    if cube_valid is not None:
        _need(cube_valid, "cube_valid", torch.int32, 1)
    if pairs is not None:
        _need(pairs, "pairs", torch.int32, 4)
    B, H, S, D = q.shape
    topk = idx.shape[3]
    if (coarse is None) != (gate is None):
        raise ValueError("coarse and gate go together")
    if coarse is not None:
        _need(coarse, "coarse", torch.float32, 4)
        _need(gate, "gate", torch.float16, 4)
    o = torch.empty_like(q) if o is None else o
    _need(o, "o", torch.float16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    if workspace is None:
        workspace = sparse_counter(stream)
    ws = None if workspace is False else workspace
    rc = load().vsa_sparse_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(pairs), int(prefix),
                               _ptr(cube_valid), _ptr(coarse), _ptr(gate),
                               _ptr(o), _ptr(lse), B, H, S, D, block, topk, _scale(scale, D),
                               _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                               _stream(stream))
    _check("vsa_sparse_fwd", rc)
    return o
