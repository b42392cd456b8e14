"""The C-ABI library builds, loads and rejects bad arguments (CPU only).

Every function declared in include/gbattn.h must be exported by
libgbattn.so.  Argument validation runs before any CUDA call, so the error
paths can be exercised on a machine without a GPU; with valid arguments and
no device the calls return GBATTN_ERR_CUDA instead of crashing.
"""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")

OK, NULL, SHAPE, UNSUPPORTED, ALIGN, ALIAS, WORKSPACE, CUDA, SCALE = range(9)


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    # Calls with valid-looking arguments reach the launch stage; they pass
    # placeholder addresses, so they must only run where no GPU is visible.
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only validation tests: they run where no GPU is visible")
    from attention_fp16_flashattention_gb300 import build
    build.build()
    import attention_fp16_flashattention_gb300 as gb
    return gb.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", text)) - {"if", "sizeof"})


def test_header_declares_the_five_entry_points():
    names = _declared_functions()
    for n in ("attn_dense_fwd", "attn_causal_prefill_fwd", "e4m3_paged_to_fp16",
              "vsa_select_blocks", "vsa_sparse_fwd"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.gbattn_version() >= 100
    for s in range(9):
        assert lib.gbattn_status_string(s)
    assert lib.gbattn_status_string(99) == b"unknown status"


def test_fault_hook_modes(lib):
    """The test hook takes modes 0..2 only (host-side state; nothing is launched)."""
    for mode in (1, 2, 0):
        assert lib.gbattn_test_inject_fault(mode) == 0
    assert lib.gbattn_test_inject_fault(3) == 2 and lib.gbattn_test_inject_fault(-1) == 2


P = ctypes.c_void_p(0x10000)      # aligned fake device addresses: never dereferenced
P2 = ctypes.c_void_p(0x20000000)
P3 = ctypes.c_void_p(0x40000000)
P4 = ctypes.c_void_p(0x60000000)
MIS = ctypes.c_void_p(0x10008)    # 8-byte aligned only
MIS2 = ctypes.c_void_p(0x10002)   # not 4-byte aligned


def _st(*v):
    return (ctypes.c_int64 * 3)(*v)


def test_dense_validation(lib):
    f = lib.attn_dense_fwd
    # q, k, v, o, lse, B, H, Sq, Skv, D, q_strides, kv_strides, o_strides, scale, stream
    N = None
    assert f(None, P2, P3, P4, None, 1, 1, 128, 128, 128, N, N, N, 0.1, None) == NULL
    assert f(P, P2, P3, P4, None, 0, 1, 128, 128, 128, N, N, N, 0.1, None) == SHAPE
    assert f(P, P2, P3, P4, None, 1, 1, 128, 128, 64, N, N, N, 0.1, None) == UNSUPPORTED
    assert f(P, P2, P3, P4, None, 1, 1, 128, 128, 128, N, N, N, 0.0, None) == SCALE
    assert f(P, P2, P3, P4, None, 1, 1, 128, 128, 128, N, N, N, float("nan"), None) == SCALE
    assert f(MIS, P2, P3, P4, None, 1, 1, 128, 128, 128, N, N, N, 0.1, None) == ALIGN
    assert f(P, P2, P3, P, None, 1, 1, 128, 128, 128, N, N, N, 0.1, None) == ALIAS
    assert f(P, P2, P3, ctypes.c_void_p(0x10000 + 4096), None, 1, 1, 128, 128, 128, N, N, N, 0.1,
             None) == ALIAS
    assert f(P, P2, P3, P4, None, 256, 256, 128, 128, 128, N, N, N, 0.1, None) == SHAPE
    # strides: {batch, head, row} elements
    packed = _st(3 * 2 * 128 * 128, 128, 3 * 2 * 128)            # [B,S,3,H,D] slice, H=2
    assert f(P, P2, P3, P4, None, 1, 2, 128, 128, 128, packed, packed, N, 0.1, None) in (CUDA, OK)
    assert f(P, P2, P3, P4, None, 1, 2, 128, 128, 128, _st(0, 128 * 128, 100), N, N, 0.1,
             None) == SHAPE                                       # row stride < D
    assert f(P, P2, P3, P4, None, 1, 2, 128, 128, 128, _st(0, 128 * 128, 132), N, N, 0.1,
             None) == SHAPE                                       # not a multiple of 8
    assert f(P, P2, P3, P4, None, 1, 2, 128, 128, 128, N, N, _st(0, 128, 128), 0.1,
             None) == SHAPE                                       # output heads overlap
    assert f(P, P2, P3, P4, None, 1, 2, 128, 128, 128, N, N, _st(0, 128, 256), 0.1,
             None) in (CUDA, OK)                                  # interleaved heads: fine
    assert f(P, P2, P3, P4, None, 1, 2, 128, 128, 128, N, N, _st(0, 0, 256), 0.1,
             None) == SHAPE                                       # zero stride
    # valid arguments, no GPU here -> CUDA error, not a crash
    assert f(P, P2, P3, P4, None, 1, 1, 128, 128, 128, N, N, N, 0.1, None) in (CUDA, OK)


def test_causal_validation(lib):
    f = lib.attn_causal_prefill_fwd
    args = lambda **kw: dict(dict(B=1, Hq=6, Hkv=1, Qp=1024, Qr=1024, KV=4096, D=256, flags=0,
                                  qs=None, os=None), **kw)

    def call(q=P, o=P4, ws=None, wsb=0, **kw):
        a = args(**kw)
        return f(q, P2, P3, o, None, a["B"], a["Hq"], a["Hkv"], a["Qp"], a["Qr"], a["KV"], a["D"],
                 a["qs"], None, a["os"], 0.0625, a["flags"], ws, wsb, None)
    assert call(q=None) == NULL
    assert call(Hq=5, Hkv=2) == SHAPE             # Hq % Hkv
    assert call(Qp=1000, Qr=1000) == SHAPE        # Q_pad % 64
    assert call(Qr=0) == SHAPE
    assert call(Qr=1025) == SHAPE                 # Q_real > Q_pad
    assert call(KV=4020) == SHAPE                 # KV % 32
    assert call(Qp=8192, Qr=8192, KV=4096) == SHAPE   # Q_real > KV
    assert call(D=128) == UNSUPPORTED
    assert call(o=P) == ALIAS
    assert call(flags=2) == SHAPE                 # unknown flag
    assert call(os=_st(0, 256, 256)) == SHAPE     # output heads overlap
    assert call(flags=1) in (CUDA, OK)
    assert call(qs=_st(0, 256, 6 * 256), os=_st(0, 256, 6 * 256)) in (CUDA, OK)   # token-major
    assert call() in (CUDA, OK)


def test_bridge_validation(lib):
    f = lib.e4m3_paged_to_fp16
    base = [P, P2, P3, 4, 32, 100, 1, 256, 0.0625, 0.125, P4, ctypes.c_void_p(0x70000000), None]

    def call(i=None, v=None):
        a = list(base)
        if i is not None:
            a[i] = v
        return f(*a)
    assert call(0, None) == NULL
    assert call(5, 0) == SHAPE
    assert call(7, 24) == UNSUPPORTED
    assert call(8, -1.0) == SCALE
    assert call(9, float("inf")) == SCALE
    assert call(10, MIS) == ALIGN
    assert call(10, P) == ALIAS
    assert call(11, P4) == ALIAS
    assert call() in (CUDA, OK)


def test_dense_mask_validation(lib):
    f = lib.attn_dense_mask_fwd
    # q, k, v, mask, stride_b, stride_h, o, lse, B, H, Sq, Skv, D, scale, stream
    base = [P, P2, P3, ctypes.c_void_p(0x70000000), 0, 0, P4, None, 1, 2, 256, 256, 128, 0.088, None]

    def call(i=None, val=None):
        a = list(base)
        if i is not None:
            a[i] = val
        return f(*a)
    assert call(3, None) == NULL
    assert call(11, 260) == SHAPE              # mask rows must be 16-byte multiples
    assert call(5, 12) == SHAPE                # head stride not a multiple of 8
    assert call(5, 8) == SHAPE                 # head slices overlapping
    assert call(4, -8) == SHAPE
    assert call(12, 64) == UNSUPPORTED
    assert call(13, 0.0) == SCALE
    assert call(3, MIS) == ALIGN
    assert call(6, ctypes.c_void_p(0x70000000)) == ALIAS
    assert call() in (CUDA, OK)


def test_decode_validation(lib):
    f = lib.attn_paged_decode_fwd
    P5, P6 = ctypes.c_void_p(0x70000000), ctypes.c_void_p(0x78000000)
    # q, k_pages, v_pages, page_table, kv_lens, o, lse, B, Hq, Hkv, nq, D, num_phys,
    # page_size, max_pages, max_kv_len, k_scale, v_scale, scale, workspace, bytes, stream
    base = [P, P2, P3, P4, P5, P6, None, 2, 6, 1, 1, 256, 64, 32, 32, 1024, 0.0625, 0.125,
            0.0625, None, 0, None]

    def call(**kw):
        a = list(base)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return f(*a)
    assert call(a0=None) == NULL
    assert call(a4=None) == NULL
    assert call(a7=0) == SHAPE
    assert call(a8=5, a9=2) == SHAPE            # Hq % Hkv
    assert call(a15=1025) == SHAPE              # max_kv_len > max_pages * page_size
    assert call(a10=2000) == SHAPE              # nq > max_kv_len
    assert call(a11=64) == UNSUPPORTED
    assert call(a13=24, a14=64) == UNSUPPORTED  # page size not a power of two
    assert call(a13=8, a14=128) == UNSUPPORTED  # page size below 16
    assert call(a16=0.0) == SCALE
    assert call(a18=float("nan")) == SCALE
    assert call(a5=MIS) == ALIGN
    assert call(a4=ctypes.c_void_p(0x70000002)) == ALIGN
    assert call(a5=P) == ALIAS
    assert call(a6=ctypes.c_void_p(0x78000000)) == ALIAS
    assert call() == WORKSPACE                  # the decode always needs a workspace
    assert call(a19=ctypes.c_void_p(0x7C000000), a20=1 << 24) in (CUDA, OK)
    assert call(a7=5000) == UNSUPPORTED         # more sequences than one launch takes
    assert lib.attn_paged_decode_workspace_size(0, 6, 1, 1, 1024, 256) == 0
    assert lib.attn_paged_decode_workspace_size(2, 6, 1, 1, 1024, 256) > 0


def test_select_and_sparse_validation(lib):
    ws = lib.vsa_select_workspace_size(1, 24, 32768, 128, 64)
    rows = 24 * 512                             # means of Q and K, norms, flags, scores
    assert ws == 2 * rows * 128 * 4 + 3 * rows * 4 + rows * 512 * 4
    f = lib.vsa_select_blocks
    assert f(P, P2, 1, 24, 32768, 128, 64, 64, 0, None, P3, P4, ws - 1, None) == WORKSPACE
    assert f(P, P2, 1, 24, 32768, 128, 32, 64, 0, None, P3, P4, ws, None) == UNSUPPORTED
    assert f(P, P2, 1, 24, 32768, 128, 64, 513, 0, None, P3, P4, ws, None) == SHAPE
    assert f(P, P2, 1, 24, 32768 + 32, 128, 64, 64, 0, None, P3, P4, ws, None) == SHAPE
    assert f(P, P2, 1, 24, 32768 + 32, 128, 64, 64, 32, None, P3, P4, ws, None) in (CUDA, OK)
    assert f(P, P2, 1, 24, 32768, 128, 64, 64, -1, None, P3, P4, ws, None) == SHAPE
    assert f(P, P2, 1, 24, 32768, 128, 64, 64, 0, MIS2, P3, P4, ws, None) == ALIGN
    assert f(P, P2, 1, 24, 32768, 128, 64, 64, 0, None, P3, P4, ws, None) in (CUDA, OK)
    g = lib.vsa_sparse_fwd
    # q, k, v, idx, pairs, prefix, cube_valid, coarse, gate, o, lse, B, H, S, D, block, topk,
    # scale, workspace, workspace_bytes, stream
    I = ctypes.c_void_p(0x70000000)
    N = None
    assert g(P, P2, P3, P4, N, 0, N, N, N, None, None, 1, 24, 32768, 128, 64, 64, 0.08, N, 0, None) == NULL
    assert g(P, P2, P3, I, N, 0, N, N, N, P, None, 1, 24, 32768, 128, 64, 64, 0.08, N, 0, None) == ALIAS
    assert g(P, P2, P3, I, N, 0, N, N, N, P4, None, 1, 24, 32768, 128, 64, 600, 0.08, N, 0, None) == SHAPE
    assert g(P, P2, P3, I, N, 64, N, N, N, P4, None, 1, 24, 32768 + 64, 128, 64, 64, 0.08, N, 0,
             None) == SHAPE                        # prefix must be whole 128-row query tiles
    assert g(P, P2, P3, I, N, 128, MIS2, N, N, P4, None, 1, 24, 32768 + 128, 128, 64, 64, 0.08, N, 0,
             None) == ALIGN
    assert g(P, P2, P3, I, MIS2, 0, N, N, N, P4, None, 1, 24, 32768, 128, 64, 64, 0.08, N, 0, None) == ALIGN
    C = ctypes.c_void_p(0x78000000)
    assert g(P, P2, P3, I, N, 0, N, C, N, P4, None, 1, 24, 32768, 128, 64, 64, 0.08, N, 0,
             None) == NULL                         # coarse without a gate
    assert g(P, P2, P3, I, N, 0, N, C, P4, P4, None, 1, 24, 32768, 128, 64, 64, 0.08, N, 0,
             None) == ALIAS                        # output over the gate
    W = ctypes.c_void_p(0x7C000000)
    assert lib.vsa_sparse_workspace_size() == 16
    assert g(P, P2, P3, I, N, 0, N, N, N, P4, None, 1, 24, 32768, 128, 64, 64, 0.08, W, 15,
             None) == WORKSPACE                    # too small a counter
    assert g(P, P2, P3, I, N, 0, N, N, N, P4, None, 1, 24, 32768, 128, 64, 64, 0.08,
             ctypes.c_void_p(0x7C000004), 16, None) == ALIGN
    assert g(P, P2, P3, I, N, 0, N, N, N, P4, None, 1, 24, 32768, 128, 64, 64, 0.08, P4, 16,
             None) == ALIAS                        # counter inside the output
    assert g(P, P2, P3, I, N, 0, N, N, N, P4, None, 1, 24, 32768, 128, 64, 64, 0.08, I, 16,
             None) == ALIAS                        # counter inside idx
    c = lib.vsa_select_blocks_coarse
    ws = lib.vsa_select_coarse_workspace_size(1, 24, 32768, 128, 64)
    assert ws == lib.vsa_select_workspace_size(1, 24, 32768, 128, 64) + 24 * 512 * 128 * 4
    assert c(P, P2, None, 1, 24, 32768, 128, 64, 64, 0, N, 0.08, P3, C, P4, ws, None) == NULL
    assert c(P, P2, I, 1, 24, 32768, 128, 64, 64, 0, N, 0.0, P3, C, P4, ws, None) == SCALE
    assert c(P, P2, I, 1, 24, 32768, 128, 64, 64, 0, N, 0.08, P3, C, P4, ws - 1, None) == WORKSPACE
    assert c(P, P2, I, 1, 24, 32768, 128, 64, 64, 0, N, 0.08, P3, P, P4, ws, None) == ALIAS
    h = lib.vsa_pair_query_cubes
    pw = lib.vsa_pair_workspace_size(1, 24, 512)
    assert pw == 24 * 512 * 16 * 4 + 24 * 512 * 32 * 2  # bitset rows, 32 int16 candidates per cube
    assert h(None, 1, 24, 512, 64, P4, W, pw, None) == NULL
    assert h(I, 1, 24, 2048, 64, P4, W, pw, None) == SHAPE   # more cubes than the pairing takes
    assert h(I, 1, 24, 512, 600, P4, W, pw, None) == SHAPE
    assert h(I, 1, 24, 512, 64, I, W, pw, None) == ALIAS
    assert h(I, 1, 24, 512, 64, P4, W, pw - 1, None) == WORKSPACE
    assert h(I, 1, 24, 512, 64, P4, None, pw, None) == WORKSPACE
    assert h(I, 1, 24, 512, 64, P4, ctypes.c_void_p(0x7C000008), pw, None) == ALIGN
    assert h(I, 1, 24, 512, 64, P4, P4, pw, None) == ALIAS   # workspace over the pairs
    assert h(I, 1, 24, 512, 64, P4, W, pw, None) in (CUDA, OK)


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "attention_fp16_flashattention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith(".py"):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), fn
