"""Seeded synthetic inputs for the attention workloads (numpy, host memory).

This module only draws random numbers and lays them out; it holds none of the
attention, bridge or selection arithmetic.  Tests, ``bench.py`` and
``__graft_entry__.smoke()`` use it to feed both the CUDA library and the CPU
oracle the same bytes.

Workloads (shapes and value distributions of the pages' workloads: D128
video-DiT heads, Hq6/Hkv1/D256 long prefill with 32-token E4M3 pages, VSA
with 64-token cubes and top-k 64):

  dense_small   B1 H2  S256   D128, Q/K/V ~ N(0,1)
  causal_small  B1 Hq6 Hkv1 D256, Q=1024 after a 3072-token prefix (KV=4096)
  dense_video   B1 H24 S32768 D128, Q/K = 0.5 N(0,1) + per-head mean offset
                (each entry N(0, 0.2^2)), V ~ N(0,1)
  vsa_video     B1 H24 S32768 D128 on an 8x64x64 latent grid split in 512
                cubes of 4x4x4; Q/K = smooth low-frequency signal + N(0,1)
  paged_e4m3    B1 Hq6 Hkv1 D256, Q=8192 at the tail of KV=131072, K/V as
                E4M3 bytes uniform over the 254 finite codes in 32-token pages
                behind a random page-table permutation; scales 1/16 and 1/8
  dense_masked  B1 H24 S8192 D128, Q/K/V ~ N(0,1), one FP16 additive mask
                [8192][8192] shared by all heads: -2^-9 |i - j| plus 3% hidden keys
  vsa_full      B1 H24 D128: 1024 prefix tokens (N(0,1)) then an 8x62x62 latent
                grid in 4x4x4 cubes (2x16x16 = 512 cubes, boundary cubes padded:
                30752 real of 32768 slots), top-k 64; Q/K as vsa_video
  paged_decode  B4 Hq6 Hkv1 D256, one new token per sequence over ragged
                caches of 131072, 122887, 98313 and 65571 tokens (K/V bytes and
                pages as paged_e4m3, every sequence's pages scattered over one
                shared physical pool); scales 1/16 and 1/8

Every tensor is drawn from its own numpy PCG64 stream keyed by
(seed, tensor tag), so shapes can be shrunk for tests without changing the
recipe.
"""

import math

import numpy as np

TAGS = {"q": 1, "k": 2, "v": 3, "kpages": 4, "vpages": 5, "table": 6,
        "qmean": 7, "kmean": 8, "qsig": 9, "ksig": 10, "rows": 11, "mask": 12}


def _rng(seed, tag):
    return np.random.default_rng([int(seed), TAGS[tag]])


def _normal_fp16(rng, shape, std=1.0):
    """N(0, std^2) values rounded to FP16 (numpy's float32 -> float16 is RNE)."""
    out = np.empty(shape, dtype=np.float16)
    flat = out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat.size, step):
        n = min(step, flat.size - i)
        x = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        flat[i:i + n] = x.astype(np.float16)
    return out


def dense_inputs(B, H, S, D, seed, skv=None, video=False):
    """Q [B][H][S][D], K/V [B][H][Skv][D] FP16.

    video=False: all three i.i.d. N(0,1).
    video=True : Q, K = 0.5 * N(0,1) + mu (mu: one vector per (tensor, head),
                 entries N(0, 0.2^2)); V ~ N(0,1).
    """
    skv = S if skv is None else skv
    if not video:
        q = _normal_fp16(_rng(seed, "q"), (B, H, S, D))
        k = _normal_fp16(_rng(seed, "k"), (B, H, skv, D))
        v = _normal_fp16(_rng(seed, "v"), (B, H, skv, D))
        return q, k, v
    out = []
    for name, mean_tag, n in (("q", "qmean", S), ("k", "kmean", skv)):
        mu = (_rng(seed, mean_tag).standard_normal((B, H, 1, D)) * 0.2).astype(np.float32)
        x = np.empty((B, H, n, D), dtype=np.float16)
        rng = _rng(seed, name)
        for b in range(B):
            for h in range(H):
                z = rng.standard_normal((n, D), dtype=np.float32) * np.float32(0.5)
                x[b, h] = (z + mu[b, h]).astype(np.float16)
        out.append(x)
    v = _normal_fp16(_rng(seed, "v"), (B, H, skv, D))
    return out[0], out[1], v


def causal_inputs(B, Hq, Hkv, Q, KV, D, seed):
    """Q [B][Hq][Q][D], K/V [B][Hkv][KV][D] FP16, all N(0,1)."""
    q = _normal_fp16(_rng(seed, "q"), (B, Hq, Q, D))
    k = _normal_fp16(_rng(seed, "k"), (B, Hkv, KV, D))
    v = _normal_fp16(_rng(seed, "v"), (B, Hkv, KV, D))
    return q, k, v


def cube_major_permutation(grid, cube):
    """Token permutation raster (t, y, x) -> cube-major order.

    Returns perm with cube_major[i] = raster[perm[i]].  Cube index
    c = ((t//ct) * (Y//cy) + y//cy) * (X//cx) + x//cx; inside a cube tokens go
    in (t%ct, y%cy, x%cx) raster order.
    """
    T, Y, X = grid
    ct, cy, cx = cube
    t, y, x = np.meshgrid(np.arange(T), np.arange(Y), np.arange(X), indexing="ij")
    c = ((t // ct) * (Y // cy) + y // cy) * (X // cx) + x // cx
    inner = ((t % ct) * cy + y % cy) * cx + x % cx
    pos = (c * (ct * cy * cx) + inner).reshape(-1)      # cube-major position of each raster token
    perm = np.empty_like(pos)
    perm[pos] = np.arange(pos.size)
    return perm


def _smooth_signal(rng, H, D, grid, n_terms=4):
    """Per head, a sum of n_terms low-frequency plane waves on the grid.

    signal[token, d] = sum_r a[r, d] * cos(2 pi (f_t t/T + f_y y/Y + f_x x/X) + phi[r, d]),
    f in {0, 1, 2} per axis and term, a ~ N(0,1)/2, phi ~ U[0, 2 pi).
    Returned in raster token order, float32 [H][T*Y*X][D].
    """
    T, Y, X = grid
    t, y, x = np.meshgrid(np.arange(T), np.arange(Y), np.arange(X), indexing="ij")
    t = t.reshape(-1)
    y = y.reshape(-1)
    x = x.reshape(-1)
    out = np.empty((H, T * Y * X, D), dtype=np.float32)
    for h in range(H):
        f = rng.integers(0, 3, size=(n_terms, 3))
        a = rng.standard_normal((n_terms, D)) / 2.0
        phi = rng.uniform(0.0, 2.0 * math.pi, size=(n_terms, D))
        theta = 2.0 * math.pi * (f[:, 0:1] * t[None] / T + f[:, 1:2] * y[None] / Y
                                 + f[:, 2:3] * x[None] / X)            # [R][N]
        basis = np.concatenate([np.cos(theta), np.sin(theta)], axis=0)   # [2R][N]
        coef = np.concatenate([a * np.cos(phi), -a * np.sin(phi)], axis=0)  # [2R][D]
        out[h] = (basis.T @ coef).astype(np.float32)
    return out


def vsa_inputs(B, H, D, seed, grid=(8, 64, 64), cube=(4, 4, 4)):
    """Q, K, V [B][H][S][D] FP16 in cube-major token order, S = T*Y*X."""
    S = grid[0] * grid[1] * grid[2]
    perm = cube_major_permutation(grid, cube)
    out = []
    for name, sig_tag in (("q", "qsig"), ("k", "ksig")):
        sig_rng = _rng(seed, sig_tag)
        rng = _rng(seed, name)
        x = np.empty((B, H, S, D), dtype=np.float16)
        for b in range(B):
            sig = _smooth_signal(sig_rng, H, D, grid)
            for h in range(H):
                z = rng.standard_normal((S, D), dtype=np.float32)
                x[b, h] = (sig[h] + z)[perm].astype(np.float16)
        out.append(x)
    v = _normal_fp16(_rng(seed, "v"), (B, H, S, D))
    return out[0], out[1], v


FINITE_E4M3 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def padded_cube_layout(grid, cube):
    """Cube-major layout with boundary padding for a grid the cube may not divide.

    Returns (slot, valid): slot[raster token] = its position in the padded
    cube-major sequence (cube c owns slots c*V .. c*V + V - 1, V = ct*cy*cx;
    its real tokens fill the first slots in (t, y, x) raster order inside the
    cube), valid[c] = real tokens of cube c.
    """
    T, Y, X = grid
    ct, cy, cx = cube
    nt, ny, nx = -(-T // ct), -(-Y // cy), -(-X // cx)
    t, y, x = (a.reshape(-1) for a in np.meshgrid(np.arange(T), np.arange(Y), np.arange(X),
                                                   indexing="ij"))
    c = ((t // ct) * ny + y // cy) * nx + x // cx
    inner = ((t % ct) * cy + y % cy) * cx + x % cx
    order = np.lexsort((inner, c))                 # raster tokens sorted by (cube, inner)
    valid = np.bincount(c, minlength=nt * ny * nx).astype(np.int32)
    first = np.concatenate([[0], np.cumsum(valid)[:-1]])
    rank = np.empty(order.size, dtype=np.int64)
    rank[order] = np.arange(order.size)
    slot = c * (ct * cy * cx) + (rank - first[c])
    return slot, valid


def vsa_full_inputs(B, H, D, seed, grid, cube=(4, 4, 4), prefix=0):
    """The full VSA layout: `prefix` prefix tokens (text/audio, N(0,1)), then the
    video tokens of `grid` in padded cube-major order (smooth low-frequency signal
    + N(0,1) for Q and K, N(0,1) for V; padding slots zero).

    Returns q, k, v [B][H][prefix + cubes*64][D] FP16 and valid int32 [cubes].
    """
    slot, valid = padded_cube_layout(grid, cube)
    nc = valid.size
    V = cube[0] * cube[1] * cube[2]
    S = prefix + nc * V
    n = grid[0] * grid[1] * grid[2]
    out = []
    for name, sig_tag in (("q", "qsig"), ("k", "ksig")):
        sig_rng = _rng(seed, sig_tag)
        rng = _rng(seed, name)
        x = np.zeros((B, H, S, D), dtype=np.float16)
        for b in range(B):
            sig = _smooth_signal(sig_rng, H, D, grid)
            for h in range(H):
                x[b, h, :prefix] = rng.standard_normal((prefix, D), dtype=np.float32)
                z = rng.standard_normal((n, D), dtype=np.float32)
                x[b, h, prefix + slot] = (sig[h] + z).astype(np.float16)
        out.append(x)
    v = np.zeros((B, H, S, D), dtype=np.float16)
    vr = _normal_fp16(_rng(seed, "v"), (B, H, prefix + n, D))
    v[:, :, :prefix] = vr[:, :, :prefix]
    v[:, :, prefix + slot] = vr[:, :, prefix:]
    return out[0], out[1], v, valid


def paged_e4m3_inputs(Hkv, KV, D, seed, page_size=32, num_phys_pages=None):
    """K/V E4M3 pages [P][page_size][Hkv][D] uint8 and an int32 page table.

    Bytes are uniform over the 254 finite E4M3 codes; the page table is a
    seeded permutation of the physical pages (logical page i -> table[i]).
    """
    n_log = -(-KV // page_size)
    P = n_log if num_phys_pages is None else num_phys_pages
    rk = _rng(seed, "kpages")
    rv = _rng(seed, "vpages")
    kp = FINITE_E4M3[rk.integers(0, FINITE_E4M3.size, size=(P, page_size, Hkv, D))]
    vp = FINITE_E4M3[rv.integers(0, FINITE_E4M3.size, size=(P, page_size, Hkv, D))]
    table = _rng(seed, "table").permutation(P)[:n_log].astype(np.int32)
    return kp, vp, table


def _e4m3_codes(rng, shape, codes):
    if codes == "finite":
        return FINITE_E4M3[rng.integers(0, FINITE_E4M3.size, size=shape)]
    if codes == "moderate":     # random sign and mantissa, exponent field 3..9
        sign = rng.integers(0, 2, size=shape, dtype=np.uint8)
        expo = rng.integers(3, 10, size=shape, dtype=np.uint8)
        mant = rng.integers(0, 8, size=shape, dtype=np.uint8)
        return (sign << 7) | (expo << 3) | mant
    raise ValueError(codes)


def paged_decode_inputs(B, Hq, Hkv, nq, kv_lens, D, seed, page_size=32, spare_pages=0,
                        codes="finite"):
    """Decode inputs: Q, K/V E4M3 pages, a page table and the sequence lengths.

    q          FP16 [B][Hq][nq][D] ~ N(0,1)
    k/v pages  uint8 [P][page_size][Hkv][D], P = every sequence's pages + spare_pages
    page_table int32 [B][max_pages]: sequence b's logical pages on a seeded
               permutation of the physical pool; entries past its last page are -1
    kv_lens    int32 [B]
    codes: "finite" (uniform over the 254 finite E4M3 codes, the paged_e4m3
    recipe) or "moderate" (|value| in [2^-4, 7.5], so the softmax spreads over
    many keys).
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    n_log = [-(-int(n) // page_size) for n in kv_lens]
    max_pages = max(n_log)
    P = sum(n_log) + spare_pages
    q = _normal_fp16(_rng(seed, "q"), (B, Hq, nq, D))
    kp = _e4m3_codes(_rng(seed, "kpages"), (P, page_size, Hkv, D), codes)
    vp = _e4m3_codes(_rng(seed, "vpages"), (P, page_size, Hkv, D), codes)
    perm = _rng(seed, "table").permutation(P).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, :n_log[b]] = perm[at:at + n_log[b]]
        at += n_log[b]
    return q, kp, vp, table, kv_lens


def additive_mask(Sq, Skv, seed, hidden_keys=0.03, slope=2.0 ** -9):
    """FP16 additive mask [Sq][Skv]: a relative-position bias -slope*|i - j| (the
    linear distance bias of ALiBi-style attention) plus a seeded set of hidden
    key columns (about hidden_keys of them, -inf), as key padding would give."""
    i = np.arange(Sq, dtype=np.float32)[:, None]
    j = np.arange(Skv, dtype=np.float32)[None, :]
    m = (-np.float32(slope) * np.abs(i - j)).astype(np.float16)
    hide = _rng(seed, "mask").random(Skv) < hidden_keys
    hide[0] = False
    m[:, hide] = -np.inf
    return m


def sample_rows(n_heads, n_rows, count, seed, row_limit=None):
    """``count`` distinct seeded (head, row) pairs, sorted; rows < row_limit."""
    lim = n_rows if row_limit is None else row_limit
    total = n_heads * lim
    rng = _rng(seed, "rows")
    pick = rng.choice(total, size=min(count, total), replace=False)
    pick.sort()
    return np.stack([pick // lim, pick % lim], axis=1).astype(np.int64)


# The eight workloads, with their seeds (1000 + workload number).
WORKLOADS = {
    "dense_small": dict(kind="dense", B=1, H=2, S=256, D=128, seed=1001),
    "causal_small": dict(kind="causal", B=1, Hq=6, Hkv=1, Q=1024, KV=4096, D=256, seed=1002),
    "dense_video": dict(kind="dense", B=1, H=24, S=32768, D=128, seed=1003, video=True),
    "vsa_video": dict(kind="vsa", B=1, H=24, D=128, grid=(8, 64, 64), cube=(4, 4, 4), topk=64,
                      seed=1004),
    "paged_e4m3": dict(kind="paged", B=1, Hq=6, Hkv=1, Q=8192, KV=131072, D=256, page_size=32,
                       k_scale=0.0625, v_scale=0.125, seed=1005),
    "dense_masked": dict(kind="masked", B=1, H=24, S=8192, D=128, seed=1007),
    "vsa_full": dict(kind="vsa_full", B=1, H=24, D=128, grid=(8, 62, 62), cube=(4, 4, 4),
                     prefix=1024, topk=64, seed=1008),
    "paged_decode": dict(kind="decode", B=4, Hq=6, Hkv=1, nq=1,
                         kv_lens=(131072, 122887, 98313, 65571), D=256, page_size=32,
                         k_scale=0.0625, v_scale=0.125, seed=1006),
}


def softmax_scale(D):
    """The FP32 scale 1/sqrt(D) (computed in double, stored as float)."""
    return float(np.float32(1.0 / math.sqrt(D)))
