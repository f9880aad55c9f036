"""Tensor-core prefill encoder versus the oracle's fp32 specification.

Long appends of bf16/f16 vectors rotate on the tensor cores (the pages plan
tensor cores for the head_dim x head_dim rotation of chunked prefill). That
cannot follow the specification's sequential fp32 rounding order, so the rule
checked here is:
  * norms are bit-exact (the kernel keeps the sequential order for them);
  * an index may differ from the oracle's only where the exact rotated
    coordinate y (fp64) lies within the fp32 error band of every midpoint that
    separates the two codes; the band is the dot-product bound
    gamma_D * sum_k |R_ik x_k| / |x| plus (gamma_D + 2^-21)|y| for the norm,
    the division and the tensor-core side's own rounding;
  * for prod keys whose indices all agree, a QJL sign may differ only where
    the exact (S r)_j lies within the propagated band of 0, and the residual
    norms differ by at most the propagated band plus the fp32 bound of a sum
    of D squares in any order;
  * group-quantised values are not rotated and stay bit-exact.
Expected values come from the oracle alone; the exact y and S r are recomputed
here in fp64 from the oracle's fp32 tables.
"""

import numpy as np
import pytest
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import read_records, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _gamma(n: int) -> float:
    return n * U / (1 - n * U)


def _bits(words: np.ndarray, D: int, b: int) -> np.ndarray:
    return np.stack([O.unpack(w, D, b) for w in words]).astype(np.int64)


def check_rotated(codec: O.Codec, X: np.ndarray, got: dict, want: dict):
    """Apply the tie-band rule to one tensor's records.

    Returns (index flips, sign flips, ambiguous coordinates): a coordinate is
    ambiguous when its exact rotated value lies within its band of a midpoint,
    and only ambiguous coordinates may flip.
    """
    D = codec.D
    gD = _gamma(D)
    x = X.astype(np.float64)
    assert np.array_equal(got["norm"].view(np.uint32), want["norm"].view(np.uint32))
    n64 = np.sqrt((x * x).sum(1))
    # the specification's fp32 norm (bit-exact on both sides) decides which
    # vectors are zero: rows at 2^-100 square to 0 in fp32 and encode as y = 0
    nz = want["norm"] > 0
    R = codec.R.astype(np.float64)
    y = np.zeros_like(x)
    ay = np.zeros_like(x)
    y[nz] = (x[nz] @ R.T) / n64[nz, None]
    ay[nz] = (np.abs(x[nz]) @ np.abs(R).T) / n64[nz, None]
    band = gD * ay + (gD + 2.0 ** -21) * np.abs(y)
    cg, cw = _bits(got["idx"], D, codec.ib), _bits(want["idx"], D, codec.ib)
    diff = cg != cw
    m = codec.m.astype(np.float64)
    for t, i in zip(*np.nonzero(diff)):
        lo, hi = sorted((int(cg[t, i]), int(cw[t, i])))
        for j in range(lo, hi):
            assert abs(y[t, i] - m[j]) <= band[t, i], \
                f"token {t} coord {i}: codes {cg[t, i]} vs {cw[t, i]}, y={y[t, i]:.9g}, " \
                f"midpoint {m[j]:.9g}, band {band[t, i]:.3g}"
    ambiguous = int(((np.abs(y[:, :, None] - m[None, None, :]) <= band[:, :, None]).any(-1) & (band > 0)).sum())
    sflips = 0
    if codec.mode == O.PROD:
        # every token, flipped or not: the residual follows the GPU's own
        # indices, r = y - c[index], and its signs and norm are checked
        # against the exact values recomputed from those indices
        c = codec.c.astype(np.float64)
        S = codec.S.astype(np.float64)
        r = y - c[cg]
        z = r @ S.T
        bz = gD * (np.abs(r) @ np.abs(S).T) + (band + 2.0 ** -23 * np.abs(r)) @ np.abs(S).T
        sg = _bits(got["sgn"], D, 1)
        sd = sg != (z >= 0)
        for t, j in zip(*np.nonzero(sd)):
            assert abs(z[t, j]) <= bz[t, j], f"token {t} sign {j}: z={z[t, j]:.9g}, band {bz[t, j]:.3g}"
        sflips = int(sd.sum())
        # the kernel sums D fp32 squares of its own residual (relative error
        # <= gamma_D / 2), whose coordinates are within `band` of r, then
        # rounds a square root
        rn = np.sqrt((r * r).sum(1))
        rband = 2.0 * np.sqrt((band * band).sum(1)) + (gD + 2.0 ** -22) * rn
        dr = np.abs(got["rnorm"].astype(np.float64) - rn)
        assert np.all(dr <= rband), f"max rnorm excess {(dr - rband).max():.3g}"
    return int(diff.sum()), sflips, ambiguous


CASES = [
    # head_dim, key codec, value codec, tokens appended, tokens already cached per sequence, dtype
    (128, ("prod", 3), ("mse", 3), 300, (0, 40), torch.bfloat16),
    (128, ("mse", 4), ("mse", 2), 200, (5,), torch.bfloat16),
    (128, ("prod", 5), ("mse", 4), 129, (0,), torch.float16),
    (128, ("prod", 2), ("mse", 1), 256, (17, 0, 100), torch.bfloat16),
    (128, ("prod", 3), ("group", 2, 32), 64, (0,), torch.bfloat16),
    (64, ("prod", 4), ("mse", 3), 190, (3, 64), torch.bfloat16),
    (64, ("mse", 2), ("group", 4, 64), 128, (0,), torch.bfloat16),
]


@pytest.mark.parametrize("D,key,value,n_new,lens,dtype", CASES)
def test_tensor_core_encode_within_tie_band(D, key, value, n_new, lens, dtype):
    Hkv, BT = 2, 16
    kspec = wl._spec(key[0], key[1], 21)
    vspec = wl._spec(value[0], value[1], 22, value[2] if len(value) > 2 else 0)
    w = wl.Workload("tc_encode", 1, len(lens), Hkv, Hkv * 2, D, tuple(lens), 1, dtype, 1.0, 7,
                    kspec, vspec, block_tokens=BT, shuffle_blocks=True, append_per_step=n_new)
    table, nblocks = wl.block_table(w, [n + n_new for n in lens])
    max_blocks = table.shape[1]
    kc_g, vc_g = tq.Codec(D, kspec.bits, kspec.mode, kspec.seed, kspec.group_size), \
        tq.Codec(D, vspec.bits, vspec.mode, vspec.seed, vspec.group_size)
    cache = tq.CompressedKVCache(kc_g, vc_g, 1, nblocks, BT, Hkv, DEV)
    assert cache.desc.encode_policy == tq.TQ_ENCODE_AUTO
    B = len(lens)
    K = wl.encoder_stress(101, B, Hkv, n_new, D, dtype, DEV)
    V = wl.encoder_stress(202, B, Hkv, n_new, D, dtype, DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    cache.append(0, K, V, sl, table.to(DEV), max_blocks)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0

    kc = O.Codec(D, kspec.bits, kspec.mode, kspec.seed)
    vc = O.Codec(D, vspec.bits, vspec.mode, vspec.seed, vspec.group_size)
    pool = cache.pool.cpu().numpy()
    Kn, Vn = to_f32_np(K), to_f32_np(V)
    flips = sflips = coords = ambiguous = 0
    for b in range(B):
        for h in range(Hkv):
            gk, gv = read_records(pool, kc, vc, Hkv, BT, table.numpy(), max_blocks, b, h, lens[b], n_new)
            wk, wv = kc.encode(Kn[b, h]), vc.encode(Vn[b, h])
            f, s, a = check_rotated(kc, Kn[b, h], gk, wk)
            flips, sflips, ambiguous = flips + f, sflips + s, ambiguous + a
            if vc.mode == O.GROUP:
                for name in ("idx", "scale", "min"):
                    assert np.array_equal(gv[name], wv[name])
            else:
                f, _, a = check_rotated(vc, Vn[b, h], gv, wv)
                flips, ambiguous = flips + f, ambiguous + a
            coords += 2 * n_new * D
    # only a coordinate whose exact value lies inside its band may flip
    assert flips <= ambiguous, f"{flips} index flips, {ambiguous} ambiguous coordinates"
    print(f"tie-band: {flips} index flips of {ambiguous} ambiguous coordinates, {sflips} sign flips, "
          f"{coords} coordinates")


def test_exact_policy_is_bit_exact_for_long_appends():
    D, Hkv, BT, n_new = 128, 2, 16, 300
    kc_g, vc_g = tq.Codec(D, 3, tq.TQ_MODE_PROD, 0), tq.Codec(D, 3, tq.TQ_MODE_MSE, 1)
    nblk = (n_new + BT - 1) // BT
    cache = tq.CompressedKVCache(kc_g, vc_g, 1, nblk, BT, Hkv, DEV, exact_encode=True)
    K = wl.encoder_stress(5, 1, Hkv, n_new, D, torch.bfloat16, DEV)
    V = wl.encoder_stress(6, 1, Hkv, n_new, D, torch.bfloat16, DEV)
    cache.append(0, K, V, torch.zeros(1, dtype=torch.int32, device=DEV), None, nblk)
    torch.cuda.synchronize()
    kc, vc = O.Codec(D, 3, O.PROD, 0), O.Codec(D, 3, O.MSE, 1)
    pool = cache.pool.cpu().numpy()
    Kn, Vn = to_f32_np(K), to_f32_np(V)
    for h in range(Hkv):
        gk, gv = read_records(pool, kc, vc, Hkv, BT, None, nblk, 0, h, 0, n_new)
        wk, wv = kc.encode(Kn[0, h]), vc.encode(Vn[0, h])
        for name in wk:
            assert np.array_equal(gk[name].view(np.uint32), wk[name].view(np.uint32)), name
        for name in wv:
            assert np.array_equal(gv[name].view(np.uint32), wv[name].view(np.uint32)), name


def test_unknown_encode_policy_is_refused():
    kc, vc = tq.Codec(128, 3, tq.TQ_MODE_PROD, 0), tq.Codec(128, 3, tq.TQ_MODE_MSE, 1)
    cache = tq.CompressedKVCache(kc, vc, 1, 4, 16, 1, DEV)
    cache.desc.encode_policy = 7
    x = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tq.TQError) as e:
        cache.append(0, x, x, torch.zeros(1, dtype=torch.int32, device=DEV), None, 4)
    assert e.value.status == 1
