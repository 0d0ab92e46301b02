"""Pins of the INT8 quantisation oracle (oracle/quant.py) against facts that
do not come from the oracle itself: the rounding bound of symmetric absmax
quantisation, exact grid points, half-to-even ties, which axis shares a
scale, which middle rows belong to complete blocks, and the reduction to
plain attention when the data sit exactly on the quantisation grid."""
import numpy as np

from oracle import attention as OA
from oracle import quant as Q


def _rng(seed=0):
    return np.random.default_rng(seed)


def test_round_trip_within_half_a_step():
    x = _rng(1).standard_normal((128, 64)).astype(np.float32) * 3
    codes, s = Q.quantize_per_channel(x)
    assert codes.dtype == np.int8 and s.shape == (64,)
    err = np.abs(Q.dequantize_per_channel(codes, s) - x)
    assert np.all(err <= s[None, :] * (0.5 + 1e-5))
    # the absmax element of each channel lands on +-127 exactly
    i = np.abs(x).argmax(axis=0)
    assert np.all(np.abs(codes[i, np.arange(64)]) == 127)
    v = _rng(2).standard_normal((128, 128)).astype(np.float32)
    vc, vs = Q.quantize_per_token(v)
    assert vs.shape == (128,)
    assert np.all(np.abs(Q.dequantize_per_token(vc, vs) - v) <= vs[:, None] * (0.5 + 1e-5))
    assert np.all(np.abs(vc).max(axis=1) == 127)


def test_grid_points_are_exact():
    # scale 2^-5 (absmax 127 * 2^-5): every j * 2^-5 is represented exactly
    j = _rng(3).integers(-127, 128, size=(128, 32))
    j[0] = 127
    x = (j * 2.0 ** -5).astype(np.float32)
    codes, s = Q.quantize_per_channel(x)
    assert np.all(s == np.float32(2.0 ** -5))
    assert np.array_equal(codes.astype(np.int64), j)


def test_ties_round_half_to_even():
    # absmax 127 gives scale 1: x / s is x itself
    x = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5]], dtype=np.float32)
    codes, s = Q.quantize_per_token(x)
    assert s[0] == 1.0
    assert list(codes[0]) == [127, 2, 4, -2, 0, 0, 2]


def test_zero_blocks_and_axes():
    z = np.zeros((128, 32), np.float32)
    c, s = Q.quantize_per_channel(z)
    assert not c.any() and not s.any()
    # one large channel changes only its own K scale ...
    k = np.ones((128, 32), np.float32)
    k[5, 3] = 100.0
    c, s = Q.quantize_per_channel(k)
    assert s[3] == np.float32(100.0) / np.float32(127) and np.all(np.delete(s, 3) == np.float32(1) / np.float32(127))
    # ... and one large token only its own V scale
    v = np.ones((128, 128), np.float32)
    v[7, 9] = -50.0
    c, s = Q.quantize_per_token(v)
    assert s[7] == np.float32(50.0) / np.float32(127) and np.all(np.delete(s, 7) == np.float32(1) / np.float32(127))
    assert c[7, 9] == -127 and c[7, 0] == 3      # 1 / (50/127) = 2.54 -> 3


def test_only_complete_blocks_are_quantised():
    S, W, d = 4, 16, 128
    kept = np.arange(0, 128, 4)                  # 32 kept channels
    rng = _rng(4)
    for M in (0, 127, 128, 129, 300):            # middle rows
        N = S + W + M
        K = rng.standard_normal((N, d)).astype(np.float32)
        V = rng.standard_normal((N, d)).astype(np.float32)
        Kq, Vq = Q.quantized_history(K, V, kept, 0, N, S, W)
        nb = M // 128
        assert Q.sealed_blocks(len(kept), N, S, W) == nb
        changed_v = np.nonzero(np.any(Vq != V, axis=1))[0]
        changed_k = np.nonzero(np.any(Kq != K, axis=1))[0]
        sealed = np.arange(S, S + 128 * nb)
        assert set(changed_v) <= set(sealed) and set(changed_k) <= set(sealed)
        assert len(changed_v) >= 0.9 * len(sealed)
        # pruned channels and everything outside the sealed rows are untouched
        pruned = np.setdiff1d(np.arange(d), kept)
        assert np.array_equal(Kq[:, pruned], K[:, pruned].astype(np.float64))
    # other policies and k = 0 heads are never quantised
    N = S + W + 256
    K = rng.standard_normal((N, d)).astype(np.float32)
    for policy, kk in ((1, kept), (2, kept), (0, np.arange(0))):
        Kq, Vq = Q.quantized_history(K, K, kk, policy, N, S, W)
        assert np.array_equal(Kq, K.astype(np.float64))


def test_on_grid_history_decodes_exactly_like_plain_attention():
    # integer-valued K, V whose every block / channel / token reaches 127:
    # quantisation is the identity and decode equals the unquantised oracle
    S, W, N, G, d = 4, 16, 4 + 16 + 256 + 50, 2, 128
    rng = _rng(5)
    K = rng.integers(-127, 128, size=(N, d)).astype(np.float32)
    V = rng.integers(-127, 128, size=(N, d)).astype(np.float32)
    K[S::7] = 127.0
    V[:, 0] = 127.0
    kept = np.arange(64)
    for blk in range(2):
        K[S + 128 * blk, kept] = 127.0
    q = rng.standard_normal((G, d)) * 0.01
    o_q = Q.decode_head_quantized(q, K, V, 0, kept, N, S, W, 0)
    o = OA.decode_head(q, K, V, 0, kept, N, S, W, 0)
    assert np.array_equal(o_q, o)
    # off the grid the two differ, by about the quantisation error
    Kf = rng.standard_normal((N, d)).astype(np.float32)
    Vf = rng.standard_normal((N, d)).astype(np.float32)
    q = rng.standard_normal((G, d))
    d_o = np.abs(Q.decode_head_quantized(q, Kf, Vf, 0, kept, N, S, W, 0)
                 - OA.decode_head(q, Kf, Vf, 0, kept, N, S, W, 0)).max()
    assert 1e-6 < d_o < 0.05


def test_quantized_resident_bytes_are_the_arrays_sizes():
    # the closed form against the sizes of the representation itself: bf16
    # rows outside sealed blocks plus, per sealed block, the int8 code arrays
    # and fp32 scale arrays that middle_blocks builds
    from oracle import footprint as F
    rs = _rng(9)
    S, W, d = 4, 16, 128
    for k in (0, 32, 64, 96, 128):
        for N in (1, S + W, S + W + 127, S + W + 128, S + W + 300, S + W + 512):
            K = rs.standard_normal((N, d)).astype(np.float32)
            V = rs.standard_normal((N, d)).astype(np.float32)
            kept = np.arange(k)
            blocks = Q.middle_blocks(K, V, kept, N, S, W)
            sealed_rows = 128 * len(blocks)
            n_full, n_mid = F.resident_tokens(0, k, N, S, W, 0)
            if k == 128:                                  # dense head: no middle region of its own
                n_full, n_mid = min(N, S + W), max(0, N - S - W)
            arrays = sum(a.nbytes for blk in blocks for a in blk)
            want = n_full * 2 * d * 2 + (n_mid - sealed_rows) * (k + d) * 2 + arrays
            if k == 0:
                want = n_full * 2 * d * 2
            assert Q.resident_bytes_quantized(0, k, N, S, W, 0) == want, (k, N)
    # a whole k = 128 block takes 132 / 256 of its bf16 bytes
    assert Q.resident_bytes_quantized(0, 128, S + W + 128, S, W, 0) == \
        (S + W) * 512 + 128 * 256 + 4 * 256
    # other policies are untouched by quantisation
    assert Q.resident_bytes_quantized(1, 0, 1000, S, W, 64) == F.resident_bytes(1, 0, 1000, S, W, 64)
    assert Q.resident_bytes_quantized(2, 0, 1000, S, W, 64, n_special=9) == 9 * 512


# ---------------------------------------------------------------------------
# FP8 (e4m3): the encoder against the format's definition and a library cast
# ---------------------------------------------------------------------------

def test_e4m3_values_of_the_format():
    # fields S.EEEE.MMM with bias 7: the largest finite value, the smallest
    # subnormal and normal, one, a negative, and the NaN pattern
    v = Q.e4m3_value(np.arange(256))
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x07] == 7 * 2.0 ** -9
    assert v[0x38] == 1.0 and v[0x39] == 1.125 and v[0x77] == 240.0 and v[0xC0] == -2.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    finite = v[:0x7F]
    assert np.all(np.diff(finite) > 0)               # codes 0..126 ascend
    assert len(np.unique(np.abs(v[np.isfinite(v)]))) == 127


def test_e4m3_encoder_round_trip_ties_and_saturation():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = Q.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(Q.encode_e4m3(vals), codes)
    pos = Q.e4m3_value(np.arange(0x7F))
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)      # exact in fp32
    got = Q.encode_e4m3(mid).astype(np.int64)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))          # ties to the even code
    up = np.nextafter(mid, np.float32(np.inf))
    dn = np.nextafter(mid, np.float32(-np.inf))
    assert np.array_equal(Q.encode_e4m3(up).astype(np.int64), lo + 1)
    assert np.array_equal(Q.encode_e4m3(dn).astype(np.int64), lo)
    assert list(Q.encode_e4m3(np.float32([448.0, 449.0, 464.0, 1e6, -1e6]))) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e4m3_encoder_matches_a_library_cast():
    # torch's float8_e4m3fn cast rounds to nearest even; inside the finite
    # range it must give the same codes, subnormals and ties included
    import torch
    rs = _rng(11)
    x = np.concatenate([rs.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = np.concatenate([x, Q.e4m3_value(np.arange(0x7F)) * 1.0625, [0.0, 2.0 ** -10, 3 * 2.0 ** -10]])
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(Q.encode_e4m3(x), ref)


def test_fp8_quantisation_bounds_and_axes():
    x = _rng(12).standard_normal((128, 64)).astype(np.float32) * 3
    codes, s = Q.quantize_per_channel(x, "fp8")
    assert codes.dtype == np.uint8 and s.shape == (64,)
    assert np.all(s == np.abs(x).max(axis=0) / np.float32(448))
    deq = Q.dequantize_per_channel(codes, s, "fp8")
    # 3 mantissa bits: within half a step, 2^-4 relative, or half the
    # smallest subnormal step (2^-10 of the scale)
    assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, s[None, :] * 2.0 ** -10) * (1 + 1e-6))
    i = np.abs(x).argmax(axis=0)
    assert np.all((codes[i, np.arange(64)] & 0x7F) == 0x7E)          # the absmax lands on +-448
    assert np.all(np.abs(deq[i, np.arange(64)]) == 448.0 * s.astype(np.float64))
    v = np.ones((128, 128), np.float32)
    v[7, 9] = -50.0
    c, sv = Q.quantize_per_token(v, "fp8")
    assert sv[7] == np.float32(50.0) / np.float32(448) and c[7, 9] == 0xFE
    assert np.all(np.delete(sv, 7) == np.float32(1) / np.float32(448))
    z, zs = Q.quantize_per_channel(np.zeros((128, 32), np.float32), "fp8")
    assert not z.any() and not zs.any()


def test_fp8_on_grid_history_decodes_exactly_like_plain_attention():
    # K, V drawn from the e4m3 values with every block / channel / token
    # reaching 448: scale 1, quantisation is the identity
    S, W, N, G, d = 4, 16, 4 + 16 + 256 + 50, 2, 128
    rng = _rng(13)
    grid = Q.e4m3_value(np.arange(0x7F))
    K = (rng.choice(grid, size=(N, d)) * rng.choice([-1.0, 1.0], size=(N, d))).astype(np.float32)
    V = (rng.choice(grid, size=(N, d)) * rng.choice([-1.0, 1.0], size=(N, d))).astype(np.float32)
    V[:, 0] = 448.0
    kept = np.arange(32)
    for blk in range(2):
        K[S + 128 * blk, kept] = 448.0
    q = rng.standard_normal((G, d)) * 1e-4
    o_q = Q.decode_head_quantized(q, K, V, 0, kept, N, S, W, 0, fmt="fp8")
    o = OA.decode_head(q, K, V, 0, kept, N, S, W, 0)
    assert np.array_equal(o_q, o)
    Kf = rng.standard_normal((N, d)).astype(np.float32)
    Vf = rng.standard_normal((N, d)).astype(np.float32)
    q = rng.standard_normal((G, d))
    d8 = np.abs(Q.decode_head_quantized(q, Kf, Vf, 0, kept, N, S, W, 0, fmt="fp8")
                - OA.decode_head(q, Kf, Vf, 0, kept, N, S, W, 0)).max()
    d_i8 = np.abs(Q.decode_head_quantized(q, Kf, Vf, 0, kept, N, S, W, 0)
                  - OA.decode_head(q, Kf, Vf, 0, kept, N, S, W, 0)).max()
    assert 1e-6 < d8 < 0.2 and d8 > d_i8          # 3 mantissa bits lose more than 7-bit codes
