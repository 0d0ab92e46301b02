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
