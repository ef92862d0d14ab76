"""Host packer: round trips, the documented byte positions, padding and errors.

The byte positions are checked against the layout as documented in
include/woq.h and the packer's layout notes (tile-major blocks of 128 rows x
128 k; scales first, row 32j+l at half-word 4l+j; int4 chunk (c, j, l) at
256 + 16 * ((4c + j) * 32 + (l ^ 2c)), word i holding k0 = 32c + 8i: low nibble of
byte b = k0+b, high nibble = k0+4+b; int6 high bits in a second region).
"""
import numpy as np
import pytest

from tests.helpers import encode_w4, encode_w6

import weight_only_quantised_gb300 as woq


def _rand(bits, N, K, seed):
    rng = np.random.default_rng(seed)
    lo, hi = (-8, 7) if bits == 4 else (-32, 31)
    wv = rng.integers(lo, hi + 1, size=(N, K))
    q = encode_w4(wv) if bits == 4 else encode_w6(wv)
    s = rng.integers(0, 1 << 16, size=(N, K // 128), dtype=np.uint32).astype(np.uint16)
    return wv, q, s


def _pack(bits, q, s, N, K):
    return (woq.woq_pack_w4 if bits == 4 else woq.woq_pack_w6)(q, s, N, K)


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("N,K", [(1, 128), (128, 128), (129, 256), (300, 384), (1000, 1024), (256, 0), (0, 256)])
def test_round_trip(bits, N, K):
    wv, q, s = _rand(bits, N, K, seed=N * 7 + K + bits)
    packed = _pack(bits, q, s, N, K)
    assert packed.nbytes == woq.woq_packed_bytes(bits, N, K)
    q2, s2 = woq.woq_unpack(bits, packed, N, K)
    assert np.array_equal(q2, q)
    assert np.array_equal(s2, s)


def test_header_fields():
    N, K = 300, 384
    _, q, s = _rand(4, N, K, 1)
    packed = _pack(4, q, s, N, K)
    h = packed[:48].view(np.uint32)
    assert h[0] == 0x31514F57 and h[1] == 2 and h[2] == 4 and h[3] == 128
    assert h[4] == N and h[5] == K and h[6] == 3 and h[7] == 3
    assert packed[8 * 4: 16 * 4].view(np.uint64).tolist()[:2] == [8448, woq.woq_packed_bytes(4, N, K)]
    assert not packed[48:256].any()


def _block(packed, bits, t, g, G):
    bb = 8448 if bits == 4 else 12544
    off = 256 + (t * G + g) * bb
    return packed[off: off + bb]


@pytest.mark.parametrize("bits", [4, 6])
def test_documented_byte_positions(bits):
    N, K = 260, 256  # three tiles (the last ragged), two groups
    G = K // 128
    wv, q, s = _rand(bits, N, K, seed=5 + bits)
    packed = _pack(bits, q, s, N, K)
    rng = np.random.default_rng(0)
    for _ in range(400):
        n = int(rng.integers(0, N))
        k = int(rng.integers(0, K))
        t, r = divmod(n, 128)
        g, kk = divmod(k, 128)
        j, l = divmod(r, 32)
        c, k32 = divmod(kk, 32)
        i, within = divmod(k32, 8)
        half, b = divmod(within, 4)
        blk = _block(packed, bits, t, g, G)
        # scale of (row, group)
        assert blk[:256].view(np.uint16)[4 * l + j] == s[n, g]
        # low four bits of the weight
        byte = blk[256 + 16 * ((4 * c + j) * 32 + (l ^ (2 * c))) + 4 * i + b]
        nib = (byte >> 4) if half else (byte & 0xF)
        assert nib == (wv[n, k] & 0xF)
        if bits == 6:
            h, e = divmod(i, 2)
            ub = blk[256 + 8192 + 8 * ((4 * c + j) * 32 + l) + 4 * h + b]
            assert ((ub >> (2 * (2 * e + half))) & 3) == ((wv[n, k] >> 4) & 3)
    # rows beyond N are zero (weights and scales)
    last = _block(packed, bits, 2, 1, G)
    for r in range(N - 256, 128):
        j, l = divmod(r, 32)
        assert last[:256].view(np.uint16)[4 * l + j] == 0
        for c in range(4):
            o = 256 + 16 * ((4 * c + j) * 32 + (l ^ (2 * c)))
            assert not last[o: o + 16].any()


def test_int4_values_in_int6_format_share_the_low_plane():
    N, K = 130, 256
    wv, q4, s = _rand(4, N, K, 11)
    p4 = _pack(4, q4, s, N, K)
    p6 = _pack(6, encode_w6(wv), s, N, K)
    G = K // 128
    for t in range(2):
        for g in range(G):
            b4 = _block(p4, 4, t, g, G)
            b6 = _block(p6, 6, t, g, G)
            assert np.array_equal(b4, b6[:8448])


def test_pack_errors():
    q = np.zeros((4, 64), dtype=np.uint8)
    s = np.zeros((4, 1), dtype=np.uint16)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_pack_w4(q, s, 4, 100)
    assert e.value.status == woq.WOQ_ERR_SHAPE
    packed = woq.woq_pack_w4(q, s, 4, 128)
    bad = packed.copy()
    bad[8] = 6  # header says int6
    with pytest.raises(woq.WoqError) as e:
        woq.woq_unpack(4, bad, 4, 128)
    assert e.value.status == woq.WOQ_ERR_LAYOUT
    with pytest.raises(woq.WoqError):
        woq.woq_unpack(4, packed, 5, 128)  # wrong N
    with pytest.raises(woq.WoqError):
        woq.woq_unpack(4, packed[:-1], 4, 128)  # truncated
