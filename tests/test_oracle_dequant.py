"""Pins for the oracle's any-precision dequantisation and stored layouts (no GPU)."""
import numpy as np
import pytest

from oracle import pw_oracle as O
from synth import get_config, make_expert


def _identity_luts(R):
    # LUT_b[r][v] = v is exact in fp16 for v < 64
    return [np.tile(np.arange(1 << b, dtype=np.float16), (R, 1)) for b in (3, 4, 5, 6)]


@pytest.mark.parametrize("b", [3, 4, 5, 6])
def test_identity_lut_gives_top_bits(b):
    rng = np.random.default_rng(b)
    code6 = rng.integers(0, 64, size=(16, 64), dtype=np.uint8)
    W = O.dequant(code6, _identity_luts(16), b)
    # the b-bit code is the top b bits of the 6-bit parent code: integer floor division
    assert np.array_equal(W, (code6 // (1 << (6 - b))).astype(np.float64))


def test_nesting_by_prefix():
    # a weight's b-bit code, extended by its next bit, is its (b+1)-bit code
    rng = np.random.default_rng(7)
    code6 = rng.integers(0, 64, size=(32, 128), dtype=np.uint8)
    for b in range(3, 6):
        cb = O.code_at_bits(code6, b)
        cb1 = O.code_at_bits(code6, b + 1)
        assert np.array_equal(cb1 // 2, cb)
        assert set(np.unique(cb1 - 2 * cb)) <= {0, 1}


def test_constant_rows_and_membership():
    rng = np.random.default_rng(1)
    R, C = 32, 128
    code6 = rng.integers(0, 64, size=(R, C), dtype=np.uint8)
    c = rng.standard_normal(R).astype(np.float16)
    luts = [np.tile(c[:, None], (1, 1 << b)) for b in (3, 4, 5, 6)]
    for b in (3, 4, 5, 6):
        W = O.dequant(code6, luts, b)
        assert np.array_equal(W, np.tile(c.astype(np.float64)[:, None], (1, C)))
    cfg = get_config("tiny")
    ex = make_expert(cfg, 0, seed=0, with_w16=True)
    for b in (3, 4, 5, 6):
        W = O.dequant(ex["code6"][2], ex["lut"][2], b)
        lut = ex["lut"][2][b - 3].astype(np.float64)
        for r in (0, 5, 511):
            assert set(W[r].tolist()) <= set(lut[r].tolist())
    assert np.array_equal(O.dequant(ex["code6"][0], ex["lut"][0], 16, ex["w16"][0]),
                          ex["w16"][0].astype(np.float64))


@pytest.mark.parametrize("R,C", [(16, 64), (32, 256), (48, 320), (16, 448), (64, 704), (16, 1408)])
def test_pack_roundtrip_and_nesting(R, C):
    rng = np.random.default_rng(R + C)
    code6 = rng.integers(0, 64, size=(R, C), dtype=np.uint8)
    planes = O.pack_planes(code6)
    assert len(planes) == 6 and all(p.shape == (R * C // 32,) for p in planes)
    assert np.array_equal(O.unpack_planes(planes, R, C), code6)
    for b in (3, 4, 5, 6):
        assert np.array_equal(O.codes_from_planes(planes[:b], R, C), code6 >> (6 - b))
    # each plane stores exactly the weights' bit (5 - p): popcounts agree
    for p in range(6):
        ones = int(((code6 >> (5 - p)) & 1).sum())
        pc = int(sum(bin(int(v)).count("1") for v in planes[p]))
        assert pc == ones


@pytest.mark.parametrize("C", [64, 256, 320, 704])
def test_single_weight_lands_in_its_tile(C):
    R = 48
    words_per_tile = C // 64 * 32
    for (r, c) in [(0, 0), (17, 63), (47, C - 1), (31, C // 2)]:
        code6 = np.zeros((R, C), dtype=np.uint8)
        code6[r, c] = 32  # only the most significant bit set -> plane 0 only
        planes = O.pack_planes(code6)
        assert all(int(planes[p].sum()) == 0 for p in range(1, 6))
        nz = np.nonzero(planes[0])[0]
        assert nz.size == 1 and bin(int(planes[0][nz[0]])).count("1") == 1
        assert nz[0] // words_per_tile == r // 16
        code6[r, c] = 1  # least significant bit -> plane 5 only
        planes = O.pack_planes(code6)
        assert all(int(planes[p].sum()) == 0 for p in range(5))
        assert np.count_nonzero(planes[5]) == 1


@pytest.mark.parametrize("R,C", [(16, 64), (32, 192), (48, 704)])
def test_f16_pack_roundtrip_and_blocks(R, C):
    rng = np.random.default_rng(R * C)
    w = rng.standard_normal((R, C)).astype(np.float16)
    pk = O.pack_f16(w)
    assert np.array_equal(O.unpack_f16(pk, R, C).view(np.uint16), w.view(np.uint16))
    # every 256-half block is one tile x one 16-column step of one chunk
    blocks = pk.reshape(-1, 256)
    nk = C // 64
    for bi in (0, blocks.shape[0] - 1):
        tau, rest = divmod(bi, nk * 4)
        kappa, s = divmod(rest, 4)
        sub = w[16 * tau:16 * tau + 16, 64 * kappa + 16 * s:64 * kappa + 16 * s + 16]
        assert sorted(blocks[bi].tolist()) == sorted(sub.view(np.uint16).reshape(-1).tolist())


def _probes():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "layout_probes.txt")
    for line in open(path):
        line = line.split("#")[0].split()
        if line:
            yield line


def test_layout_hand_probes():
    n = 0
    for p in _probes():
        if p[0] == "plane":
            R, C, r, c, code, plane, word, bit = map(int, p[1:])
            code6 = np.zeros((R, C), dtype=np.uint8)
            code6[r, c] = code
            planes = O.pack_planes(code6)
            for q in range(6):
                exp = np.zeros(R * C // 32, dtype=np.uint32)
                if q == plane:
                    exp[word] = np.uint32(1) << np.uint32(bit)
                assert np.array_equal(planes[q], exp), (p, q)
        else:
            R, C, r, c, hidx = map(int, p[1:])
            w = np.zeros((R, C), dtype=np.float16)
            w[r, c] = 1.0
            pk = O.pack_f16(w)
            assert np.nonzero(pk)[0].tolist() == [hidx]
        n += 1
    assert n == 7
