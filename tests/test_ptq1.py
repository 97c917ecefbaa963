"""ptq1_0, the 1.75-bit file: the oracle's definition pinned against the page
("how i made a 27b ternary model ... faster", section *the detour that lost*)
and against the independent pq2_0 packer of the synthetic data."""
import itertools

import numpy as np

import oracle
import synth


def test_threshold_form_all_bytes():
    """The page's two forms of one trit agree on every byte: floor(3 v / 256)
    (the oracle) and (v >= 86) + (v >= 171), v = b * 3^n mod 256."""
    for b in range(256):
        for n in range(5):
            v = (b * 3 ** n) % 256
            assert oracle.ptq1_trit(b, n) == int(v >= 86) + int(v >= 171)


def test_every_tuple_round_trips_and_is_the_smallest_byte():
    decoded = {b: tuple(oracle.ptq1_trit(b, n) for n in range(5)) for b in range(256)}
    for t in itertools.product(range(3), repeat=5):
        b = oracle.ptq1_byte(t)
        assert decoded[b] == t
        assert b == min(c for c, d in decoded.items() if d == t)
    # 243 tuples: every byte decodes to some tuple, so 13 bytes are aliases
    assert len(set(decoded.values())) == 243


def test_hand_worked_block():
    """All w = 0 (u = 1): 25 bytes of trits (1,1,1,1,1) -> q = 121 ->
    ceil(121 * 256 / 243) = 128, and the last byte (1,1,1,0,0) -> q = 117 ->
    ceil(117 * 256 / 243) = 124; the fp16 scale 1.0 = 0x3C00 first."""
    w = np.zeros((1, 128), np.int8)
    sb = np.full((1, 1), 0x3C00, np.uint16)
    blk = oracle.encode_ptq1_0(w, sb)
    assert blk.tolist() == [0x00, 0x3C] + [128] * 25 + [124]
    # one weight at +1 (u = 2): weight 7 is trit 2 of byte 1: q = 121 + 9 = 130
    w[0, 7] = 1
    blk = oracle.encode_ptq1_0(w, sb)
    assert blk[2 + 1] == (130 * 256 + 242) // 243 == 137
    assert [oracle.ptq1_trit(int(blk[3]), n) for n in range(5)] == [1, 1, 2, 1, 1]


def test_size_is_1_75_bits():
    assert oracle.PTQ1_BYTES * 8 / 128 == 1.75
    assert round(1 - oracle.PTQ1_BYTES / oracle.PQ2_BYTES, 2) == 0.18


def test_conversion_matches_the_pq2_0_packer():
    """ptq1_0 -> pq2_0 through the oracle's decoder gives the bytes the
    synthetic-data packer writes for the same weights (random rows, every code
    position and the last byte's padding covered)."""
    for rows, cols, seed in [(3, 128, 1), (17, 512, 2), (64, 1024, 3)]:
        s = synth.seeds(seed)
        codes = synth.ternary_codes(rows, cols, s["weights"])
        scales = synth.group_scales(rows, cols, s["scales"])
        sb = np.ascontiguousarray(scales.astype(np.float16)).view(np.uint16)
        wpt = oracle.encode_ptq1_0(codes.astype(np.int8) - 1, sb)
        assert wpt.size == rows * cols // 128 * 28
        assert np.array_equal(oracle.ptq1_0_to_pq2_0(wpt, rows, cols),
                              synth.pack_pq2_0(codes, scales))


def test_synthetic_ptq1_packer_matches_oracle_encoder():
    """The input generator's ptq1_0 packer (used where only generators may run)
    writes the bytes of the oracle's encoder, which the tests above pin."""
    rows, cols = 9, 640
    s = synth.seeds(5)
    codes = synth.ternary_codes(rows, cols, s["weights"])
    scales = synth.group_scales(rows, cols, s["scales"])
    sb = np.ascontiguousarray(scales.astype(np.float16)).view(np.uint16)
    assert np.array_equal(synth.pack_ptq1_0(codes, scales),
                          oracle.encode_ptq1_0(codes.astype(np.int8) - 1, sb))
