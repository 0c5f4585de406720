"""The seeded generators reproduce the streams printed on the pages."""
import numpy as np

import synth


def test_lcg_bytes_follow_fill_quant_bytes():
    # cera 0.4.0 examples/wgpu_gemm_bench.rs, fn fill_quant_bytes, seeded with 1
    s, want = 1, []
    for i in range(4096):
        s = (s * 1664525 + 1013904223) & 0xFFFFFFFF
        b = (s >> 16) & 0xFF
        want.append(b & 0xBF if i % 2 == 1 else b)
    assert synth.lcg_bytes(1, 4096).tolist() == want
    # odd offsets never carry bit 6 (f16 scale high bytes stay finite); even do
    got = synth.lcg_bytes(1, 1 << 16)
    assert not np.any(got[1::2] & 0x40)
    assert np.any(got[0::2] & 0x40)
    assert np.any(got[1::2] & 0x80)  # the sign bit is kept


def test_vecf_follows_xorshift64():
    # memra-engine 0.128.0 moe_rows_ceiling_bench.rs, fn vecf
    mask = (1 << 64) - 1
    s = ((2 * 0x9E3779B97F4A7C15) & mask) | 1
    want = []
    for _ in range(2048):
        s ^= (s << 13) & mask
        s ^= s >> 7
        s ^= (s << 17) & mask
        want.append(np.float32((np.float32(s >> 40) / np.float32(1 << 24) - np.float32(0.5)) * np.float32(2.0)))
    got = synth.vecf(2, 2048)
    assert np.array_equal(got, np.array(want, np.float32))
    big = synth.vecf(2, 1 << 18)
    assert big.min() >= -1.0 and big.max() < 1.0
    assert abs(float(big.mean())) < 0.01


def test_nvfp4_rows_follow_synth_rows():
    # memra-engine 0.128.0 moe_rows_ceiling_bench.rs, struct Lcg / fn synth_rows
    s, want = 0x8181, []
    for _g in range(2 * 4096 // 64):
        for i in range(36):
            s = (s * 1664525 + 1013904223) & 0xFFFFFFFF
            b = s >> 24
            want.append((b & 7) | 0x38 if i < 4 else b)
    assert synth.nvfp4_rows(0x8181, 2, 4096).tolist() == want


def test_matrix_seeds_are_distinct():
    seeds = {synth.nvfp4_matrix_seed(c, j, p) for c in range(4) for j in range(8) for p in range(2)}
    assert len(seeds) == 64
