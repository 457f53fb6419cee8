"""Host checks of the tcgen05 descriptor encoders in ``csrc/kda_sm100.cuh`` (no GPU).

The FlashInfer PR #4262 notes (section 8) print the instruction descriptor of the
fused M128 x N160 update with bf16 A/B, fp32 D and an MN-major B: 0x08290490.  The
encoder must reproduce it; the K-major variants this library uses differ from it in
the B-major bit only.  The core-matrix offsets are checked against a brute-force
rendering of the canonical no-swizzle K-major layout (8-row x 16-byte core matrices).
"""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gated_delta_rule_36_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <initializer_list>
#include "kda_sm100.cuh"
int main() {
    std::printf("%08x\n", kda::make_idesc_bf16_f32(128, 160, true));
    std::printf("%08x %08x %08x\n", kda::make_idesc_bf16_f32(128, 64), kda::make_idesc_bf16_f32(128, 32),
                kda::make_idesc_bf16_f32(128, 160));
    unsigned long long d = kda::make_sdesc_kmajor_noswizzle(0x1a2b0u, 128u, 2048u);
    std::printf("%016llx\n", d);
    for (int kt : {32, 128})
        for (int r = 0; r < 64; ++r)
            for (int k = 0; k < kt; ++k) std::printf("%u\n", kda::core_offset(r, k, kt));
    return 0;
}
"""


@pytest.fixture(scope="module")
def output(tmp_path_factory):
    d = tmp_path_factory.mktemp("desc")
    src = d / "t.cpp"
    src.write_text(PROGRAM)
    exe = d / "t"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()


def test_idesc_matches_printed_value(output):
    assert output[0] == "08290490"


def test_idesc_fields(output):
    g1, g2, g3 = (int(x, 16) for x in output[1:4])
    for val, n in ((g1, 64), (g2, 32), (g3, 160)):
        assert (val >> 4) & 3 == 1            # D = f32
        assert (val >> 7) & 7 == 1            # A = bf16
        assert (val >> 10) & 7 == 1           # B = bf16
        assert (val >> 15) & 3 == 0           # both K-major
        assert ((val >> 17) & 0x3F) << 3 == n
        assert ((val >> 24) & 0x1F) << 4 == 128
    assert g3 | (1 << 16) == 0x08290490


def test_sdesc_fields(output):
    d = int(output[4], 16)
    assert d & 0x3FFF == 0x1a2b0 >> 4
    assert ((d >> 16) & 0x3FFF) << 4 == 128
    assert ((d >> 32) & 0x3FFF) << 4 == 2048
    assert (d >> 46) & 3 == 1
    assert d >> 61 == 0


def test_core_offsets_are_the_canonical_layout(output):
    offs = [int(x) for x in output[5:]]
    pos = 0
    for kt in (32, 128):
        tile = {}
        for r in range(64):
            for k in range(kt):
                tile[(r, k)] = offs[pos]
                pos += 1
        # brute force: core matrix (r // 8, k // 8) stored as 128 contiguous bytes,
        # K-adjacent core matrices 128 B apart, 8-row groups kt / 8 * 128 B apart
        for (r, k), o in tile.items():
            core = (r // 8) * (kt // 8) + (k // 8)
            assert o == core * 128 + (r % 8) * 16 + (k % 8) * 2
        assert sorted(tile.values()) == list(range(0, 64 * kt * 2, 2))
