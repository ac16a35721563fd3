"""The tensor-core kernel's on-chip layout, read from its source: shared-memory buffers must
not overlap, must start on the 1024-byte boundary the 128-byte swizzle needs, and must fit
the 227 KB a CTA may have; the TMEM regions must fit the 512 columns one CTA allocates."""
import os
import re

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "linear_attention_prefill_chunked_gb300", "csrc", "kda_prefill_tc.cu")

# bytes of each buffer (tile shapes as the source's layout comments state them)
SMEM_SIZES = {"QK": 2 * 128 * 128, "VB": 2 * 64 * 128, "CB": 3 * 128 * 128, "KG": 128 * 64 * 2,
              "TM": 64 * 64 * 2, "WB": 128 * 64 * 2, "QG": 128 * 64 * 2, "BB": 64 * 64 * 2,
              "KR": 128 * 64 * 2, "AM": 2 * 128 * 128, "PI": 4 * 128 * 4, "NI": 64 * 64 * 2}
TMEM_COLS = {"U": 64, "O": 64, "SB": 64, "S": 128, "AB": 192}


def _consts(prefix):
    src = open(SRC).read()
    return {m.group(1): int(m.group(2)) for m in
            re.finditer(r"constexpr uint32_t " + prefix + r"_(\w+) = (\d+);", src)}


def test_shared_memory_buffers_are_disjoint_aligned_and_fit():
    off = _consts("OFF")
    spans = sorted((off[n], off[n] + SMEM_SIZES[n], n) for n in SMEM_SIZES)
    for (a0, a1, an), (b0, b1, bn) in zip(spans, spans[1:]):
        assert a1 <= b0, f"{an} [{a0}, {a1}) overlaps {bn} at {b0}"
    assert all(off[n] % 1024 == 0 for n in SMEM_SIZES), "swizzled tiles need 1024-byte alignment"
    assert spans[-1][1] <= off["SMALL"], "the control block starts after the last buffer"
    # control block (~2 KB) and the alignment slack must stay within 227 KB per CTA
    assert off["SMALL"] + 2048 + 1024 <= 232448


def test_tmem_regions_are_disjoint_and_fit_512_columns():
    tm = _consts("TM")
    spans = sorted((tm[n], tm[n] + TMEM_COLS[n], n) for n in TMEM_COLS)
    for (a0, a1, an), (b0, b1, bn) in zip(spans, spans[1:]):
        assert a1 <= b0, f"TMEM {an} overlaps {bn}"
    assert spans[-1][1] <= 512
