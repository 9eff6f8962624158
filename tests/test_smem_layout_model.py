"""A model, on the CPU, of the shared-memory layout the TMA ring holds and of
the mma.sync consumers' reads from it: lane coverage (every element a k-step
needs is read exactly once) and bank conflicts (the number of shared-memory
wavefronts each warp-wide access takes).

Layout: a TMA box lands in 128-byte rows at a 1024-byte-aligned base with
the 128-byte swizzle, so byte c of row r sits at r*128 + ((c//16) ^ (r%8))*16
+ c%16. A tile holds 16 keys of HG consecutive KV heads, row (key*HG + head)
of each slab. The access patterns below restate the consumers' address
arithmetic. Per-head tiles (HG = 1) read without conflicts. Head-group
tiles meet only 8/HG of the eight swizzle phases within one head's rows: the
fp16 tiles' ldmatrix reads take HG wavefronts per phase (2- or 4-way). The
one-byte tiles' 16-byte reads use chunks 2 t4 + ss, one parity class of the
eight chunk positions, so any head grouping leaves them on 4 positions:
8 wavefronts instead of 4 (2-way) for HG = 2 and 4 alike.
"""
import pytest

BANK_BYTES, BANKS = 4, 32


def swizzled(row, byte):
    return row * 128 + (((byte // 16) ^ (row % 8)) * 16) + byte % 16


def wavefronts(accesses):
    """Shared-memory wavefronts for one warp-wide access: `accesses` lists
    (address, width) per lane. Lanes that read the same 4-byte word share it;
    a wavefront serves each bank once."""
    per_bank = {}
    for addr, width in accesses:
        for w in range(addr // BANK_BYTES, (addr + width) // BANK_BYTES):
            per_bank.setdefault(w % BANKS, set()).add(w)
    return max(len(words) for words in per_bank.values())


def ldmatrix_phases(row_addrs):
    """ldmatrix .x4: four phases of eight 16-byte row reads; returns the
    wavefronts of each phase."""
    return [wavefronts([(a, 16) for a in row_addrs[8 * p: 8 * p + 8]]) for p in range(4)]


@pytest.mark.parametrize("HG", [1, 2, 4])
@pytest.mark.parametrize("th", [0, 1, 3])
def test_fp16_k_fragment_reads(HG, th):
    """S^T = K Q^T, fp16 tiles: ldmatrix.x4 of a 16-key x 16-dim A fragment;
    lane l gives row (key = l % 8 + 8 ((l // 8) % 2), head th) and 16-byte
    chunk 2 (ks % 4) + l // 16 of slab ks // 4."""
    if th >= HG:
        pytest.skip("head outside the tile")
    for ks in range(16):  # D = 256: 16 k-steps of 16 dims
        addrs, elems = [], set()
        for lane in range(32):
            key = (lane & 7) + ((lane >> 3) & 1) * 8
            srow = key * HG + th
            slab, chunk = ks >> 2, (ks & 3) * 2 + (lane >> 4)
            addrs.append(slab * 16 * HG * 128 + swizzled(srow, chunk * 16))
            for e in range(8):  # the 8 fp16 values of this 16-byte row read
                elems.add((key, 16 * ks + 8 * (lane >> 4) + e))
        # coverage: the 16 keys x 16 dims of this k-step, each once
        assert elems == {(k, 16 * ks + d) for k in range(16) for d in range(16)}
        assert len(set(addrs)) == 32
        assert max(ldmatrix_phases(addrs)) == HG


@pytest.mark.parametrize("HG", [1, 2, 4])
def test_fp16_v_fragment_reads(HG):
    """O^T += V^T P^T: ldmatrix.x4.trans of 16 keys x 16 dims of V; lane l
    gives row (key = l % 8 + 8 (l // 16), head) and chunk 2 (mt % 4) +
    (l // 8) % 2 of slab mt // 4."""
    for mt in range(16):
        addrs = []
        for lane in range(32):
            key = (lane & 7) + (lane >> 4) * 8
            srow = key * HG
            slab, chunk = mt >> 2, (mt & 3) * 2 + ((lane >> 3) & 1)
            addrs.append(slab * 16 * HG * 128 + swizzled(srow, chunk * 16))
        assert len(set(addrs)) == 32
        assert max(ldmatrix_phases(addrs)) == HG


@pytest.mark.parametrize("HG", [1, 2, 4])
def test_one_byte_k_reads(HG):
    """One-byte tiles: lane (g, t4) reads 16 bytes of rows (key g, head th)
    and (key g + 8, head th) at chunk (2 t4 + ss) of the slab, the dims
    128 slab + 16 (2 t4 + ss) .. +15. The four lanes of a key cover half of
    its 128-byte slab row in each super-step ss and the whole row over the
    two, each byte once."""
    for slab in range(2):
        for rows8 in (0, 8):
            covered = []
            for ss in range(2):
                accesses = []
                for lane in range(32):
                    g, t4 = lane >> 2, lane & 3
                    srow = (g + rows8) * HG
                    chunk = 2 * t4 + ss
                    accesses.append((slab * 16 * HG * 128 + swizzled(srow, chunk * 16), 16))
                    covered += [(g, 16 * chunk + b) for b in range(16)]
                # 512 bytes need at least 4 wavefronts; grouped heads share
                # swizzle phases, and one parity class of chunks leaves 4 of
                # the 8 positions: twice the minimum
                assert wavefronts(accesses) == (4 if HG == 1 else 8)
            assert sorted(covered) == [(g, b) for g in range(8) for b in range(128)]
