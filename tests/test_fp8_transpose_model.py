"""Host-side model of attn_fp8_transpose_v's lane arithmetic (no GPU).

The kernel writes Vᵀ [B, Hkv, 64, Lp] (keys contiguous, Lp = L rounded up to 16,
keys L .. Lp - 1 zero) from V [B, L, Hkv, 64] in e4m3 bytes: a CTA of 4 warps per
128 keys, warp w moving bytes 16w .. 16w + 15 of d, lane l keys 4l .. 4l + 3. A lane
loads its four keys' 16-byte pieces, transposes each 4 x 4 byte block with byte
permutes and stores one 32-bit word per d row. This test replays exactly those
index and permute steps (the permute as its documented byte selection) and
compares the result with numpy's transpose; every output byte must be written once.
"""
import numpy as np
import pytest


def byte_perm(x, y, sel):
    """Byte n of the result is byte (sel >> 4n) & 7 of the eight bytes y:x (x = 0..3)."""
    src = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    return sum(src[(sel >> (4 * n)) & 7] << (8 * n) for n in range(4))


def transpose_model(v, Lp):
    B, L, Hkv, _ = v.shape
    vt = np.full((B, Hkv, 64, Lp), 0xAB, dtype=np.uint8)  # poison: every byte must be written
    written = np.zeros(vt.shape, dtype=np.int32)
    flat = v.reshape(-1)
    for b in range(B):
        for g in range(Hkv):
            for bx in range((Lp + 127) // 128):
                for w in range(4):
                    for lane in range(32):
                        k = bx * 128 + 4 * lane
                        if k >= Lp:
                            continue
                        a = [[0] * 4 for _ in range(4)]
                        for i in range(4):
                            if k + i < L:
                                off = ((b * L + k + i) * Hkv + g) * 64 + 16 * w
                                for q in range(4):
                                    a[i][q] = int.from_bytes(flat[off + 4 * q:off + 4 * q + 4].tobytes(), "little")
                        for q in range(4):
                            t0 = byte_perm(a[0][q], a[1][q], 0x5140)
                            t1 = byte_perm(a[2][q], a[3][q], 0x5140)
                            t2 = byte_perm(a[0][q], a[1][q], 0x7362)
                            t3 = byte_perm(a[2][q], a[3][q], 0x7362)
                            col = [byte_perm(t0, t1, 0x5410), byte_perm(t0, t1, 0x7632),
                                   byte_perm(t2, t3, 0x5410), byte_perm(t2, t3, 0x7632)]
                            for e in range(4):
                                d = 16 * w + 4 * q + e
                                vt[b, g, d, k:k + 4] = np.frombuffer(col[e].to_bytes(4, "little"), dtype=np.uint8)
                                written[b, g, d, k:k + 4] += 1
    return vt, written


@pytest.mark.parametrize("B,L,Hkv", [(1, 1, 1), (1, 127, 2), (2, 129, 1), (1, 300, 3), (1, 1000, 1)])
def test_transpose_model_matches_numpy(B, L, Hkv):
    rng = np.random.default_rng(L * 7 + Hkv)
    v = rng.integers(0, 256, size=(B, L, Hkv, 64), dtype=np.uint8)
    Lp = (L + 15) // 16 * 16
    vt, written = transpose_model(v, Lp)
    assert (written == 1).all()
    want = np.zeros((B, Hkv, 64, Lp), dtype=np.uint8)
    want[..., :L] = v.transpose(0, 2, 3, 1)
    assert np.array_equal(vt, want)


def test_a_wrong_selector_is_caught():
    """Swapping two selectors of the second permute stage breaks the transpose."""
    a = [0x03020100, 0x13121110, 0x23222120, 0x33323130]  # byte j of key i = 16 i + j
    t0, t1 = byte_perm(a[0], a[1], 0x5140), byte_perm(a[2], a[3], 0x5140)
    good = byte_perm(t0, t1, 0x5410)
    assert good == 0x30201000  # byte 0 of keys 0, 1, 2, 3
    assert byte_perm(t0, t1, 0x7632) != good
