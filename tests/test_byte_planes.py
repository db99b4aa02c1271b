"""Host check of the byte-permute selection that the input-gradient kernel
uses to turn 4-bit codes into operand pairs from per-block byte planes
(`dequant16_4bit_planes` in csrc/tc_gemm.cu), with the permute's default mode
emulated bit for bit: for every code byte in every position of a code word,
the selected pair is (operand of the high nibble, operand of the low nibble),
the high nibble's in the low half. The kernel's output is pinned on the GPU
by tests/test_operands_gpu.py; this pins the selector constants on the CPU."""
import numpy as np


def prmt(a, b, s):
    """PTX prmt.b32 default mode: result byte i = byte (s >> 4 i) & 7 of
    {b, a}, replaced by the sign of that byte when bit 3 of the nibble is set."""
    pool = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    r = 0
    for i in range(4):
        sel = (s >> (4 * i)) & 0xF
        byte = pool[sel & 7]
        if sel & 8:
            byte = 0xFF if byte & 0x80 else 0
        r |= byte << (8 * i)
    return r


def planes(ops):
    """Byte planes of 16 16-bit operands as the kernel builds them from the
    packed pairs (op 2k low, op 2k + 1 high)."""
    pair = [ops[2 * k] | (ops[2 * k + 1] << 16) for k in range(8)]
    lo = [prmt(pair[2 * q], pair[2 * q + 1], 0x6420) for q in range(4)]
    hi = [prmt(pair[2 * q], pair[2 * q + 1], 0x7531) for q in range(4)]
    return lo, hi


def select_word(w, lo, hi):
    """The four operand words of one 32-bit code word (bytes 0..3)."""
    m = w & 0x77777777
    s = ((w >> 1) & 0x44444444) | 0x32103210
    out = []
    for hf in range(2):
        mh, sh = m >> (16 * hf), s >> (16 * hf)
        l_ = prmt(prmt(lo[0], lo[1], mh), prmt(lo[2], lo[3], mh), sh)
        h_ = prmt(prmt(hi[0], hi[1], mh), prmt(hi[2], hi[3], mh), sh)
        out += [prmt(l_, h_, 0x4051), prmt(l_, h_, 0x6273)]
    return out


def test_every_code_byte_in_every_position_selects_its_pair():
    rng = np.random.default_rng(3)
    for _ in range(4):
        ops = [int(v) for v in rng.integers(0, 1 << 16, 16)]
        lo, hi = planes(ops)
        for pos in range(4):
            for byte in range(256):
                fill = int(rng.integers(0, 1 << 32))
                w = (fill & ~(0xFF << (8 * pos))) | (byte << (8 * pos))
                got = select_word(w, lo, hi)[pos]
                assert got == ops[byte >> 4] | (ops[byte & 15] << 16), (pos, byte)


def test_selectors_never_set_the_sign_replicate_bit():
    for w in (0, 0xFFFFFFFF, 0x88888888, 0x77777777, 0xF0F0F0F0):
        m = w & 0x77777777
        s = ((w >> 1) & 0x44444444) | 0x32103210
        for v in (m, s, 0x6420, 0x7531, 0x4051, 0x6273):
            assert all(((v >> (4 * i)) & 8) == 0 for i in range(8))
