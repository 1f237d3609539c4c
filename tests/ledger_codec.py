"""The INT2 ledger entry's byte layout, restated for the tests: where each
key / value code, scale and zero of a (window, layer, KV head) entry lives.
The entry is laid out for the attention kernel's tensor-core fragments: per
16-token tile, lane 4 g + t owns 4 consecutive code words.  A key word has 8
fields f, each holding two codes (half e) as plain 2-bit numbers at bits
2 f + 16 e (low bit) and 2 f + 16 e + 1; a key's field is 3 (s % 3) + s / 3 for
its k-step s, in word 2 i + h.  A value word holds 8 registers (slot = register
% 8) of two codes (half e), each code as a sign bit at (15 + 16 e + 2 slot) % 32
and a magnitude bit at (6 + 16 e + 2 slot) % 32 (sign: code <= 1; magnitude:
code 0 or 3)."""
import numpy as np

W, D = 128, 128
KC, KS, KZ, VC, VS, VZ, BYTES = 0, 4096, 5120, 6144, 10240, 11264, 12288


def key_field(s):
    return 3 * (s % 3) + s // 3


def key_bit(field, e):
    """Low bit of the key code in half e of a field (the high bit is the next)."""
    return 2 * field + 16 * e


def code_bits(reg, e):
    """(sign bit, magnitude bit) positions of half e of value register reg."""
    slot = reg & 7
    return (15 + 16 * e + 2 * slot) % 32, (6 + 16 * e + 2 * slot) % 32


def key_place(tok, c, d: int = D):
    """Key code (token, channel): token 16 ti + 8 i + g, channel 16 s + 8 h +
    2 t + e sits in field key_field(s) of word 2 i + h of lane 4 g + t, half e.
    Returns (word index among the code words, field, half)."""
    ti, i, g = tok >> 4, (tok >> 3) & 1, tok & 7
    s_, h, t, e = c >> 4, (c >> 3) & 1, (c & 7) >> 1, c & 1
    return ti * d + (4 * g + t) * (d // 32) + 2 * i + h, key_field(s_), e


def value_place(tok, c, d: int = D):
    """Value code (token, channel): token 16 ti + 8 h + 2 t + e, channel
    8 j + g sits in register 2 j + h of lane 4 g + t, half e."""
    ti, h, t, e = tok >> 4, (tok >> 3) & 1, (tok & 7) >> 1, tok & 1
    j, g = c >> 3, c & 7
    reg = 2 * j + h
    return ti * d + (4 * g + t) * (d // 32) + (reg >> 3), reg, e


def key_scale_index(grp, c, d: int = D):
    """fp16 key scale / zero of (32-token group, channel)."""
    return grp * d + ((c & 7) >> 1) * (d // 4) + 4 * (c >> 4) + 2 * ((c >> 3) & 1) + (c & 1)


def value_scale_index(tok, cg, d: int = D):
    """fp16 value scale / zero of (token, 32-channel group)."""
    ng = d // 32
    return (tok >> 4) * 16 * ng + ((tok & 7) >> 1) * 4 * ng + ((tok >> 3) & 1) * 2 * ng + 2 * cg + (tok & 1)


def _key_codes(words, d):
    tok = np.arange(W)[:, None]
    c = np.arange(d)[None, :]
    word, field, e = key_place(tok, c, d)
    return ((words[word] >> key_bit(field, e)) & 3).astype(np.uint8)


def _value_codes(words, d):
    tok = np.arange(W)[:, None]
    c = np.arange(d)[None, :]
    word, reg, e = value_place(tok, c, d)
    sb, mb = code_bits(reg, e)
    x = words[word]
    sign, mag = (x >> sb) & 1, (x >> mb) & 1
    return np.where(sign == 1, np.where(mag == 1, 0, 1), np.where(mag == 1, 3, 2)).astype(np.uint8)


def decode_ledger(entry: np.ndarray, d: int = D):
    """Codes and fp16 scale/zero of one device ledger entry (12288 bytes):
    key codes [token][channel], key scale/zero [group][channel], value codes
    [token][channel], value scale/zero [token][channel group]."""
    kq = _key_codes(entry[KC:KS].view(np.uint32), d)
    vq = _value_codes(entry[VC:VS].view(np.uint32), d)
    kidx = key_scale_index(np.arange(W // 32)[:, None], np.arange(d)[None, :], d)
    vidx = value_scale_index(np.arange(W)[:, None], np.arange(d // 32)[None, :], d)
    ks, kz = entry[KS:KZ].view(np.float16)[kidx], entry[KZ:VC].view(np.float16)[kidx]
    vs, vz = entry[VS:VZ].view(np.float16)[vidx], entry[VZ:BYTES].view(np.float16)[vidx]
    return kq, ks, kz, vq, vs, vz
