"""The INT2 ledger layout the CUDA kernels use (LedgerLayout, compiled here
for the host from the kernels' own header) agrees entry for entry with the
tests' statement of it (tests/ledger_codec.py), which the GPU tests use to
read the device ledger; every code bit, scale and zero has exactly one
place, a value code survives the sign / magnitude encoding, and the attention
kernel's key field extraction (a shift by 6 (f / 3) and a mask) gives every key
register the bf16 pair code * 2^(2 (f % 3)) * 2^-133, one scale class per
k-step."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import ledger_codec as LC

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def dump(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("ledger") / "ledger_layout_dump")
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-o", exe,
                    os.path.join(HERE, "ledger_layout_dump.cu")], check=True,
                   capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    rows = {}
    for line in out.splitlines():
        f = line.split()
        rows.setdefault(f[0], []).append([int(x) for x in f[1:]])
    return {k: np.array(v) for k, v in rows.items()}


def test_offsets(dump):
    assert dump["offsets"][0].tolist() == [LC.KC, LC.KS, LC.KZ, LC.VC, LC.VS, LC.VZ, LC.BYTES]


def test_key_places_agree_and_are_a_bijection(dump):
    d = dump["k"]
    tok, c = d[:, 0], d[:, 1]
    word, field, e = LC.key_place(tok, c)
    assert np.array_equal(d[:, 2], word)
    assert np.array_equal(d[:, 3], field)
    assert np.array_equal(d[:, 4], LC.key_bit(field, e))
    lo = word * 32 + LC.key_bit(field, e)
    bits = np.concatenate([lo, lo + 1])
    assert len(np.unique(bits)) == 2 * 128 * 128        # every bit of the 4 KiB used once
    assert bits.min() >= 0 and bits.max() < 4096 * 8


def test_value_places_agree_and_are_a_bijection(dump):
    d = dump["v"]
    tok, c = d[:, 0], d[:, 1]
    word, reg, e = LC.value_place(tok, c)
    sb, mb = LC.code_bits(reg, e)
    assert np.array_equal(d[:, 2], word)
    assert np.array_equal(d[:, 3], sb)
    assert np.array_equal(d[:, 4], mb)
    bits = np.concatenate([word * 32 + sb, word * 32 + mb])
    assert len(np.unique(bits)) == 2 * 128 * 128
    assert bits.min() >= 0 and bits.max() < 4096 * 8


def _bf16_value(bits16):
    return (np.asarray(bits16, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_key_field_extraction_gives_the_scaled_codes():
    """The kernel's register of key field f: the word shifted right by
    6 (f / 3), masked to bits 2 (f % 3), +1 of each half: both bf16 halves
    are the code times 2^(2 (f % 3)) 2^-133, exactly (subnormals); the fields
    of k-steps 0-2, 3-5 and 6-7 are classes 0, 1 and 2."""
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 4, (1000, 8, 2))
    words = np.zeros(1000, np.uint64)
    for f in range(8):
        for e in range(2):
            words |= codes[:, f, e].astype(np.uint64) << np.uint64(LC.key_bit(f, e))
    words = words.astype(np.uint32)
    for f in range(8):
        reg = (words >> np.uint32(6 * (f // 3))) & np.uint32(0x00030003 << (2 * (f % 3)))
        for e in range(2):
            half = (reg >> np.uint32(16 * e)) & np.uint32(0xFFFF)
            want = codes[:, f, e] * 2.0 ** (2 * (f % 3)) * 2.0 ** -133
            assert np.array_equal(_bf16_value(half), want)
    assert [LC.key_field(s) % 3 for s in range(8)] == [0, 0, 0, 1, 1, 1, 2, 2]
    assert sorted(LC.key_field(s) for s in range(8)) == list(range(8))


def test_scale_indices_agree_and_are_permutations(dump):
    ks = dump["ks"]
    assert np.array_equal(ks[:, 2], LC.key_scale_index(ks[:, 0], ks[:, 1]))
    assert sorted(ks[:, 2].tolist()) == list(range(512))
    vs = dump["vs"]
    assert np.array_equal(vs[:, 2], LC.value_scale_index(vs[:, 0], vs[:, 1]))
    assert sorted(vs[:, 2].tolist()) == list(range(512))


def test_code_encoding_round_trips(dump):
    for c, sign, mag, back in dump["code"]:
        assert back == c
        assert sign == (c <= 1) and mag == (c in (0, 3))


def test_decoder_reads_an_entry_written_by_the_placement():
    """Encode random codes / scales with the placements, decode with the
    GPU tests' reader: the round trip is the identity."""
    rng = np.random.default_rng(5)
    kq = rng.integers(0, 4, (128, 128))
    vq = rng.integers(0, 4, (128, 128))
    ks = rng.standard_normal((4, 128)).astype(np.float16)
    vs = rng.standard_normal((128, 4)).astype(np.float16)
    entry = np.zeros(LC.BYTES, np.uint8)
    for base, q, place in ((LC.KC, kq, LC.key_place), (LC.VC, vq, LC.value_place)):
        words = np.zeros(1024, np.uint32)
        for tok in range(128):
            for c in range(128):
                code = int(q[tok, c])
                if place is LC.key_place:
                    w, f, e = place(tok, c)
                    words[w] |= np.uint32(code << int(LC.key_bit(f, e)))
                else:
                    w, reg, e = place(tok, c)
                    sb, mb = LC.code_bits(reg, e)
                    words[w] |= np.uint32((int(code <= 1) << sb) | (int(code in (0, 3)) << mb))
        entry[base:base + 4096] = words.view(np.uint8)
    k16 = entry[LC.KS:LC.KZ].view(np.float16)
    for grp in range(4):
        for c in range(128):
            k16[LC.key_scale_index(grp, c)] = ks[grp, c]
    v16 = entry[LC.VS:LC.VZ].view(np.float16)
    for tok in range(128):
        for cg in range(4):
            v16[LC.value_scale_index(tok, cg)] = vs[tok, cg]
    dk, dks, _, dv, dvs, _ = LC.decode_ledger(entry)
    assert np.array_equal(dk, kq) and np.array_equal(dv, vq)
    assert np.array_equal(dks, ks) and np.array_equal(dvs, vs)
