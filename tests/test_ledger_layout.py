"""The INT2 ledger layout the CUDA kernels use (LedgerLayout, compiled here
for the host from the kernels' own header) agrees entry for entry with the
tests' statement of it (tests/ledger_codec.py), which the GPU tests use to
read the device ledger; every code bit, scale and zero has exactly one
place, and a code survives the sign / magnitude encoding."""
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


@pytest.mark.parametrize("kind,place", [("k", LC.key_place), ("v", LC.value_place)])
def test_code_places_agree_and_are_a_bijection(dump, kind, place):
    d = dump[kind]
    tok, c = d[:, 0], d[:, 1]
    word, reg, e = place(tok, c)
    sb, mb = LC.code_bits(reg, e)
    assert np.array_equal(d[:, 2], word)
    assert np.array_equal(d[:, 3], sb)
    assert np.array_equal(d[:, 4], mb)
    bits = np.concatenate([word * 32 + sb, word * 32 + mb])
    assert len(np.unique(bits)) == 2 * 128 * 128        # every bit of the 4 KiB used once
    assert bits.min() >= 0 and bits.max() < 4096 * 8


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
                w, reg, e = place(tok, c)
                sb, mb = LC.code_bits(reg, e)
                code = int(q[tok, c])
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
