"""The selection kernel stages a sequence's keys in shared memory exactly
when its launch reserved the memory for them.  The rule is compiled here for
the host from the kernels' own header: a launch over at most `n` keys per
sequence stages when its longest chunk fits the cap and then reserves that
chunk's bytes; every sequence of the launch (block mode: those with fewer
live blocks too) then has a chunk no longer than the reservation, and a
launch that does not stage reserves nothing and no sequence of it stages
(a shorter sequence whose own chunk would fit must not)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def rows(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("sel") / "select_staging_dump")
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-o", exe,
                    os.path.join(HERE, "select_staging_dump.cu")], check=True,
                   capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.splitlines()
    cap = int(out[-1].split()[1])
    return cap, [tuple(int(x) for x in ln.split()) for ln in out[:-1]]


def _chunk(n, cl):
    return -(-n // cl)


def test_staging_follows_the_launch(rows):
    cap, table = rows
    assert cap > 0
    for cl, n, staged, smem, chunk in table:
        assert chunk == _chunk(n, cl)
        assert staged == (chunk <= cap)
        assert smem == (4 * chunk if staged else 0)
        # every sequence of the launch holds at most n keys: its chunk fits
        # the reservation whenever the kernel stages
        for m in {1, n // 3 + 1, n - 1, n}:
            if 1 <= m <= n and staged:
                assert 4 * _chunk(m, cl) <= smem


def test_a_short_sequence_of_a_long_launch_does_not_stage(rows):
    """The case that faulted under the per-sequence rule: block mode with
    more than 8 x cap live blocks at most, and a sequence with fewer."""
    cap, table = rows
    big = [r for r in table if r[0] == 8 and r[1] > 8 * cap]
    assert big, "the dump covers launches past the cap"
    for cl, n, staged, smem, _ in big:
        assert staged == 0 and smem == 0
    # some of them hold a sequence whose own chunk fits: a per-sequence rule
    # would have staged it into the 0 bytes the launch reserved
    assert any(_chunk(n // 2, cl) <= cap for cl, n, *_ in big)
