"""bench.py's roofline traffic comes from the committed ncu records only
while they match the kernel code they were taken on: a record whose code
hash differs (the kernel changed since the capture) gives null; an edit of
comments or whitespace alone keeps it."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _records():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as fh:
        return json.load(fh)


@pytest.mark.parametrize("key,src", [("attention", "attn.cu"), ("attention_paged", "attn.cu"),
                                     ("attention_int2", "attn_int2.cu")])
def test_records_name_their_source_and_ratios_are_close_to_one(key, src):
    rec = _records()[key]
    assert rec["code_sha256"] is None or len(rec["code_sha256"]) == 64
    path = os.path.join(ROOT, "decoding_kv_cache_split_gb300", "csrc", src)
    current = bench.code_sha256(open(path, encoding="utf-8").read())
    if key == "attention":
        got = bench.ncu_traffic(src, 1000.0)
        expect = rec["bytes_per_token_layer"] * 1000.0
    else:
        got = bench.traffic_ratio(key, src)
        expect = rec["ratio_to_algorithmic"]
        assert 1.0 <= expect < 1.05     # DRAM bytes at most a few % above the algorithmic ones
    if rec["code_sha256"] == current:
        assert got == pytest.approx(expect)
    else:
        assert got is None


def test_a_changed_source_gives_no_traffic(tmp_path, monkeypatch):
    recs = _records()
    for rec in recs.values():
        rec["code_sha256"] = "0" * 64
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.json").write_text(json.dumps(recs))
    csrc = tmp_path / "decoding_kv_cache_split_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("attn.cu", "attn_int2.cu"):
        (csrc / f).write_text("// another kernel\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("attn.cu", 10.0) is None
    assert bench.traffic_ratio("attention_paged", "attn.cu") is None
    assert bench.traffic_ratio("attention_int2", "attn_int2.cu") is None


def test_code_hash_ignores_comments_and_whitespace_only():
    a = 'int a; // note\n/* block */ int  b; const char* s = "//kept";\n'
    b = 'int a;\nint b; const char* s = "//kept";'
    c = 'int a;\nint b; const char* s = "//kept!";'
    d = 'int a;\nint c; const char* s = "//kept";'
    assert bench.code_sha256(a) == bench.code_sha256(b)
    assert bench.code_sha256(b) != bench.code_sha256(c)
    assert bench.code_sha256(b) != bench.code_sha256(d)
