"""Host-side logic of the streamed validator: batching and the resumable log."""
import json

import pytest

from decode_gemv_sign_gb300 import synth, validate


def test_batches_respect_budget_and_order():
    specs = synth.workload_checkpoint(layers=2)
    budget = 4 << 30
    batches = list(validate._batches(specs, budget))
    flat = [s for b in batches for s in b]
    assert [s.name for s in flat] == [s.name for s in specs]
    for b in batches:
        size = sum(2 * s.n for s in b)
        assert size <= budget or len(b) == 1  # a single tensor larger than the budget goes alone


def test_log_round_trip(tmp_path):
    p = tmp_path / "log.jsonl"
    recs = [{"name": "a", "scheme": 0, "n": 10, "escapes": 1, "serialized_bytes": 100, "entropy_bpw": 12.0,
             "exact": True},
            {"name": "a", "scheme": 1, "n": 10, "escapes": 2, "serialized_bytes": 90, "entropy_bpw": 11.0,
             "exact": True}]
    p.write_text("".join(json.dumps(r) + "\n" for r in recs) + "\n")
    done = validate._read_log(str(p))
    assert set(done) == {("a", 0), ("a", 1)}
    assert done[("a", 1)]["escapes"] == 2
    assert validate._read_log(str(tmp_path / "missing.jsonl")) == {}


def test_log_resumes_after_a_torn_write(tmp_path):
    p = tmp_path / "log.jsonl"
    rec = lambda name, sc: {"name": name, "scheme": sc, "n": 4, "escapes": 0, "serialized_bytes": 8,
                            "entropy_bpw": 12.0, "exact": True}
    good = json.dumps(rec("a", 0)) + "\n" + json.dumps(rec("b", 0)) + "\n"
    # the writer died in the middle of the third record, and (separately) after a record but before its newline
    for tail in (json.dumps(rec("c", 0))[:17], json.dumps(rec("c", 0))):
        p.write_text(good + tail)
        assert set(validate._read_log(str(p))) == {("a", 0), ("b", 0)}
        # reopening drops the unterminated tail; the next record lands on its own line
        with validate._open_log(str(p)) as f:
            f.write(json.dumps(rec("c", 0)) + "\n")
        assert p.read_text() == good + json.dumps(rec("c", 0)) + "\n"
        assert set(validate._read_log(str(p))) == {("a", 0), ("b", 0), ("c", 0)}
    # a damaged line before the end is an error, not something to skip
    p.write_text(json.dumps(rec("a", 0)) + "\n" + "{not json\n" + json.dumps(rec("b", 0)) + "\n")
    with pytest.raises(json.JSONDecodeError):
        validate._read_log(str(p))
    # a log with no complete line yet
    p.write_text('{"name": "a"')
    assert validate._read_log(str(p)) == {}
    with validate._open_log(str(p)) as f:
        pass
    assert p.read_text() == ""


def test_checkpoint_recipe_matches_description():
    specs = synth.workload_checkpoint()
    assert len(specs) == 1923
    assert abs(synth.total_elements(specs) * 2 / 2**30 - 120.0) < 0.01
    shapes = {(s.N, s.K) for s in specs}
    assert shapes == {(151552, 6144), (6144, 6144), (16384, 6144), (6144, 16384), (2048, 6144), (1, 6144)}
    assert max(s.n for s in specs) < 2**32
