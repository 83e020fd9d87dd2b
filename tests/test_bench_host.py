"""bench.py host logic that needs no GPU: the code hash that keys the measured DRAM traffic, and
the algorithmic work of a step (what the pages define, checked against closed forms)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_hash_ignores_comments_only(bench):
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    assert bench._code_only(code) == bench._code_only(
        "// a header\nint f(int x) {\n  /* a\n     block */ return x + 1;\n\n}\n")
    assert bench._code_only(code) != bench._code_only(code.replace("x + 1", "x + 2"))


def test_known_traffic_matches_current_code(bench):
    """The traffic table names the current code's hash (or the figures read null)."""
    h = bench.kernel_sources_hash()
    assert any(key[1] == h for key in bench.KNOWN_TRAFFIC), h


def test_work_of_closed_forms(bench):
    """Decode bytes and prefill FLOPs of a step against the definitions: a decode of c cached
    tokens reads (c + 1) keys of K and V per kv head; a fresh prefill of q tokens does
    4 nh hd q (q + 1) / 2 FLOPs over the visible keys."""
    nh, nkv, hd, B = 32, 8, 128, 16
    w = bench.work_of([(100, 1)], nh, nkv, hd, B, 1, 1, 1, 1, 4096)
    assert w["decode_bytes"] >= 101 * 2 * nkv * hd * 2
    assert w["prefill_flops"] == 0
    w = bench.work_of([(0, 200)], nh, nkv, hd, B, 200, 200, 1, 1, 4096)
    assert w["prefill_flops"] == 4 * nh * hd * (200 * 201 // 2)
