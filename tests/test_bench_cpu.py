"""Host logic of bench.py that needs no GPU: the key of the DRAM-traffic record."""
import importlib.util
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_text_ignores_comments_and_layout_but_not_code():
    b = _bench()
    a = "int x = 1;  // one\n/* block\n comment */ float y = x * 2.0f;\n"
    assert b.code_text(a) == b.code_text("int x = 1;\nfloat   y = x * 2.0f;")
    assert b.code_text(a) != b.code_text("int x = 2; float y = x * 2.0f;")


def test_attention_code_hash_is_stable_and_the_record_is_well_formed():
    b = _bench()
    h = b.attention_code_sha256()
    assert re.fullmatch(r"[0-9a-f]{64}", h) and h == b.attention_code_sha256()
    with open(os.path.join(ROOT, "profiles", "attention_traffic.json")) as f:
        rec = json.load(f)
    assert re.fullmatch(r"[0-9a-f]{64}", rec["code_sha256"])
    assert rec["bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert rec["workload"].startswith("H3 Ref2VA block N=152263")


def test_cpu_baseline_record_on_the_tiny_block():
    # all-core and one-core oracle timings, per-row times extrapolated to the block
    from serving_tcgen05_streamed_gb300 import inputs
    b = _bench()
    fp, fa = b.flops(inputs.TINY.n, inputs.TINY.hidden)
    rec = b.cpu_baseline(inputs.TINY, fp, fa, proj_rows=4, attn_rows=2, single_proj_rows=2, single_attn_rows=1)
    assert rec["kind"] == "oracle" and rec["cores"] >= 1 and rec["single_core"]["cores"] == 1
    assert rec["value"] > 0 and rec["single_core"]["value"] > 0
    assert abs(rec["block_s_extrapolated"] - (rec["s_per_projection_row"] + rec["s_per_query_row"]) * 1024) < 1e-9
    assert isinstance(rec["cpu_model"], str) and rec["cpu_model"]


def test_query_chunks_tile_the_rows_and_end_small():
    b = _bench()
    for n in (1, 255, 2048, 2049, 19456, 40000, 152263, 217088):
        ch = b.query_chunks(n)
        assert ch[0][0] == 0 and sum(ln for _, ln in ch) == n
        assert all(a + ln == c for (a, ln), (c, _) in zip(ch, ch[1:]))
        assert all(0 < ln <= b.E2E_OUT_CHUNK for _, ln in ch)
        assert ch[-1][1] <= 2048 or n <= 2048
