"""bench.py host logic on CPU: the traffic record is keyed on the prefill
kernels' code, so a comment edit keeps it and a code edit discards it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = """// header comment
#include <x.h>
/* a block
   comment */
__device__ int f(int a) {  // trailing comment
  return a + 1;   /* inline */
}
"""


def test_source_code_drops_comments_and_blank_lines():
    assert bench.source_code(SRC) == "#include <x.h>\n__device__ int f(int a) {\nreturn a + 1;\n}"


def test_comment_edit_keeps_code_and_code_edit_changes_it():
    commented = SRC.replace("// trailing comment", "// another remark\n\n// more")
    assert bench.source_code(commented) == bench.source_code(SRC)
    edited = SRC.replace("a + 1", "a + 2")
    assert bench.source_code(edited) != bench.source_code(SRC)


def test_traffic_record_matches_current_source_or_is_ignored():
    rec = json.load(open(os.path.join(ROOT, "profiles", "chunk_prefill_traffic.json")))
    traffic = bench.recorded_traffic()
    if rec["kernel_sha"] == bench.kernel_hash():
        assert traffic == float(rec["dram_bytes_per_launch_full_size"])
    else:
        assert traffic is None
