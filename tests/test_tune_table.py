"""The library's measured launch table (csrc/qmv_tune_table.h) is exactly what
the committed tuning records generate, so a record edited without regenerating
the table, or a table edited by hand, fails here (no GPU needed)."""
import glob
import os

from weight_quantized_decode_gb300 import tune

PKG = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "weight_quantized_decode_gb300")


def test_launch_table_matches_the_tuning_records(tmp_path):
    out = tmp_path / "qmv_tune_table.h"
    tune.emit_header(sorted(glob.glob(os.path.join(PKG, "tuning", "*.json"))), str(out))
    with open(os.path.join(PKG, "csrc", "qmv_tune_table.h")) as f:
        committed = f.read()
    assert out.read_text() == committed


def test_table_ids_match_the_planner():
    # the planner looks entries up by these ids (plain formats 0..2, Q8_1 forms 3 and 4)
    with open(os.path.join(PKG, "csrc", "qmv_api.cu")) as f:
        src = f.read()
    assert "tune_lookup(p.xq8 ? (fmt == kQ8_0 ? 4 : 3) : fmt" in src
    assert tune.TABLE_IDS == {"q4_0": 0, "q8_0": 1, "q2w": 2, "q4_0_q8_1": 3, "q8_0_q8_1": 4}
