"""Pins for the pipeline-trace analysis in attention_forward_tma_gb300/trace.py: the
tensor-pipe occupancy model and the merged per-role timeline, on hand-made stamp lists
whose answers follow from the model's definition (no GPU)."""
import importlib
import os


def _trace_module():
    # importing the module selects the tracing build for later library loads in this
    # process; the CPU tests keep the plain build
    old = os.environ.get("FA_GB300_TRACE")
    try:
        return importlib.import_module("attention_forward_tma_gb300.trace")
    finally:
        if old is None:
            os.environ.pop("FA_GB300_TRACE", None)
        else:
            os.environ["FA_GB300_TRACE"] = old


def test_pipe_model_charges_idle_time_to_the_preceding_wait():
    T = _trace_module()
    mma = [(0, "IssueBegin", 0), (560, "S0", 5),                        # 8 MMAs: busy [0, 568)
           (700, "PO1", 5), (800, "IssueBegin", 0), (900, "PV1a", 5),   # idle [568, 800) after PO1; busy to 1226
           (950, "IssueBegin", 0), (1000, "PV1b", 5),                   # queued behind PV1a: busy to 1368
           (1500, "IssueBegin", 0), (1510, "S1", 4)]                    # idle [1368, 1500), no wait passed
    m = T.pipe_model({"mma": mma}, mma_cycles=71)
    assert m["busy"] == 71 * 24
    assert m["span"] == 1500 + 8 * 71
    assert m["idle"] == {"PO1": [232], "issue": [132]}
    assert m["issue"] == {"S0": [560], "PV1a": [100], "PV1b": [50], "S1": [10]}


def test_pipe_model_without_idle_time():
    T = _trace_module()
    mma = [(0, "IssueBegin", 0), (400, "PV0a", 1), (420, "P2_0", 1), (430, "IssueBegin", 0), (431, "PV0b", 1)]
    m = T.pipe_model({"mma": mma}, mma_cycles=100)
    assert m["idle"] == {}
    assert m["busy"] == m["span"] == 800


def test_timeline_merges_roles_in_clock_order():
    T = _trace_module()
    roles = {"mma": [(5, "S1", 2), (10, "S0", 3), (30, "PO0", 3)],
             "softmax0": [(20, "SFull", 3), (40, "Half1", 3)],
             "correction": [(25, "CorrFull0", 3)]}
    assert T.timeline(roles, start=1, count=4) == [(0, "mma", "S0", 3), (10, "softmax0", "SFull", 3),
                                                    (15, "correction", "CorrFull0", 3), (20, "mma", "PO0", 3)]
    assert T.timeline({"mma": []}, 0, 5) == []
