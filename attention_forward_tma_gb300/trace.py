"""Pipeline traces from the tracing build of the library (libfa_gb300_trace.so).

python -m attention_forward_tma_gb300.trace [--workload NAME] [--ctas N] [--json FILE] [--pass fwd|bwd]

Runs one attention forward (or backward) of a synthetic workload with clock
stamps at every hand-off of the pipeline (TMA issue, MMA issue, softmax phases,
correction and epilogue; for the backward: Q/dO loads, the five products, the
P and dS phases and the dQ reduce) for the first N CTAs, then prints per-role
cycle statistics. Stamps are SM clock cycles (the 32-bit clock, unwrapped) of the
CTA's own SM.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

os.environ["FA_GB300_TRACE"] = "1"

EVENTS = {1: "Q0", 2: "K", 3: "Q1", 4: "V", 10: "S0", 11: "S1", 12: "PO0", 13: "PV0a", 14: "P2_0", 15: "PV0b",
          16: "PO1", 17: "PV1a", 18: "P2_1", 19: "PV1b", 20: "KVfull_V", 21: "KVfull_K", 30: "SFull", 31: "SMax",
          32: "Mail", 33: "Half1", 34: "Half2", 35: "Stats", 40: "CorrFull0", 41: "CorrFull1", 42: "CorrDone0",
          43: "CorrDone1", 44: "EpiStart0", 45: "EpiStart1", 46: "EpiEnd0", 47: "EpiEnd1", 48: "Task",
          50: "IssueBegin", 60: "QLoad", 61: "dV", 62: "S", 63: "dKdQ", 64: "dP", 70: "SFull", 71: "PReady",
          72: "dPFull", 73: "dSReady", 80: "dQFull", 81: "dPEmpty", 82: "Staged", 83: "Reduced"}
ROLES = ["producer", "mma", "softmax0", "softmax1", "correction"]


last_rescales = (0, 0)   # forward of the last capture(): (row updates from later key blocks, rescales)


def capture(run, ctas: int = 2):
    """Call run() (which launches fa_fwd / fa_fwd_varlen) with tracing on; return decoded events
    as {cta: {role: [(clock, event, block), ...]}}. For the forward, last_rescales then
    holds the softmax rows' updates from a later key block over every CTA and how many of
    them moved the row's reference (an O rescale under the delayed-rescale rule)."""
    import ctypes

    import numpy as np
    import torch

    from . import library
    lib = library()
    roles, slots = ctypes.c_int(), ctypes.c_int()
    lib.fa_trace_layout(ctypes.byref(roles), ctypes.byref(slots))
    stamps = ctas * roles.value * slots.value
    buf = torch.zeros(stamps + 2, dtype=torch.int64, device="cuda")   # + the forward's rescale counters
    st = lib.fa_trace_configure(buf.data_ptr(), ctas)
    if st != 0:
        raise RuntimeError(f"fa_trace_configure failed with status {st} (not a tracing build?)")
    try:
        run()
        torch.cuda.synchronize()
    finally:
        lib.fa_trace_configure(None, 0)
    words = buf.cpu().numpy().view(np.uint64)
    global last_rescales
    last_rescales = (int(words[stamps]), int(words[stamps + 1]))
    raw = words[:stamps].reshape(ctas, roles.value, slots.value)
    out = {}
    for c in range(ctas):
        out[c] = {}
        for r in range(roles.value):
            ev = []
            high = 0          # the 32-bit clock wraps every 2^32 cycles: unwrap in order
            last = None
            for word in raw[c, r]:
                word = int(word)
                if word == 0:
                    break
                clk = word >> 32
                if last is not None and clk < last:
                    high += 1 << 32
                last = clk
                code, blk = (word >> 24) & 0xFF, word & 0xFFFFFF
                if blk >= 1 << 23:
                    blk -= 1 << 24
                ev.append((high + clk, EVENTS.get(code, str(code)), blk))
            out[c][ROLES[r]] = ev
    return out


def _pairs(events, a, b):
    """Cycle gaps from each event a to the next event b."""
    out, start = [], None
    for clk, name, _ in events:
        if name == a:
            start = clk
        elif name == b and start is not None:
            out.append(clk - start)
            start = None
    return out


def summarize(trace) -> dict:
    res = {}
    for c, roles in trace.items():
        t0 = min((ev[0][0] for ev in roles.values() if ev), default=0)
        d = {"span_cycles": max((ev[-1][0] for ev in roles.values() if ev), default=0) - t0}
        for t in (0, 1):
            ev = roles[f"softmax{t}"]
            d[f"softmax{t}_sfull_to_half2"] = _pairs(ev, "SFull", "Half2")
            d[f"softmax{t}_sfull_to_max"] = _pairs(ev, "SFull", "SMax")
            d[f"softmax{t}_half1_to_half2"] = _pairs(ev, "Half1", "Half2")
            d[f"softmax{t}_half2_to_next_sfull"] = _pairs(ev, "Half2", "SFull")
        m = roles["mma"]
        d["mma_wait_po0"] = _pairs(m, "PV1b", "PO0")
        d["mma_wait_po1"] = _pairs(m, "S0", "PO1")
        d["mma_wait_p2_0"] = _pairs(m, "PV0a", "P2_0")
        d["mma_wait_p2_1"] = _pairs(m, "PV1a", "P2_1")
        s0 = [clk for clk, name, _ in m if name == "S0"]
        d["mma_s0_period"] = [b - a for a, b in zip(s0, s0[1:])]
        cor = roles["correction"]
        d["epilogue"] = _pairs(cor, "EpiStart0", "EpiEnd1")
        res[c] = d
    return res


def _gaps(events, a, b):
    """Per step (the event's block field): cycles from event a to event b of the same step."""
    ta = {blk: clk for clk, name, blk in events if name == a}
    return [clk - ta[blk] for clk, name, blk in events if name == b and blk in ta]


def _period(events, a):
    t = [clk for clk, name, _ in events if name == a]
    return [y - x for x, y in zip(t, t[1:])]


def summarize_bwd(trace) -> dict:
    res = {}
    for c, roles in trace.items():
        m, s0, g = roles["mma"], roles["softmax0"], roles["correction"]
        d = {"steps": len([1 for _, n_, _ in m if n_ == "dV"])}
        d["step_period(dSReady)"] = _period(s0, "dSReady")
        d["mma_dV_to_S(next)"] = _gaps_shift(m, "dV", "S", 1)
        d["mma_dV_to_dKdQ"] = _gaps(m, "dV", "dKdQ")
        d["mma_dKdQ_to_dP(next)"] = _gaps_shift(m, "dKdQ", "dP", 1)
        d["wg0_SFull_to_PReady"] = _gaps(s0, "SFull", "PReady")
        d["wg0_PReady_to_dPFull"] = _gaps(s0, "PReady", "dPFull")
        d["wg0_dPFull_to_dSReady"] = _gaps(s0, "dPFull", "dSReady")
        d["wg2_dQFull_to_dPEmpty"] = _gaps(g, "dQFull", "dPEmpty")
        d["wg2_dQFull_to_Staged"] = _gaps(g, "dQFull", "Staged")
        d["wg2_Staged_to_Reduced"] = _gaps(g, "Staged", "Reduced")
        d["dSReady_to_dQFull"] = _cross(s0, "dSReady", g, "dQFull")
        d["dPEmpty_to_dPFull(next)"] = _cross(g, "dPEmpty", s0, "dPFull", 1)
        d["Reduced_to_QLoad(k+2)"] = _cross(g, "Reduced", roles["producer"], "QLoad", 2)
        d["QLoad_to_SFull"] = _cross(roles["producer"], "QLoad", s0, "SFull")
        res[c] = d
    return res


def _gaps_shift(events, a, b, shift):
    ta = {blk: clk for clk, name, blk in events if name == a}
    return [clk - ta[blk - shift] for clk, name, blk in events if name == b and blk - shift in ta]


def _cross(ea, a, eb, b, shift=0):
    ta = {blk: clk for clk, name, blk in ea if name == a}
    return [clk - ta[blk - shift] for clk, name, blk in eb if name == b and blk - shift in ta]


# tcgen05.mma M128 N128 K16 (bf16/fp16 in, fp32 accumulate) measured on a GB300 by a
# one-warp issue probe: 71 cycles with both operands in shared memory, 68 with A in
# tensor memory. Products per group of the forward's MMA warp: QK^T is 8 K16 steps
# over d = 128, PV 6 + 2 steps over the 96 + 32 columns of P.
MMA_CYCLES = 71.0
FWD_GROUP_MMAS = {"S0": 8, "S1": 8, "PV0a": 6, "PV1a": 6, "PV0b": 2, "PV1b": 2}
FWD_WAITS = ("PO0", "PO1", "P2_0", "P2_1", "KVfull_K", "KVfull_V")


def pipe_model(roles, mma_cycles: float = MMA_CYCLES, group_mmas=None) -> dict:
    """Tensor-pipe occupancy of one CTA from its MMA warp's stamps (forward, d = 128).

    Each issue group (IssueBegin ... the group's end stamp) is taken to enter the pipe
    at its IssueBegin stamp, or when the pipe finishes the previous group if that is
    later, and to keep it busy for (its MMAs) x mma_cycles. Time the pipe spends idle
    before a group is charged to the wait the MMA warp passed just before that group
    ("issue" when it passed none: the commit and bookkeeping between two groups)."""
    group_mmas = group_mmas or FWD_GROUP_MMAS
    ev = roles["mma"]
    free = t_first = None
    busy = 0.0
    idle, issue = {}, {}
    last_wait = None
    for i, (clk, name, _) in enumerate(ev):
        if name in FWD_WAITS:
            last_wait = name
        if name != "IssueBegin":
            continue
        j = i + 1
        while j < len(ev) and ev[j][1] not in group_mmas:
            j += 1
        if j == len(ev):
            break
        n = group_mmas[ev[j][1]]
        issue.setdefault(ev[j][1], []).append(ev[j][0] - clk)
        if free is None:
            free = t_first = clk
        if clk > free:
            idle.setdefault(last_wait or "issue", []).append(clk - free)
            free = clk
        free += n * mma_cycles
        busy += n * mma_cycles
        last_wait = None
    span = (free - t_first) if free is not None else 0.0
    return {"span": span, "busy": busy, "idle": idle, "issue": issue}


def timeline(roles, start: int = 0, count: int = 60):
    """The CTA's stamps of every role merged in clock order: `count` of them from the
    `start`-th stamp of the MMA warp on, as (cycles since that stamp, role, event, block)."""
    merged = sorted((clk, role, name, blk) for role, ev in roles.items() for clk, name, blk in ev)
    mma = roles["mma"]
    if not mma:
        return []
    t0 = mma[min(start, len(mma) - 1)][0]
    out = [(clk - t0, role, name, blk) for clk, role, name, blk in merged if clk >= t0]
    return out[:count]


def _fmt(v):
    if isinstance(v, list):
        if not v:
            return "-"
        return f"n={len(v):3d} median={statistics.median(v):8.0f} min={min(v):7d} max={max(v):8d}"
    return str(v)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c4_b1h32n16384d128_causal_spiky")
    ap.add_argument("--ctas", type=int, default=2)
    ap.add_argument("--json", default=None)
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"])
    ap.add_argument("--timeline", type=int, default=0, metavar="N",
                    help="print N merged stamps of CTA 0 from its MMA warp's --timeline-from-th stamp on")
    ap.add_argument("--timeline-from", type=int, default=200, metavar="I")
    ap.add_argument("--pipe", action="store_true",
                    help="forward: modelled tensor-pipe occupancy and idle time by the preceding wait")
    a = ap.parse_args()
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import numpy as np
    import torch

    import fa_inputs

    from . import fa_fwd, fa_fwd_varlen
    w = fa_inputs.WORKLOADS[a.workload]
    x = fa_inputs.make_workload(w)

    def dev(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
    if a.which == "bwd":
        from . import fa_bwd
        dout = dev(fa_inputs.make_qkv(w.B, w.N, w.H, w.d, w.seed + 1000, dtype=w.dtype)[0])
        o, lse = fa_fwd(q, k, v, scale=w.scale, causal=w.causal)
        run = lambda: fa_bwd(q, k, v, o, dout, lse, scale=w.scale, causal=w.causal)  # noqa: E731
    elif w.varlen:
        cu = torch.from_numpy(x["cu_seqlens"]).cuda()
        run = lambda: fa_fwd_varlen(q, k, v, cu, int(x["lengths"].max()), scale=w.scale, causal=w.causal)  # noqa: E731
    else:
        run = lambda: fa_fwd(q, k, v, scale=w.scale, causal=w.causal)  # noqa: E731
    run()
    torch.cuda.synchronize()
    tr = capture(run, a.ctas)
    if a.json:
        with open(a.json, "w") as f:
            json.dump({str(c): r for c, r in tr.items()}, f)
    if a.which == "fwd":
        upd, resc = last_rescales
        print(f"row updates from a later key block: {upd}, of which rescaled O (tau = 8): {resc} "
              f"({100.0 * resc / max(upd, 1):.3f} %)")
    for c, d in (summarize_bwd(tr) if a.which == "bwd" else summarize(tr)).items():
        print(f"CTA {c}")
        for key, val in d.items():
            print(f"  {key:28s} {_fmt(val)}")
    if a.pipe and a.which == "fwd":
        for c in tr:
            m = pipe_model(tr[c])
            if not m["span"]:
                continue
            print(f"CTA {c}: tensor pipe busy {m['busy']:.0f} of {m['span']:.0f} cycles "
                  f"({100 * m['busy'] / m['span']:.1f} %, {MMA_CYCLES:.0f} cycles per MMA)")
            for name, v in sorted(m["idle"].items(), key=lambda kv: -sum(kv[1])):
                print(f"  idle after {name:9s} {100 * sum(v) / m['span']:5.1f} % of the span "
                      f"(n={len(v)}, median {statistics.median(v):.0f} cycles)")
            for name, v in m["issue"].items():
                print(f"  issue of {name:5s} median {statistics.median(v):.0f} cycles "
                      f"({FWD_GROUP_MMAS[name]} MMAs)")
    if a.timeline:
        print(f"CTA 0 timeline (cycles from the MMA warp's stamp {a.timeline_from}):")
        for dt, role, name, blk in timeline(tr[0], a.timeline_from, a.timeline):
            print(f"  {dt:8d}  {role:10s} {name:10s} {blk}")


if __name__ == "__main__":
    main()
