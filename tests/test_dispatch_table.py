"""The dispatch table against the committed sweep of every path
(profiles/dispatch_sweep.md: apply time of the decode, split and tensor-core
paths over tokens x rank x adapter sharing, measured on GB300).

The host does not see how the batch's tokens share adapters (the pair lists
are on the device), so the table reads the phase from the token count, as the
LoRAForge page keys its dispatch on phase, rank and shape ("Approach" (5)):
batches up to 256 tokens are decode batches (every token its own adapters,
share = 1), longer ones prefill chunks (runs of tokens sharing a request's
adapters, share = 16 or 256).  On every swept point of the phase its size
implies, lora_dispatch_choose must pick the measured-fastest path -- or, where
the two prefill-like sharings disagree, a path within 1.5x of the fastest on
both; on each of the metric's workloads it must pick the fastest path."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "profiles", "dispatch_sweep.md")
PATHS = ["decode", "split", "mma"]


@pytest.fixture(scope="module")
def native():
    from tenant_composite_lora_gb300 import build, native
    build.build()
    native.load()
    return native


def _rows(section_pred):
    rows, head = [], None
    for line in open(TABLE, encoding="utf-8"):
        line = line.strip()
        if not line.startswith("|") or set(line) <= set("|-"):
            continue
        cells = [c.strip() for c in line.strip("|").split("|")]
        if cells[0] in ("T", "workload"):
            head = cells
            continue
        if head and section_pred(head):
            rows.append(dict(zip(head, cells)))
    return rows


def sweep_points():
    pts = []
    for r in _rows(lambda h: h[0] == "T"):
        t = {p: (None if r[f"{p} us"] == "-" else float(r[f"{p} us"])) for p in PATHS}
        pts.append({"T": int(r["T"]), "r": int(r["r"]), "share": r["share"], "P": int(r["P"]), "t": t})
    return pts


def workloads():
    return [dict(r) for r in _rows(lambda h: h[0] == "workload")]


def fastest(t):
    return min((p for p in PATHS if t[p] is not None), key=lambda p: t[p])


def test_table_is_complete():
    pts = sweep_points()
    assert len(pts) >= 100
    assert {p["r"] for p in pts} >= {8, 16, 64}
    assert {p["share"] for p in pts} == {"1", "16", "256", "zipf"}
    assert all(p["t"]["decode"] is not None and p["t"]["mma"] is not None for p in pts)
    assert {w["workload"] for w in workloads()} == {"distinct", "zipf", "prefill", "sweep1", "sweep8",
                                                   "sweep64", "sweep256"}


def test_choice_is_fastest_for_the_phase_its_size_implies(native):
    names = {native.LORA_PATH_DECODE: "decode", native.LORA_PATH_SPLIT: "split", native.LORA_PATH_MMA: "mma"}
    by_cell = {}
    for p in sweep_points():
        by_cell.setdefault((p["T"], p["r"]), {})[p["share"]] = p
    checked = 0
    for (T, r), cell in sorted(by_cell.items()):
        got = names[native.lora_dispatch_choose(T, 2 * T, r, 4096, 4096)]
        typical = ["1"] if T <= 256 else ["16", "256"]
        best = {fastest(cell[s]["t"]) for s in typical}
        if len(best) == 1:
            assert got in best, f"T={T} r={r}: chose {got}, fastest {best}"
        else:
            for s in typical:
                t = cell[s]["t"]
                assert t[got] <= 1.5 * t[fastest(t)], f"T={T} r={r} share={s}: {got} {t}"
        checked += 1
    assert checked >= 30


def test_choice_is_fastest_on_every_workload(native):
    import workloads as W
    names = {native.LORA_PATH_DECODE: "decode", native.LORA_PATH_SPLIT: "split", native.LORA_PATH_MMA: "mma"}
    for w in workloads():
        wl = W.make(w["workload"])
        got = names[native.lora_dispatch_choose(wl.T, wl.P, wl.r_max, wl.d_in, wl.d_out)]
        t = {p: float(w[f"{p} us"]) for p in PATHS}
        assert got == fastest(t), f"{w['workload']}: chose {got}, times {t}"
