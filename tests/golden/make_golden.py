"""Writes tests/golden/oracle_tiny.json: the float64 oracle's outputs on one tiny
seeded case of each routine.  It calls only the oracle and the seeded input
generator; run it from the repository root with ``python -m tests.golden.make_golden``.
The stored numbers guard the oracle against unintended changes: a deliberate
change to its arithmetic must regenerate this file and say why in its commit."""
import json
import os

from selective_scan_mamba_gb300 import synth


def compute(oracle):
    out = {}
    m1 = synth.mamba1(1, 3, 4, 9, dtype=synth.F32, with_z=True, with_h0=True, seed=0)
    f = m1.f64
    y, hf = oracle.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), D=f("D"), z=f("z"),
                               delta_bias=f("delta_bias"), h0=f("h0"))
    out["mamba1_y"] = y.ravel().tolist()
    out["mamba1_h"] = hf.ravel().tolist()
    y, hf = oracle.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), D=f("D"),
                               delta_bias=f("delta_bias"), disc=oracle.DISC_ZOH)
    out["mamba1_zoh_y"] = y.ravel().tolist()
    s = synth.ssd(1, 10, 2, 3, 4, 1, dtype=synth.F32, with_z=True, with_h0=True, seed=0)
    g = s.f64
    y, hf = oracle.ssd_chunked(g("x"), g("dt"), g("A"), g("B"), g("C"), 4, D=g("D"), z=g("z"),
                               dt_bias=g("dt_bias"), h0=g("h0"))
    out["ssd_y"] = y.ravel().tolist()
    out["ssd_h"] = hf.ravel().tolist()
    return out


def main():
    import oracle
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    doc = {"source": "float64 oracle (oracle/oracle.c) on seeded synthetic inputs; written by "
                     "tests/golden/make_golden.py",
           "values": compute(oracle)}
    with open(path, "w") as fh:
        json.dump(doc, fh, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
