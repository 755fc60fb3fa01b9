"""Readers for the text fixtures under tests/golden/ (no arithmetic of the method)."""
import os
import struct

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(HERE, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line.split()


def load_worked_groups():
    """{group: {"scale": float32 value, "scale_bits": int, "entries": [(x, code)]}}"""
    out = {}
    for tok in _lines("e4m3_worked_groups.txt"):
        g = out.setdefault(tok[0], {"entries": []})
        if tok[1] == "scale":
            bits = int(tok[2], 16)
            g["scale_bits"] = bits
            g["scale"] = struct.unpack("<f", struct.pack("<I", bits))[0]
        else:
            g["entries"].append((float(tok[1]), int(tok[2], 16)))
    return out


def load_granularity():
    """{tensor: (rows, cols)} from the pages' quantization table."""
    return {t[0]: (int(t[2]), int(t[3])) for t in _lines("quant_granularity.txt")}


def load_metric_band():
    d = {t[0]: float(t[1]) for t in _lines("metric_band.txt")}
    return d["accepted_low"], d["accepted_high"]
