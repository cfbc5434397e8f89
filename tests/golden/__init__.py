"""Parsers for the hand-derived fixtures in this folder (no expected value here
comes from any program: each is printed by the pages or derived by hand)."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def hand_blocks():
    """-> list of (type_name, case_name, {index: value}, expected_bytes)."""
    cases = []
    with open(os.path.join(HERE, "hand_blocks.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            t, name, inputs, hexbytes = (p.strip() for p in line.split("|"))
            vals = {}
            if inputs != "-":
                for kv in inputs.split(","):
                    k, v = kv.split("=")
                    vals[int(k)] = float(v)
            cases.append((t, name, vals, bytes.fromhex(hexbytes.replace(" ", ""))))
    return cases


def sizes():
    """-> {key: float} of the size facts the pages print."""
    out = {}
    with open(os.path.join(HERE, "sizes.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v, _src = (p.strip() for p in line.split("|"))
            out[k] = float(v)
    return out


def kquant_worked():
    """-> list of (name, type_name, {index: value}, {field: value or list})."""
    cases = []
    with open(os.path.join(HERE, "kquant_worked.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, t, inputs, fields = (p.strip() for p in line.split("|"))
            vals = {int(k): float(v) for k, v in (kv.split("=") for kv in inputs.split(","))}
            exp = {}
            for kv in fields.split(";"):
                k, v = kv.split("=")
                nums = [float(x) for x in v.split(",")]
                exp[k] = nums if len(nums) > 1 else nums[0]
            cases.append((name, t, vals, exp))
    return cases
