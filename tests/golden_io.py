"""Readers for the hand-written fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def prepare_cases():
    """Parse prepare_hand_worked.txt into a list of dicts."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "prepare_hand_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = {"name": parts[1]}
            elif parts[0] == "end":
                cases.append(cur)
                cur = None
            else:
                vals = [int(v) for v in parts[1:]]
                if parts[0] in ("T", "K", "E", "A", "R", "P", "status"):
                    cur[parts[0]] = vals[0]
                else:
                    cur[parts[0]] = vals
    return cases


def rounding_cases():
    """Parse combine_rounding.txt: (name, K, [row bits], expected bits)."""
    out = []
    with open(os.path.join(GOLDEN, "combine_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            name, K = parts[0], int(parts[1])
            rows = [int(v, 16) for v in parts[2:2 + K]]
            expected = int(parts[2 + K], 16)
            out.append((name, K, rows, expected))
    return out


def shard_cases():
    """Parse shard_hand_worked.txt into a list of dicts."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "shard_hand_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = {"name": parts[1]}
            elif parts[0] == "end":
                cases.append(cur)
                cur = None
            else:
                vals = [int(v) for v in parts[1:]]
                cur[parts[0]] = vals[0] if parts[0] in ("N", "K", "E", "A", "R") else vals
    return cases


RM_FLOAT_KEYS = ("w", "rw", "part", "out", "gw", "gout")


def rank_major_cases():
    """Parse rank_major_hand_worked.txt into a list of dicts (float fields:
    weights, partial rows, results, weight gradients)."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "rank_major_hand_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = {"name": parts[1]}
            elif parts[0] == "end":
                cases.append(cur)
                cur = None
            else:
                key = parts[0]
                is_float = key.rstrip("0123456789") in RM_FLOAT_KEYS
                vals = [float(v) if is_float else int(v) for v in parts[1:]]
                cur[key] = vals[0] if key in ("N", "K", "E", "R") else vals
    return cases
