"""Reader for the round-by-round ring fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LETTERS = "abcdefgh"


def parse_cell(cell: str, chunk: int):
    """'b0+a0' -> frozenset of ranks {1, 0}; '.' or '?' -> None (unchecked)."""
    cell = cell.strip()
    if cell in (".", "?"):
        return None
    ranks = set()
    for term in cell.split("+"):
        term = term.strip()
        letter, digit = term[0], int(term[1:])
        if digit != chunk:
            raise ValueError(f"cell {cell!r} mixes chunks (column {chunk})")
        ranks.add(LETTERS.index(letter))
    return frozenset(ranks)


def load(name: str):
    """Returns {('rs'|'ag', round_1based): {'sends': [(s,d,c)], 'rows': [[set|None]]}}."""
    out, cur = {}, None
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                phase, idx = line.strip("[]").split()
                cur = {"sends": [], "rows": []}
                out[(phase, int(idx))] = cur
            elif line.startswith("send"):
                _, s, d, c = line.split()
                cur["sends"].append((int(s), int(d), int(c)))
            else:
                cells = line.split("|")
                cur["rows"].append([parse_cell(c, j) for j, c in enumerate(cells)])
    return out
