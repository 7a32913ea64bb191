"""Readers for the text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_blocks(name):
    """Blocks of 'key: value' lines separated by blank lines; '#' starts a comment."""
    blocks, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.rstrip("\n")
            if line.startswith("#"):
                continue
            if not line.strip():
                if cur:
                    blocks.append(cur)
                    cur = {}
                continue
            key, _, val = line.partition(":")
            cur[key.strip()] = val.strip()
    if cur:
        blocks.append(cur)
    return blocks


def read_tree(name):
    """rank: parent | children  ->  (parent list, children lists)."""
    parent, kids = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            r, _, rest = line.partition(":")
            p, _, cs = rest.partition("|")
            parent[int(r)] = int(p)
            kids[int(r)] = [int(c) for c in cs.split()]
    W = len(parent)
    return [parent[r] for r in range(W)], [kids[r] for r in range(W)]
