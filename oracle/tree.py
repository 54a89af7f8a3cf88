"""Draft-tree bookkeeping, oracle side (test infrastructure only).

[P3] feature list: the verify step checks a DDTree draft tree (block size
16, default budget 22). A tree of ``N = budget + 1`` nodes is given by
``parent``: node 0 is the root (its entry is ignored) and every other node
``i`` has ``0 <= parent[i] < i``, so parents precede children.
"""

import numpy as np


def validate(parent):
    parent = np.asarray(parent, dtype=np.int64)
    n = parent.shape[0]
    if n < 1:
        raise ValueError("a tree has at least the root")
    for i in range(1, n):
        if not (0 <= parent[i] < i):
            raise ValueError(f"parent[{i}] = {parent[i]} is not in [0, {i})")
    return parent


def depths(parent):
    """depth[0] = 0, depth[i] = depth[parent[i]] + 1."""
    parent = validate(parent)
    depth = np.zeros(parent.shape[0], dtype=np.int64)
    for i in range(1, parent.shape[0]):
        depth[i] = depth[parent[i]] + 1
    return depth


def ancestors_or_self(parent):
    """For each node, the sorted list of its ancestors and itself."""
    parent = validate(parent)
    out = []
    for i in range(parent.shape[0]):
        chain = [i]
        while chain[-1] != 0:
            chain.append(int(parent[chain[-1]]))
        out.append(sorted(chain))
    return out


def children(parent):
    """For each node, its children in increasing index order."""
    parent = validate(parent)
    kids = [[] for _ in range(parent.shape[0])]
    for i in range(1, parent.shape[0]):
        kids[parent[i]].append(i)
    return kids
