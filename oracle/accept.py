"""Greedy acceptance, oracle side (test infrastructure only).

[P3] feature list: verification is greedy only ([P3] constraints paragraph:
temperature / top_p are accepted by the server but ignored). Greedy
verification of a draft tree therefore needs:

* the target's token at every node: ``argmax`` over the node's vocabulary
  logits, ties going to the lowest index (``-0.0`` equals ``+0.0``; inputs
  hold no NaN);
* a walk from the root: while some child ``c`` of the last accepted node has
  ``token[c] == argmax[last]``, accept the lowest-index such child.

The root is always accepted (its K/V row is committed). The tokens emitted
by the step are the accepted draft tokens followed by the bonus token
``argmax[last]``.
"""

import numpy as np

from . import tree as _tree


def node_argmax(logits):
    """argmax over the last axis of float64(logits); numpy returns the first
    occurrence of the maximum, i.e. the lowest index on ties."""
    return np.argmax(np.asarray(logits, dtype=np.float64), axis=-1).astype(np.int64)


def greedy_walk(parent, tokens, target):
    """Return ``(path, out_tokens)``; ``len(path)`` is the accept length."""
    kids = _tree.children(parent)
    path = [0]
    while True:
        last = path[-1]
        nxt = None
        for c in kids[last]:            # increasing index order
            if int(tokens[c]) == int(target[last]):
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
    out_tokens = [int(tokens[c]) for c in path[1:]] + [int(target[path[-1]])]
    return np.array(path, dtype=np.int64), np.array(out_tokens, dtype=np.int64)
